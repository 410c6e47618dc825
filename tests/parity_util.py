"""Shared helpers for the GPU parity tests: tolerances, comparisons and the
near-tie protocol for routing. Expected values always come from the oracle
(or from the inputs themselves, indexed by the oracle's permutation)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances for the layer output and the FFN intermediates.
BF16_REL_L2 = 2e-3
BF16_MAX_ABS = 2e-2
FP8_MAX_ABS = 5e-2
F32_REL_L2 = 1e-5
F32_MAX_ABS = 1e-5
# Router: weights max-abs, logits max-abs, and the gap below which two
# logits count as tied (fp32 accumulation cannot order them reliably).
W_MAX_ABS = 1e-6
LOGIT_MAX_ABS = 1e-5
TIE_GAP = 1e-5


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.cpu().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a tensor (for bit-exact comparisons)."""
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def assert_close(got, ref, rel, max_abs, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_l2(got, ref)
    m = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert r <= rel and m <= max_abs, f"{what}: rel_l2={r:.3e} (<= {rel}), max_abs={m:.3e} (<= {max_abs})"
    return r, m


def out_tolerance(cfg):
    if cfg.dtype == "f32":
        return F32_REL_L2, F32_MAX_ABS
    return BF16_REL_L2, (FP8_MAX_ABS if cfg.payload_fp8 else BF16_MAX_ABS)


def near_tie_tokens(L64: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose top k+1 logits (fp64) hold two within TIE_GAP of each
    other: their selection or slot order can legitimately flip in fp32."""
    E = L64.shape[1]
    m = min(k + 1, E)
    top = -np.sort(-L64, axis=1)[:, :m]
    if m < 2:
        return np.zeros(L64.shape[0], dtype=bool)
    gaps = top[:, :-1] - top[:, 1:]
    return gaps.min(axis=1) < TIE_GAP


def topk_of(L: np.ndarray, k: int) -> np.ndarray:
    """Top-k by (value desc, id asc), written independently of the oracle."""
    T, E = L.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -L), axis=1)
    return order[:, :k]


def check_route(cfg, L_oracle, idx_oracle, w_oracle, L_gpu, idx_gpu, w_gpu):
    """Near-tie protocol. Returns the number of near-tie tokens."""
    L_gpu = np.asarray(L_gpu, np.float64)
    dl = np.max(np.abs(L_gpu - L_oracle))
    assert dl <= LOGIT_MAX_ABS, f"logits max-abs {dl:.3e}"
    tie = near_tie_tokens(L_oracle, cfg.k)
    clear = ~tie
    assert np.array_equal(idx_gpu[clear], idx_oracle[clear]), \
        f"{int((idx_gpu[clear] != idx_oracle[clear]).any(1).sum())} clear tokens routed differently"
    dw = np.max(np.abs(w_gpu[clear] - w_oracle[clear])) if clear.any() else 0.0
    assert dw <= W_MAX_ABS, f"weights max-abs {dw:.3e}"
    if tie.any():
        # the GPU's choice must be the exact top-k of its own logits
        own = topk_of(L_gpu[tie], cfg.k)
        assert np.array_equal(idx_gpu[tie], own)
        same = np.all(idx_gpu[tie] == idx_oracle[tie], axis=1)
        dw_t = np.max(np.abs(w_gpu[tie][same] - w_oracle[tie][same])) if same.any() else 0.0
        assert dw_t <= W_MAX_ABS
    return int(tie.sum())
