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
# Group-limited router: two group scores (sums of fp32 exponentials of
# logits that are themselves good to ~1e-5) closer than this relative gap
# count as tied.
GROUP_TIE_REL = 5e-5
ROUTER_GROUP_LIMITED = 2


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


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits): 2^(e - 7) for
    |v| in [2^e, 2^(e+1)); the subnormal spacing below 2^-126."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def assert_close_bf16_stored(got, ref, rel, max_abs, what=""):
    """assert_close for values stored in bf16 (the expert FFN's H): both
    sides round an fp32 (GPU) or fp64 (oracle) sum to bf16, and a sum that
    lies next to a rounding midpoint may round to the neighbouring bf16
    value on one side. Each element may therefore also differ by one bf16
    ulp of its value; rel-L2 stays bounded as usual."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_l2(got, ref)
    d = np.abs(got - ref)
    bad = d > np.maximum(max_abs, bf16_ulp(ref))
    assert r <= rel and not bad.any(), (
        f"{what}: rel_l2={r:.3e} (<= {rel}), {int(bad.sum())} elements beyond max(max_abs "
        f"{max_abs}, one bf16 ulp), largest difference {float(d.max()) if d.size else 0.0:.3e}")
    return r, float(d.max()) if d.size else 0.0


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


def group_scores(L64: np.ndarray, n_group: int) -> np.ndarray:
    """sum over each group's experts of exp(L - max L): ranks the groups as
    their mean softmax probability does."""
    T, E = L64.shape
    z = np.exp(L64 - L64.max(axis=1, keepdims=True))
    return z.reshape(T, n_group, E // n_group).sum(axis=2)


def near_tie_tokens_group(L64: np.ndarray, cfg) -> np.ndarray:
    """Group-limited router: tokens whose topk_group-th and next group scores
    are within GROUP_TIE_REL, or whose top k+1 logits inside the kept groups
    hold two within TIE_GAP."""
    T, E = L64.shape
    G, M = cfg.n_group, cfg.topk_group
    gs = E // G
    sc = group_scores(L64, G)
    order = np.lexsort((np.broadcast_to(np.arange(G), (T, G)), -sc), axis=1)
    tie = np.zeros(T, dtype=bool)
    if M < G:
        a = sc[np.arange(T), order[:, M - 1]]
        b = sc[np.arange(T), order[:, M]]
        tie |= (a - b) <= GROUP_TIE_REL * a
    allowed = np.zeros((T, E), dtype=bool)
    for j in range(M):
        g = order[:, j]
        for i in range(gs):
            allowed[np.arange(T), g * gs + i] = True
    Lk = np.where(allowed, L64, -np.inf)
    m = min(cfg.k + 1, M * gs)
    if m >= 2:
        top = -np.sort(-Lk, axis=1)[:, :m]
        tie |= (top[:, :-1] - top[:, 1:]).min(axis=1) < TIE_GAP
    return tie


def route_ties(cfg, L64: np.ndarray) -> np.ndarray:
    """Tokens whose routing fp32 cannot decide reliably, for any router."""
    if getattr(cfg, "router", 0) == 3:     # soft gating selects nothing
        return np.zeros(L64.shape[0], dtype=bool)
    if getattr(cfg, "router", 0) == ROUTER_GROUP_LIMITED:
        return near_tie_tokens_group(L64, cfg)
    return near_tie_tokens(L64, cfg.k)


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
    tie = route_ties(cfg, L_oracle)
    clear = ~tie
    assert np.array_equal(idx_gpu[clear], idx_oracle[clear]), \
        f"{int((idx_gpu[clear] != idx_oracle[clear]).any(1).sum())} clear tokens routed differently"
    dw = np.max(np.abs(w_gpu[clear] - w_oracle[clear])) if clear.any() else 0.0
    assert dw <= W_MAX_ABS, f"weights max-abs {dw:.3e}"
    if tie.any() and getattr(cfg, "router", 0) == ROUTER_GROUP_LIMITED:
        _check_group_choice(cfg, L_gpu[tie], idx_gpu[tie], w_gpu[tie])
    elif tie.any():
        # the GPU's choice must be the exact top-k of its own logits
        own = topk_of(L_gpu[tie], cfg.k)
        assert np.array_equal(idx_gpu[tie], own)
        same = np.all(idx_gpu[tie] == idx_oracle[tie], axis=1)
        dw_t = np.max(np.abs(w_gpu[tie][same] - w_oracle[tie][same])) if same.any() else 0.0
        assert dw_t <= W_MAX_ABS
    return int(tie.sum())


def _check_group_choice(cfg, L_own, idx, w):
    """A group-limited choice is valid for the GPU's own logits when its
    experts come from at most topk_group groups, each scoring within
    GROUP_TIE_REL of the topk_group-th best, when they are the top k of the
    union of their own groups, and when the weights are those logits'
    renormalised softmax."""
    L_own = np.asarray(L_own, np.float64)
    n, E = L_own.shape
    G, M, k = cfg.n_group, cfg.topk_group, cfg.k
    gs = E // G
    sc = group_scores(L_own, G)
    thr = -np.sort(-sc, axis=1)[:, M - 1]
    for t in range(n):
        groups = sorted(set(int(e) // gs for e in idx[t]))
        assert len(groups) <= M, (t, idx[t])
        assert all(sc[t, g] >= thr[t] * (1 - GROUP_TIE_REL) for g in groups), (t, idx[t])
        cand = np.array([e for g in groups for e in range(g * gs, (g + 1) * gs)])
        sub = L_own[t, cand]
        best = cand[np.lexsort((cand, -sub))[:k]]
        assert list(idx[t]) == list(best), (t, idx[t], best)
        z = np.exp(L_own[t, idx[t]] - L_own[t, idx[t]].max())
        assert np.max(np.abs(w[t] - z / z.sum())) <= W_MAX_ABS


def e4m3_step(q: np.ndarray) -> np.ndarray:
    """Distance from an E4M3 value to its neighbour away from zero (at most
    the distance to either neighbour): 2^(e-3) for normals |q| in
    [2^e, 2^(e+1)), 2^-9 for subnormals and zero."""
    a = np.abs(np.asarray(q, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


def assert_close_output_fp8(cfg, got, ref_out, w, yq_slots, ys_slots, gpu_codes=None, what=""):
    """Layer output with the FP8 expert-output payload. The GPU quantises its
    own fp32 expert outputs, which differ from the oracle's in the last bits
    (fp32 accumulation order, bf16 rounding of H), so a value next to an E4M3
    rounding midpoint may take the neighbouring code. The bound: each slot
    may be off by one E4M3 step of its oracle code times its scale; what is
    left after that slack must meet the layer's max-abs and rel-L2. With
    ``gpu_codes`` (the GPU's own E4M3 values, decoded by torch, in slot
    layout) the share of flipped codes is checked too: under 1 %."""
    rel, mabs = out_tolerance(cfg)
    got = np.asarray(got, np.float64)
    ref_out = np.asarray(ref_out, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    step = e4m3_step(yq_slots)
    slack = np.einsum("tj,tj,tjc->tc", np.abs(w), ys_slots, step)
    excess = np.maximum(np.abs(got - ref_out) - slack, 0.0)
    den = np.linalg.norm(ref_out)
    r = float(np.linalg.norm(excess) / den) if den > 0 else float(np.linalg.norm(excess))
    assert r <= rel, f"{what}: rel_l2 beyond one E4M3 step = {r:.3e} (<= {rel})"
    assert excess.max() <= mabs, f"{what}: max-abs beyond one E4M3 step = {excess.max():.3e}"
    if gpu_codes is not None:
        # a systematic error (wrong zero point or scale, truncation) changes
        # most codes; legitimate flips are rare. A flip may span more than one
        # step where |q| is small: one bf16 rounding flip of H moves y by
        # ~|W2| * 2^-8 |H|, several steps of (y - zero)/s near zero.
        gq = np.asarray(gpu_codes, np.float64)
        flip = gq != yq_slots
        print(f"{what}: FP8 output codes differing from the oracle's: {flip.mean():.4%}")
        assert flip.mean() <= 1e-2, f"{what}: {flip.mean():.2%} of the FP8 codes differ"
    return r
