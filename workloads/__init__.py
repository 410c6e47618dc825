"""Seeded synthetic workloads for one routed mixture-of-experts layer forward.

This module holds the layer shapes and the seeded input generator, and nothing
of the layer's arithmetic: no gate, softmax, selection, permutation, FFN or
combine step lives here. Both the CUDA path and the CPU oracle take their
inputs from this module, so a disagreement between them can never come from a
shared helper.

Shapes follow the workloads the source pages discuss:
  * 8 experts, top-2, a batch of 1024 tokens (ThunderEP, "MoE expert parallel
    communication", section 2.1: a 1024x2 int32 routing-index array);
  * 64 experts, top-2 (DeepSeek-V4 EP article, section 2.1);
  * batch 32 x seq 512, hidden 5120, 16 experts, top-2 with an FP8 payload
    (Deepseek-MoE sync-tax article, sections 2.1 and 3.1);
  * top-8 routing over 256 fine-grained experts (DeepSeek V3/V4 parallel
    strategy article, EP section).

Recipe (the draw order is part of the definition): x, W_g, bias, W1[0..E-1],
W2[0..E-1], then the outlier mask and signs, then the Zipf expert permutation.
Every normal draw is fp32 from a ``torch.Generator`` seeded with the config's
seed on the generating device, multiplied by its standard deviation and, for
bf16 layers, rounded to bf16 (round to nearest even). CPU and CUDA generators
give different streams; within one process both sides of a comparison always
see the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

__all__ = ["MoEConfig", "CONFIGS", "VARIANTS", "BENCH_CONFIG", "get_config", "make_inputs",
           "ROUTER_RENORM", "ROUTER_PREK_SOFTMAX", "ROUTER_GROUP_LIMITED",
           "ROUTER_SOFT_GUMBEL"]

# Router modes (mirrors the values in include/moe.h).
ROUTER_RENORM = 0        # softmax over all E, keep top-k, divide by their sum
ROUTER_PREK_SOFTMAX = 1  # softmax over the pre_k largest logits, keep top-k as is
ROUTER_GROUP_LIMITED = 2  # top-k inside the topk_group best of n_group expert groups
ROUTER_SOFT_GUMBEL = 3    # Gumbel-softmax over all E experts (k = E), temperature tau


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens
    d: int            # hidden size
    E: int            # experts
    k: int            # experts per token
    f: int            # expert FFN inner size
    dtype: str        # "f32" or "bf16": activations and weights
    router: int = ROUTER_RENORM
    pre_k: int = 8
    n_group: int = 1          # expert groups (group-limited router only)
    topk_group: int = 1       # groups kept per token (group-limited router only)
    payload_fp8: int = 0      # 0 none, 1 per-token absmax FP8, 2 FP8 with one static scale
    payload_scale: float = 0.0  # the static scale (payload_fp8 == 2)
    output_fp8: int = 0       # 1: expert outputs reach the combine as FP8 (min/max affine)
    tau: float = 1.0          # soft gating temperature
    gemm_tile_n: int = 0      # expert GEMM pair-tile width: 0 = the library's choice, 256, 512
    x_perm_mode: int = 0      # 0 = the library's choice, 1 = packed rows, 2 = gathered by the W1 GEMM
    keep_z: int = 0           # 1: the forward keeps the pre-activation Z for the backward
    bias: str = "zero"        # "zero" | "normal" (variance bias_var) | "zipf" (exponent zipf_s)
    bias_var: float = 0.0
    zipf_s: float = 0.0
    outlier_rate: float = 0.0  # fraction of x entries replaced by +-outlier_mag
    outlier_mag: float = 20.0
    seed: int = 0

    @property
    def R(self) -> int:
        """Routed rows: one per (token, chosen expert) pair."""
        return self.T * self.k

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# The five layer shapes. Seeds: the tiny layer states seed 0; the others take
# seed i-1 for the i-th shape.
CONFIGS = {
    "tiny_T256_d128_E8_k2_f256_fp32": MoEConfig(
        "tiny_T256_d128_E8_k2_f256_fp32", T=256, d=128, E=8, k=2, f=256,
        dtype="f32", seed=0),
    "balanced_T1024_d4096_E8_k2_f11008": MoEConfig(
        "balanced_T1024_d4096_E8_k2_f11008", T=1024, d=4096, E=8, k=2, f=11008,
        dtype="bf16", seed=1),
    "many_expert_T8192_d2048_E64_k2_f1408_prek8": MoEConfig(
        "many_expert_T8192_d2048_E64_k2_f1408_prek8", T=8192, d=2048, E=64, k=2,
        f=1408, dtype="bf16", router=ROUTER_PREK_SOFTMAX, pre_k=8,
        bias="normal", bias_var=0.5, seed=2),
    "wide_fp8_T16384_d5120_E16_k2_f1536": MoEConfig(
        "wide_fp8_T16384_d5120_E16_k2_f1536", T=32 * 512, d=5120, E=16, k=2,
        f=1536, dtype="bf16", payload_fp8=True, outlier_rate=1e-3,
        outlier_mag=20.0, seed=3),
    "skewed_T16384_d7168_E256_k8_f2048_zipf": MoEConfig(
        "skewed_T16384_d7168_E256_k8_f2048_zipf", T=16384, d=7168, E=256, k=8,
        f=2048, dtype="bf16", bias="zipf", zipf_s=1.1, seed=4),
}
CONFIG_ORDER = list(CONFIGS)

# Variants of the five shapes for the router and payload options the pages
# describe besides the default path. Node-limited routing: the fine-grained
# layer (256 experts, top-8) with its experts in 8 groups of 32 ("nodes") and
# each token's 8 experts taken from its 4 best groups (DeepSeek V3/V4
# parallel-strategy article, EP section).
# Static global FP8 scale (sync-tax article, section 3.1, "static global"):
# the wide layer with one payload scale fixed ahead of time, 20/448, so the
# largest magnitude in the data (the +-20 outliers) maps to the E4M3 maximum.
# FP8 expert outputs: the wide layer with both FP8 payloads of the sync-tax
# article (section 3.1), per-token absmax on the expert inputs and per-row
# min/max affine on the expert outputs.
# Soft gating (sync-tax article, section 3.3): the wide layer's 16 experts,
# every token weighted over all of them by a Gumbel-softmax at tau = 1.
VARIANTS = {
    "soft_gumbel_T16384_d5120_E16_f1536": MoEConfig(
        "soft_gumbel_T16384_d5120_E16_f1536", T=32 * 512, d=5120, E=16, k=16, f=1536,
        dtype="bf16", router=ROUTER_SOFT_GUMBEL, tau=1.0, seed=3),
    "wide_fp8_T16384_d5120_E16_k2_f1536_outfp8": MoEConfig(
        "wide_fp8_T16384_d5120_E16_k2_f1536_outfp8", T=32 * 512, d=5120, E=16, k=2,
        f=1536, dtype="bf16", payload_fp8=1, output_fp8=1, outlier_rate=1e-3,
        outlier_mag=20.0, seed=3),
    "wide_fp8static_T16384_d5120_E16_k2_f1536": MoEConfig(
        "wide_fp8static_T16384_d5120_E16_k2_f1536", T=32 * 512, d=5120, E=16, k=2,
        f=1536, dtype="bf16", payload_fp8=2, payload_scale=20.0 / 448.0, outlier_rate=1e-3,
        outlier_mag=20.0, seed=3),
    "skewed_T16384_d7168_E256_k8_f2048_zipf_group8top4": MoEConfig(
        "skewed_T16384_d7168_E256_k8_f2048_zipf_group8top4", T=16384, d=7168, E=256, k=8,
        f=2048, dtype="bf16", router=ROUTER_GROUP_LIMITED, n_group=8, topk_group=4,
        bias="zipf", zipf_s=1.1, seed=4),
}
# A scaled-down copy of the fine-grained skewed layer (same d, f, k, router
# and Zipf bias; 32 experts over 2048 tokens keep its mean of 512 rows per
# expert): small enough for detailed profiler captures of its kernels.
VARIANTS["skewed_small_T2048_d7168_E32_k8_f2048_zipf"] = MoEConfig(
    "skewed_small_T2048_d7168_E32_k8_f2048_zipf", T=2048, d=7168, E=32, k=8, f=2048,
    dtype="bf16", bias="zipf", zipf_s=1.1, seed=4)

# The layer the headline throughput is quoted on: the largest that fits one
# GPU, the fine-grained skewed layer (256 experts, top-8).
BENCH_CONFIG = CONFIG_ORDER[4]


def get_config(name: str) -> MoEConfig:
    if name in CONFIGS:
        return CONFIGS[name]
    if name in VARIANTS:
        return VARIANTS[name]
    # also accept a 1-based position ("1".."5") or a unique prefix
    if name.isdigit() and 1 <= int(name) <= len(CONFIG_ORDER):
        return CONFIGS[CONFIG_ORDER[int(name) - 1]]
    hits = [n for n in CONFIG_ORDER if n.startswith(name)]
    if len(hits) == 1:
        return CONFIGS[hits[0]]
    raise KeyError(f"unknown MoE config {name!r}; known: {CONFIG_ORDER}")


def _normal(gen, shape, std, device, dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t if dtype == torch.float32 else t.to(dtype)


def make_inputs(cfg: MoEConfig, device="cpu") -> dict:
    """Draw the layer's inputs for ``cfg`` on ``device``.

    Returns a dict of tensors on ``device``:
      x    [T, d]     activations (fp32 or bf16), x ~ N(0, 1)
      Wg   [d, E]     gate weights, N(0, 1/d)
      bias [E]        fp32 per-expert gate bias (zeros unless the shape has one)
      W1   [E, d, f]  expert up projections, N(0, 1/d)
      W2   [E, f, d]  expert down projections, N(0, 1/f)
      gumbel [T, E]   fp32 Gumbel(0, 1) samples, soft gating only: the random
                      numbers the router draws, passed to both sides as an
                      input (drawn last, as -ln of Exp(1) draws)
    """
    dev = torch.device(device)
    dt = cfg.torch_dtype
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    T, d, E, f = cfg.T, cfg.d, cfg.E, cfg.f

    x = _normal(gen, (T, d), 1.0, dev, dt)
    Wg = _normal(gen, (d, E), 1.0 / math.sqrt(d), dev, dt)
    if cfg.bias == "normal":
        bias = _normal(gen, (E,), math.sqrt(cfg.bias_var), dev, torch.float32)
    else:
        bias = torch.zeros(E, dtype=torch.float32, device=dev)
    W1 = torch.empty((E, d, f), dtype=dt, device=dev)
    for e in range(E):
        W1[e] = _normal(gen, (d, f), 1.0 / math.sqrt(d), dev, dt)
    W2 = torch.empty((E, f, d), dtype=dt, device=dev)
    for e in range(E):
        W2[e] = _normal(gen, (f, d), 1.0 / math.sqrt(f), dev, dt)

    if cfg.outlier_rate > 0.0:
        hit = torch.rand((T, d), generator=gen, device=dev) < cfg.outlier_rate
        neg = torch.rand((T, d), generator=gen, device=dev) < 0.5
        mag = torch.full((T, d), cfg.outlier_mag, dtype=torch.float32, device=dev)
        mag = torch.where(neg, -mag, mag).to(dt)
        x = torch.where(hit, mag, x)

    if cfg.bias == "zipf":
        # Zipf(s) popularity over a random expert order, put into the logits as
        # log-probabilities: the r-th most popular expert gets -s*ln(r). The
        # normalising constant is dropped (it shifts every logit equally).
        perm = torch.randperm(E, generator=gen, device=dev)
        ranks = torch.arange(1, E + 1, dtype=torch.float64, device=dev)
        vals = (-cfg.zipf_s * torch.log(ranks)).to(torch.float32)
        bias = torch.empty(E, dtype=torch.float32, device=dev)
        bias[perm] = vals

    out = {"x": x.contiguous(), "Wg": Wg.contiguous(), "bias": bias.contiguous(),
           "W1": W1, "W2": W2}
    if cfg.router == ROUTER_SOFT_GUMBEL:
        ex = torch.empty((T, E), dtype=torch.float32, device=dev).exponential_(generator=gen)
        out["gumbel"] = (-torch.log(ex)).contiguous()
    return out
