"""Layer shapes and cached inputs/oracle results for the GPU parity tests.

Inputs are drawn on the GPU by ``workloads.make_inputs`` (seeded) and copied
to the host for the oracle; the oracle never sees anything the CUDA path
produced."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from workloads import (CONFIGS, CONFIG_ORDER, VARIANTS, MoEConfig, ROUTER_PREK_SOFTMAX,
                       ROUTER_GROUP_LIMITED, ROUTER_SOFT_GUMBEL)

# Small shapes that exercise ragged tails, partial tiles and degenerate cases.
SMALL = {
    "ragged_T129_d256_E8_k2_f320": MoEConfig("ragged_T129_d256_E8_k2_f320", T=129, d=256, E=8,
                                             k=2, f=320, dtype="bf16", seed=11),
    "one_token_T1_d128_E4_k2_f128": MoEConfig("one_token_T1_d128_E4_k2_f128", T=1, d=128, E=4,
                                              k=2, f=128, dtype="bf16", pre_k=4, seed=12),
    "T7_d192_E16_k3_f192": MoEConfig("T7_d192_E16_k3_f192", T=7, d=192, E=16, k=3, f=192,
                                     dtype="bf16", seed=13),
    "single_expert_T70_d128_E1_k1_f192": MoEConfig("single_expert_T70_d128_E1_k1_f192", T=70,
                                                   d=128, E=1, k=1, f=192, dtype="bf16",
                                                   pre_k=1, seed=14),
    "k_eq_E_T33_d128_E4_k4_f128": MoEConfig("k_eq_E_T33_d128_E4_k4_f128", T=33, d=128, E=4,
                                            k=4, f=128, dtype="bf16", pre_k=4, seed=15),
    "wide_E40_T100_d256_k3_f256": MoEConfig("wide_E40_T100_d256_k3_f256", T=100, d=256, E=40,
                                            k=3, f=256, dtype="bf16", bias="normal",
                                            bias_var=2.0, seed=16),
    "fp8_T64_d256_E4_k2_f256": MoEConfig("fp8_T64_d256_E4_k2_f256", T=64, d=256, E=4, k=2,
                                         f=256, dtype="bf16", pre_k=4, payload_fp8=True,
                                         outlier_rate=0.01, seed=17),
    "prek_T200_d256_E64_k2_f128": MoEConfig("prek_T200_d256_E64_k2_f128", T=200, d=256, E=64,
                                            k=2, f=128, dtype="bf16",
                                            router=ROUTER_PREK_SOFTMAX, bias="normal",
                                            bias_var=0.5, seed=18),
    "f32_T50_d64_E5_k2_f128": MoEConfig("f32_T50_d64_E5_k2_f128", T=50, d=64, E=5, k=2,
                                        f=128, dtype="f32", pre_k=5, seed=19),
    "multi_mtile_T300_d512_E2_k1_f768": MoEConfig("multi_mtile_T300_d512_E2_k1_f768", T=300,
                                                  d=512, E=2, k=1, f=768, dtype="bf16",
                                                  pre_k=2, seed=20),
    "skew_T256_d128_E64_k8_f128_zipf": MoEConfig("skew_T256_d128_E64_k8_f128_zipf", T=256,
                                                 d=128, E=64, k=8, f=128, dtype="bf16",
                                                 bias="zipf", zipf_s=3.0, seed=21),
    # tensor-core gate: E = 192 (half-width column offset 96), a 1-block last
    # K chunk (d = 320), 3 token tiles with a 44-token tail
    "gate_E192_T300_d320_k4_f128": MoEConfig("gate_E192_T300_d320_k4_f128", T=300, d=320,
                                             E=192, k=4, f=128, dtype="bf16", bias="normal",
                                             bias_var=1.0, seed=22),
    "gate_E256_T130_d192_k8_f128": MoEConfig("gate_E256_T130_d192_k8_f128", T=130, d=192,
                                             E=256, k=8, f=128, dtype="bf16", seed=23),
    "gate_E128_T1_d1024_k2_f128_prek": MoEConfig("gate_E128_T1_d1024_k2_f128_prek", T=1,
                                                 d=1024, E=128, k=2, f=128, dtype="bf16",
                                                 router=ROUTER_PREK_SOFTMAX, seed=24),
    # 512-feature GEMM tiles (K >= 1024, N >= 512): 300 rows per expert = a full
    # 256-row tile + a swapped 44-row tail; f = 1600 leaves a last feature
    # block of 64 (one box, one of the two MMAs)
    "wide_tile_T300_d1024_E2_k2_f1600": MoEConfig("wide_tile_T300_d1024_E2_k2_f1600", T=300,
                                                  d=1024, E=2, k=2, f=1600, dtype="bf16",
                                                  pre_k=2, seed=25),
    "wide_tile_fp8_T520_d1024_E4_k1_f1024": MoEConfig("wide_tile_fp8_T520_d1024_E4_k1_f1024",
                                                      T=520, d=1024, E=4, k=1, f=1024,
                                                      dtype="bf16", pre_k=4, payload_fp8=True,
                                                      seed=26),
    # merged remainder tiles (one full 256-row tile + 1..32 rows): 270 rows
    # per expert (remainder 14) with partial last 224-feature blocks; 544
    # rows (remainder 32, FP8 row scales, a plain full tile before the
    # merged one); 257 rows (remainder 1)
    "merged_tail_T270_d256_E2_k2_f320": MoEConfig("merged_tail_T270_d256_E2_k2_f320", T=270,
                                                  d=256, E=2, k=2, f=320, dtype="bf16",
                                                  pre_k=2, seed=27),
    "merged_tail_fp8_T544_d512_E1_k1_f576": MoEConfig("merged_tail_fp8_T544_d512_E1_k1_f576",
                                                      T=544, d=512, E=1, k=1, f=576,
                                                      dtype="bf16", pre_k=1, payload_fp8=True,
                                                      outlier_rate=0.01, seed=28),
    "merged_tail_T257_d128_E1_k1_f256": MoEConfig("merged_tail_T257_d128_E1_k1_f256", T=257,
                                                  d=128, E=1, k=1, f=256, dtype="bf16",
                                                  pre_k=1, seed=29),
    # tensor-core gate for E < 64 (T >= 4096): E = 16 with a 4-token last
    # tile; E = 40 (weight boxes past E zero-filled) with a bias and a
    # one-block last K chunk
    "gate_E16_T4100_d256_k2_f128": MoEConfig("gate_E16_T4100_d256_k2_f128", T=4100, d=256,
                                             E=16, k=2, f=128, dtype="bf16", seed=30),
    "gate_E40_T4096_d320_k3_f128": MoEConfig("gate_E40_T4096_d320_k3_f128", T=4096, d=320,
                                             E=40, k=3, f=128, dtype="bf16", bias="normal",
                                             bias_var=1.0, seed=31),
    # group-limited router on each gate kernel: narrow (E <= 32, bf16 and
    # fp32), tiled (fp32, E = 64, bias), tensor-core (E = 256 Zipf; E = 128
    # in 32 groups of 4; E = 16 at T >= 4096 with groups of 2); fp32 E = 16
    # at T >= 4096 takes the K-split tiled kernel
    "group_E16_T300_d256_k2_f128_g4top2": MoEConfig(
        "group_E16_T300_d256_k2_f128_g4top2", T=300, d=256, E=16, k=2, f=128, dtype="bf16",
        router=ROUTER_GROUP_LIMITED, n_group=4, topk_group=2, seed=40),
    "group_f32_E8_T256_d128_k2_f256_g4top2": MoEConfig(
        "group_f32_E8_T256_d128_k2_f256_g4top2", T=256, d=128, E=8, k=2, f=256, dtype="f32",
        router=ROUTER_GROUP_LIMITED, n_group=4, topk_group=2, seed=41),
    "group_f32_E64_T500_d256_k4_f128_g8top3": MoEConfig(
        "group_f32_E64_T500_d256_k4_f128_g8top3", T=500, d=256, E=64, k=4, f=128, dtype="f32",
        router=ROUTER_GROUP_LIMITED, n_group=8, topk_group=3, bias="normal", bias_var=0.5,
        seed=42),
    "group_E256_T1100_d512_k8_f128_g8top4_zipf": MoEConfig(
        "group_E256_T1100_d512_k8_f128_g8top4_zipf", T=1100, d=512, E=256, k=8, f=128,
        dtype="bf16", router=ROUTER_GROUP_LIMITED, n_group=8, topk_group=4, bias="zipf",
        zipf_s=1.1, seed=43),
    "group_E128_T600_d256_k6_f128_g32top3": MoEConfig(
        "group_E128_T600_d256_k6_f128_g32top3", T=600, d=256, E=128, k=6, f=128,
        dtype="bf16", router=ROUTER_GROUP_LIMITED, n_group=32, topk_group=3, seed=44),
    "group_E16_T4100_d256_k2_f128_g8top1": MoEConfig(
        "group_E16_T4100_d256_k2_f128_g8top1", T=4100, d=256, E=16, k=2, f=128, dtype="bf16",
        router=ROUTER_GROUP_LIMITED, n_group=8, topk_group=1, seed=45),
    # static FP8 payload scale: 4/448 saturates the +-20 outliers and the
    # largest normal values; 20/448 on a ragged 8-expert layer
    "fp8static_T300_d512_E4_k2_f256": MoEConfig(
        "fp8static_T300_d512_E4_k2_f256", T=300, d=512, E=4, k=2, f=256, dtype="bf16",
        pre_k=4, payload_fp8=2, payload_scale=4.0 / 448.0, outlier_rate=0.01, seed=47),
    "fp8static_T129_d256_E8_k2_f320": MoEConfig(
        "fp8static_T129_d256_E8_k2_f320", T=129, d=256, E=8, k=2, f=320, dtype="bf16",
        payload_fp8=2, payload_scale=20.0 / 448.0, outlier_rate=0.001, seed=48),
    # FP8 expert-output payload (per-row min/max affine) before the combine:
    # bf16 with a ragged batch, fp32 out with k = 3, k = 8, and together with
    # the FP8 input payload
    "outfp8_T300_d512_E4_k2_f256": MoEConfig(
        "outfp8_T300_d512_E4_k2_f256", T=300, d=512, E=4, k=2, f=256, dtype="bf16", pre_k=4,
        output_fp8=1, seed=49),
    "outfp8_f32_T64_d128_E4_k3_f128": MoEConfig(
        "outfp8_f32_T64_d128_E4_k3_f128", T=64, d=128, E=4, k=3, f=128, dtype="f32", pre_k=4,
        output_fp8=1, seed=50),
    "outfp8_T100_d256_E16_k8_f128": MoEConfig(
        "outfp8_T100_d256_E16_k8_f128", T=100, d=256, E=16, k=8, f=128, dtype="bf16",
        output_fp8=1, seed=51),
    "outfp8_fp8in_T200_d256_E8_k2_f256": MoEConfig(
        "outfp8_fp8in_T200_d256_E8_k2_f256", T=200, d=256, E=8, k=2, f=256, dtype="bf16",
        payload_fp8=1, output_fp8=1, outlier_rate=0.01, seed=52),
    # soft gating (every token to every expert): narrow gate and a merged
    # remainder-free pair GEMM (bf16, E = 8); fp32 (SIMT GEMM, tau 0.5); the
    # tensor-core gate with 16 experts at T = 4100 (merged remainders of 4
    # rows, 16-row combine); fp32 K-split tiled gate; FP8 expert outputs
    "soft_E8_T300_d256_f256": MoEConfig(
        "soft_E8_T300_d256_f256", T=300, d=256, E=8, k=8, f=256, dtype="bf16",
        router=ROUTER_SOFT_GUMBEL, seed=53),
    "soft_f32_E4_T64_d128_f128_tau05": MoEConfig(
        "soft_f32_E4_T64_d128_f128_tau05", T=64, d=128, E=4, k=4, f=128, dtype="f32", pre_k=4,
        router=ROUTER_SOFT_GUMBEL, tau=0.5, seed=54),
    "soft_E16_T4100_d256_f128": MoEConfig(
        "soft_E16_T4100_d256_f128", T=4100, d=256, E=16, k=16, f=128, dtype="bf16",
        router=ROUTER_SOFT_GUMBEL, bias="normal", bias_var=1.0, seed=55),
    "soft_f32_E16_T4100_d128_f128": MoEConfig(
        "soft_f32_E16_T4100_d128_f128", T=4100, d=128, E=16, k=16, f=128, dtype="f32",
        router=ROUTER_SOFT_GUMBEL, tau=2.0, seed=56),
    "soft_outfp8_E16_T1000_d512_f256": MoEConfig(
        "soft_outfp8_E16_T1000_d512_f256", T=1000, d=512, E=16, k=16, f=256, dtype="bf16",
        router=ROUTER_SOFT_GUMBEL, output_fp8=1, seed=57),
    "group_f32_E16_T4100_d128_k3_f128_g4top2": MoEConfig(
        "group_f32_E16_T4100_d128_k3_f128_g4top2", T=4100, d=128, E=16, k=3, f=128,
        dtype="f32", router=ROUTER_GROUP_LIMITED, n_group=4, topk_group=2, seed=46),
    # small-batch gate with W_g and the tokens' rows in shared memory (d >=
    # 1024, W_g rows of 16/32/64 bytes): bf16 E = 16 (4 tokens per CTA, a
    # ragged last CTA) and E = 32 (2 per CTA, group-limited); fp32 E = 4 (16
    # tokens per CTA, more than the 8 warps: each warp selects two) and E = 16
    # (soft gating)
    "smemgate_E16_T99_d1024_k2_f128": MoEConfig(
        "smemgate_E16_T99_d1024_k2_f128", T=99, d=1024, E=16, k=2, f=128, dtype="bf16",
        bias="normal", bias_var=0.5, seed=60),
    "smemgate_E32_T70_d2048_k4_f128_g8top2": MoEConfig(
        "smemgate_E32_T70_d2048_k4_f128_g8top2", T=70, d=2048, E=32, k=4, f=128,
        dtype="bf16", router=ROUTER_GROUP_LIMITED, n_group=8, topk_group=2, seed=61),
    "smemgate_f32_E4_T37_d1024_k2_f128": MoEConfig(
        "smemgate_f32_E4_T37_d1024_k2_f128", T=37, d=1024, E=4, k=2, f=128, dtype="f32",
        pre_k=4, seed=62),
    "smemgate_f32_E16_T50_d1024_f128_soft": MoEConfig(
        "smemgate_f32_E16_T50_d1024_f128_soft", T=50, d=1024, E=16, k=16, f=128, dtype="f32",
        router=ROUTER_SOFT_GUMBEL, tau=1.0, seed=63),
}
ALL = dict(SMALL)
ALL.update(CONFIGS)
ALL.update(VARIANTS)
SMALL_NAMES = list(SMALL)
FULL_NAMES = CONFIG_ORDER
VARIANT_NAMES = list(VARIANTS)
# configs whose whole-layer oracle is cheap enough to run on every token
ORACLE_FULL_OK = set(SMALL_NAMES) | {CONFIG_ORDER[0], CONFIG_ORDER[1]}


@functools.lru_cache(maxsize=2)
def layer(name: str):
    """(cfg, gpu inputs, host fp64 inputs) for a named shape."""
    cfg = ALL[name]
    inp = make(cfg)
    host = oracle.inputs_to_numpy({k: v for k, v in inp.items()})
    return cfg, inp, host


def make(cfg):
    from workloads import make_inputs
    return make_inputs(cfg, device="cuda")


@functools.lru_cache(maxsize=2)
def oracle_route(name: str):
    cfg, inp, host = layer(name)
    L = oracle.gate_logits(host["x"], host["Wg"], host["bias"])
    idx, w = oracle.route(L, cfg.k, cfg.router, cfg.pre_k, cfg.n_group, cfg.topk_group,
                          host.get("gumbel"), cfg.tau)
    return L, idx, w


@functools.lru_cache(maxsize=2)
def oracle_dispatch(name: str):
    cfg, _, _ = layer(name)
    _, idx, _ = oracle_route(name)
    return oracle.dispatch(idx, cfg.E)


def sample_rows(offsets: np.ndarray, max_experts: int = 6, per_expert: int = 6, seed: int = 0):
    """Rows to check per expert: first, last (the ragged tail of the last
    m-tile) and a few random ones, from a spread of non-empty experts."""
    rng = np.random.default_rng(seed)
    E = len(offsets) - 1
    nonempty = [e for e in range(E) if offsets[e + 1] > offsets[e]]
    if len(nonempty) > max_experts:
        pick = [nonempty[0], nonempty[-1]]
        counts = np.diff(offsets)
        pick.append(int(np.argmax(counts)))
        rest = [e for e in nonempty if e not in pick]
        pick += list(rng.choice(rest, size=max_experts - len(pick), replace=False))
        nonempty = sorted(set(int(e) for e in pick))
    rows = {}
    for e in nonempty:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        r = {lo, hi - 1}
        if hi - lo > 2:
            r |= set(int(v) for v in rng.integers(lo, hi, size=min(per_expert, hi - lo)))
        rows[e] = sorted(r)
    return rows


def payload_static(cfg):
    """The static payload scale of a shape, or None for per-token scales."""
    return cfg.payload_scale if int(cfg.payload_fp8) == 2 else None


@functools.lru_cache(maxsize=1)
def oracle_payload(name: str):
    """Per-token FP8 payload of the oracle: (q values, scales)."""
    cfg, _, host = layer(name)
    return oracle.quantize_payload_fp8(host["x"], payload_static(cfg))


def tile_class_experts(offsets: np.ndarray, bm: int = 256, tail_max: int = 32) -> dict:
    """One expert of each GEMM tile form, from a dispatch's offsets: the
    heaviest; the smallest whose rows end in a merged remainder (at least one
    full 256-row tile, then 1..32 rows); the smallest with a swapped remainder
    (33..255 rows after its full tiles, or fewer than 256 rows in all); the
    smallest with a single row. A form no expert has is left out."""
    counts = np.diff(np.asarray(offsets, np.int64))
    order = np.argsort(counts, kind="stable")
    out = {"heaviest": int(np.argmax(counts))}
    for e in order:
        c, e = int(counts[e]), int(e)
        rem = c % bm
        if c == 0:
            continue
        if "merged_tail" not in out and c > bm and 1 <= rem <= tail_max:
            out["merged_tail"] = e
        if "swapped_tail" not in out and rem > tail_max:
            out["swapped_tail"] = e
        if "one_row" not in out and c == 1:
            out["one_row"] = e
    return out


def tile_rows(offsets: np.ndarray, e: int, bm: int = 256) -> np.ndarray:
    """Routed rows of expert e in its first tile and in its last full tile
    plus remainder (all its rows when it has at most two tiles' worth)."""
    lo, hi = int(offsets[e]), int(offsets[e + 1])
    full = (hi - lo) // bm
    last = lo + max(full - 1, 0) * bm
    return np.unique(np.concatenate([np.arange(lo, min(hi, lo + bm)), np.arange(last, hi)]))


def targeted_tokens(offsets: np.ndarray, src: np.ndarray) -> np.ndarray:
    """Tokens routed to the first and last tiles of each expert that
    tile_class_experts picks (every such token, not a sample)."""
    rows = [tile_rows(offsets, e) for e in tile_class_experts(offsets).values()]
    return np.unique(np.asarray(src)[np.concatenate(rows)])
