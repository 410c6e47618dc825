"""GPU parity of the backward pass (moe_backward through the C ABI) against
the fp64 oracle's backward.

Small layers (every router mode, fp32 and bf16, a single expert, experts
with no rows, ragged batches) are compared element by element on every
gradient; the 1024-token d=4096 E=8 layer on dx of sampled tokens. Both sides
start from the same inputs and dout; the routing is checked equal first.

Tolerances, from the arithmetic: the GPU sums in fp32 (fp32 FMA, or fp32
accumulation on the tensor cores for the recomputed pre-activation Z) where
the oracle sums in fp64: relative errors ~sqrt(K) * 2^-24, K <= 4096, so
fp32 layers are held to rel-L2 1e-4. bf16 layers carry the forward's stored
bf16 H into dW2 (and dw through Y): H values next to a bf16 rounding midpoint
round one way on the GPU and the other in the oracle (the same flips the
forward's 2e-3 output bound allows for), so bf16 layers get that forward
bound, rel-L2 2e-3. Max-abs errors are bounded at 10x those fractions of the
tensor's largest magnitude."""
import numpy as np
import pytest
import torch

import mixture_experts_routed_gb300 as moe
import oracle
from workloads import MoEConfig, ROUTER_GROUP_LIMITED, ROUTER_PREK_SOFTMAX, \
    ROUTER_SOFT_GUMBEL, get_config, make_inputs

pytestmark = pytest.mark.gpu

SHAPES = {
    "bwd_bf16_T129_d256_E8_k2_f320": MoEConfig(
        "bwd_bf16_T129_d256_E8_k2_f320", T=129, d=256, E=8, k=2, f=320, dtype="bf16",
        bias="normal", bias_var=0.5, seed=70),
    "bwd_f32_T50_d64_E5_k2_f128": MoEConfig(
        "bwd_f32_T50_d64_E5_k2_f128", T=50, d=64, E=5, k=2, f=128, dtype="f32", pre_k=5,
        seed=71),
    "bwd_prek_T200_d256_E64_k2_f128": MoEConfig(
        "bwd_prek_T200_d256_E64_k2_f128", T=200, d=256, E=64, k=2, f=128, dtype="bf16",
        router=ROUTER_PREK_SOFTMAX, bias="normal", bias_var=0.5, seed=72),
    "bwd_group_T300_d256_E16_k2_f128": MoEConfig(
        "bwd_group_T300_d256_E16_k2_f128", T=300, d=256, E=16, k=2, f=128, dtype="bf16",
        router=ROUTER_GROUP_LIMITED, n_group=4, topk_group=2, seed=73),
    "bwd_soft_T100_d256_E8_f128": MoEConfig(
        "bwd_soft_T100_d256_E8_f128", T=100, d=256, E=8, k=8, f=128, dtype="bf16",
        router=ROUTER_SOFT_GUMBEL, tau=0.7, seed=74),
    "bwd_soft_f32_T64_d128_E4_f128": MoEConfig(
        "bwd_soft_f32_T64_d128_E4_f128", T=64, d=128, E=4, k=4, f=128, dtype="f32", pre_k=4,
        router=ROUTER_SOFT_GUMBEL, tau=1.0, seed=75),
    "bwd_single_T70_d128_E1_k1_f192": MoEConfig(
        "bwd_single_T70_d128_E1_k1_f192", T=70, d=128, E=1, k=1, f=192, dtype="bf16", pre_k=1,
        seed=76),
    "bwd_skew_T256_d128_E64_k8_f128_zipf": MoEConfig(
        "bwd_skew_T256_d128_E64_k8_f128_zipf", T=256, d=128, E=64, k=8, f=128, dtype="bf16",
        bias="zipf", zipf_s=3.0, seed=77),
    "bwd_tiny_fp32_layer": get_config("tiny_T256_d128_E8_k2_f256_fp32"),
    # one token: most experts have no rows
    "bwd_one_token_T1_d64_E4_k2_f64": MoEConfig(
        "bwd_one_token_T1_d64_E4_k2_f64", T=1, d=64, E=4, k=2, f=64, dtype="bf16", pre_k=4,
        seed=78),
    # d = 192, f = 448: pair tiles whose odd half is partly or wholly past M / N
    "bwd_ragged_T96_d192_E3_k2_f448": MoEConfig(
        "bwd_ragged_T96_d192_E3_k2_f448", T=96, d=192, E=3, k=2, f=448, dtype="bf16",
        pre_k=3, seed=79),
    # E = 128: both gate GEMMs on the tensor cores; experts of a few rows
    "bwd_gate_tc_T160_d128_E128_k4_f64": MoEConfig(
        "bwd_gate_tc_T160_d128_E128_k4_f64", T=160, d=128, E=128, k=4, f=64, dtype="bf16",
        bias="normal", bias_var=0.5, seed=80),
    # a single expert of exactly 128 rows (whole 64-row blocks, no tail)
    "bwd_whole_blocks_T128_d128_E1_k1_f128": MoEConfig(
        "bwd_whole_blocks_T128_d128_E1_k1_f128", T=128, d=128, E=1, k=1, f=128,
        dtype="bf16", pre_k=1, seed=81),
}


def _dout(cfg, seed=5):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    t = torch.randn((cfg.T, cfg.d), generator=g, device="cuda", dtype=torch.float32)
    return t.to(torch.bfloat16 if cfg.dtype == "bf16" else torch.float32)


def _run(cfg):
    inp = make_inputs(cfg, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                noise=inp.get("gumbel"))
    dout = _dout(cfg)
    bws = moe.alloc_workspace(cfg, "backward")
    g = moe.backward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], dout,
                     fwd_ws=ws, ws=bws, noise=inp.get("gumbel"))
    torch.cuda.synchronize()
    assert moe.get_device_error(bws) == moe.MOE_OK
    assert moe.get_device_error(ws) == moe.MOE_OK
    return inp, ws, dout, {k: v.cpu().numpy().astype(np.float64) for k, v in g.items()}


def _close(got, ref, rel, name):
    err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mabs = np.abs(got - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err <= rel and mabs <= 10 * rel * max(scale, 1e-30), (name, err, mabs, scale)


@pytest.mark.parametrize("name", list(SHAPES))
def test_backward_matches_oracle(cuda_ok, name):
    cfg = SHAPES[name]
    inp, ws, dout, g = _run(cfg)
    host = oracle.inputs_to_numpy(inp)
    ref_f = oracle.forward(cfg, host)
    idx = moe.forward_views(cfg, ws)["topk_idx"].cpu().numpy()
    assert np.array_equal(idx, ref_f["topk_idx"])
    ref = oracle.backward(cfg, host, ref_f, dout.float().cpu().numpy())
    rel = 1e-4 if cfg.dtype == "f32" else 2e-3
    for n in ("dx", "dWg", "dbias", "dW1", "dW2"):
        _close(g[n], ref[n], rel, n)


def test_backward_sampled_tokens_full_layer(cuda_ok):
    cfg = get_config("balanced_T1024_d4096_E8_k2_f11008")
    inp, ws, dout, g = _run(cfg)
    host = oracle.inputs_to_numpy(inp)
    tokens = [0, 1, 511, 777, 1023]
    ref = oracle.backward_tokens(cfg, host, dout.float().cpu().numpy(), tokens)
    idx = moe.forward_views(cfg, ws)["topk_idx"].cpu().numpy()[tokens]
    assert np.array_equal(idx, ref["topk_idx"])
    _close(g["dx"][tokens], ref["dx"], 2e-3, "dx")
    # properties at full size: an expert's dW is zero exactly when it has no rows
    counts = moe.forward_views(cfg, ws)["counts"].cpu().numpy()
    for e in range(cfg.E):
        assert (counts[e] == 0) == (not np.any(g["dW1"][e]))


def test_backward_is_bitwise_reproducible(cuda_ok):
    cfg = SHAPES["bwd_prek_T200_d256_E64_k2_f128"]
    _, _, _, g1 = _run(cfg)
    _, _, _, g2 = _run(cfg)
    for n in g1:
        assert np.array_equal(g1[n], g2[n]), n


def test_backward_rejects_fp8_payloads(cuda_ok):
    cfg = get_config("wide_fp8_T16384_d5120_E16_k2_f1536").with_(T=64)
    inp = make_inputs(cfg, device="cuda")
    ws = moe.alloc_workspace(cfg)
    bws = moe.alloc_workspace(cfg, "backward")
    with pytest.raises(moe.MoEError):
        moe.backward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], _dout(cfg),
                     fwd_ws=ws, ws=bws)
