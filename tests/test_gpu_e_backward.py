"""GPU parity of the backward pass (moe_backward through the C ABI) against
the fp64 oracle's backward.

Small layers (every router mode, fp32 and bf16, a single expert, experts
with no rows, ragged batches) are compared element by element on every
gradient; the 1024-token d=4096 E=8 layer on dx of sampled tokens. Both sides
start from the same inputs and dout; the routing is checked equal first.

Tolerances, from the arithmetic: the GPU sums in fp32 (fp32 FMA on fp32
layers; on bf16 layers fp32 accumulation on the tensor cores, with every
fp32 gradient operand carried as bf16 hi + lo, ~2^-17 relative) where the
oracle sums in fp64: relative errors ~sqrt(K) * 2^-24, K <= 4096, so fp32
layers are held to rel-L2 1e-4. bf16 layers carry the forward's stored
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
from backward_shapes import SHAPES
from workloads import get_config, make_inputs

pytestmark = pytest.mark.gpu



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
