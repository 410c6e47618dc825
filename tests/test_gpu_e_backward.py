"""GPU parity of the backward pass (moe_backward through the C ABI) against
the fp64 oracle's backward.

Small layers (every router mode, fp32 and bf16, a single expert, experts
with no rows, ragged batches) are compared element by element on every
gradient. Two full-size layers, the 1024-token d=4096 E=8 one and a
2048-token copy of the 256-expert layer's shape (d=7168, f=2048, top-8 of 32
Zipf-skewed experts), are compared in full on the gate's gradients (dW_g,
db), on dW1 and dW2 of one expert of each GEMM tile form, and on dx of 256+
tokens. Both sides start from the same inputs and dout; the routing is
checked equal first.

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
from gpu_layers import tile_class_experts
from workloads import get_config, make_inputs

pytestmark = pytest.mark.gpu


def _dout(cfg, seed=5):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    t = torch.randn((cfg.T, cfg.d), generator=g, device="cuda", dtype=torch.float32)
    return t.to(torch.bfloat16 if cfg.dtype == "bf16" else torch.float32)


def _run_dev(cfg):
    """Forward then backward on the GPU; the gradients stay in device memory."""
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
    return inp, ws, dout, g


def _host(t):
    return t.cpu().numpy().astype(np.float64)


def _run(cfg):
    inp, ws, dout, g = _run_dev(cfg)
    return inp, ws, dout, {k: _host(v) for k, v in g.items()}


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


FULL_BWD = ["balanced_T1024_d4096_E8_k2_f11008", "skewed_small_T2048_d7168_E32_k8_f2048_zipf"]


@pytest.mark.parametrize("name", FULL_BWD)
def test_backward_full_layer(cuda_ok, name):
    cfg = get_config(name)
    inp, ws, dout, g = _run_dev(cfg)
    host = oracle.inputs_to_numpy(inp)
    fwd = oracle.forward(cfg, host, keep_h=False)
    views = moe.forward_views(cfg, ws)
    assert np.array_equal(views["topk_idx"].cpu().numpy(), fwd["topk_idx"])
    dout_h = dout.float().cpu().numpy()
    # the gate's gradients over every token
    r = oracle.backward_router(cfg, host, fwd, dout_h)
    _close(_host(g["dWg"]), r["dWg"], 2e-3, f"{name} dWg")
    _close(_host(g["dbias"]), r["dbias"], 2e-3, f"{name} dbias")
    # whole weight gradients of one expert of each tile form, and the lightest
    counts = np.diff(fwd["offsets"])
    pick = set(tile_class_experts(fwd["offsets"]).values())
    pick.add(int(np.argmin(np.where(counts > 0, counts, np.iinfo(np.int64).max))))
    for e in sorted(pick):
        pe = oracle.backward_expert(cfg, host, fwd, dout_h, e)
        _close(_host(g["dW1"][e]), pe["dW1"], 2e-3, f"{name} dW1[{e}] ({counts[e]} rows)")
        _close(_host(g["dW2"][e]), pe["dW2"], 2e-3, f"{name} dW2[{e}] ({counts[e]} rows)")
    # dx of 256 random tokens
    tokens = np.sort(np.random.default_rng(9).choice(cfg.T, 256, replace=False))
    ref = oracle.backward_tokens(cfg, host, dout_h, tokens)
    _close(_host(g["dx"][torch.from_numpy(tokens).cuda()]), ref["dx"], 2e-3, f"{name} dx")
    print(f"{name}: experts compared {sorted(pick)}")


def _fwd_bwd(cfg, inp, dout):
    ws = moe.alloc_workspace(cfg)
    out = moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                      noise=inp.get("gumbel"))
    bws = moe.alloc_workspace(cfg, "backward")
    g = moe.backward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], dout,
                     fwd_ws=ws, ws=bws, noise=inp.get("gumbel"))
    torch.cuda.synchronize()
    assert moe.get_device_error(bws) == moe.MOE_OK
    assert moe.get_device_error(ws) == moe.MOE_OK
    return out, moe.forward_views(cfg, ws), g


def _check_keep_z(cfg, rows_mode=0):
    """keep_z: the forward's output and H are the same bits, its Z is X_e W1_e
    (fp32 summation against the oracle's fp64), and the backward that reads
    it gives the same bits as the one that recomputes Z."""
    base = cfg.with_(x_perm_mode=rows_mode)
    inp = make_inputs(base, device="cuda")
    dout = _dout(base)
    out0, v0, g0 = _fwd_bwd(base, inp, dout)
    out1, v1, g1 = _fwd_bwd(base.with_(keep_z=1), inp, dout)
    assert v0["z"] is None and v1["z"] is not None
    assert torch.equal(out0, out1)
    assert torch.equal(v0["h"], v1["h"])
    for n in g0:
        assert torch.equal(g0[n], g1[n]), n
    host = oracle.inputs_to_numpy(inp)
    off = v1["offsets"].cpu().numpy()
    src = v1["src"].cpu().numpy()
    z = _host(v1["z"])
    ref = np.zeros_like(z)
    for e in range(cfg.E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            ref[lo:hi] = host["x"][src[lo:hi]] @ oracle.moe_oracle._expert(host["W1"], e)
    _close(z, ref, 1e-5, "Z")


@pytest.mark.parametrize("name", list(SHAPES))
def test_keep_z_matches_recompute(cuda_ok, name):
    _check_keep_z(SHAPES[name])


# merged remainder tiles (256-feature tiles: 270 rows per expert, a 14-row
# remainder; 257 rows, a 1-row remainder), packed and gathered rows: the
# epilogue's remainder path writes Z too
@pytest.mark.parametrize("rows_mode", [1, 2])
@pytest.mark.parametrize("name", ["merged_tail_T270_d256_E2_k2_f320",
                                  "merged_tail_T257_d128_E1_k1_f256"])
def test_keep_z_merged_tail_tiles(cuda_ok, name, rows_mode):
    from gpu_layers import SMALL
    _check_keep_z(SMALL[name].with_(gemm_tile_n=256), rows_mode)


# the 256-expert layer's shape at 2048 tokens: 512-feature W1 tiles, merged
# and swapped remainders; packed and gathered rows (the gathered W1 pass
# writes Z from the same epilogue)
@pytest.mark.parametrize("rows_mode", [1, 2])
def test_keep_z_matches_recompute_full_layer(cuda_ok, rows_mode):
    _check_keep_z(get_config("skewed_small_T2048_d7168_E32_k8_f2048_zipf"), rows_mode)


# a training step (the forward keeping Z, then the backward) captured in one
# CUDA graph: no host synchronisation inside either call; replays give the
# eager results bit for bit, also after a new batch is copied into the
# captured input buffer
@pytest.mark.parametrize("name", ["bwd_bf16_T129_d256_E8_k2_f320", "bwd_f32_T50_d64_E5_k2_f128",
                                  "bwd_soft_T100_d256_E8_f128"])
def test_training_step_in_cuda_graph(cuda_ok, name):
    cfg = SHAPES[name].with_(keep_z=1)
    inp = make_inputs(cfg, device="cuda")
    dout = _dout(cfg)
    out0, _, g0 = _fwd_bwd(cfg, inp, dout)
    x = inp["x"].clone()
    ws = moe.alloc_workspace(cfg)
    bws = moe.alloc_workspace(cfg, "backward")
    out = torch.empty_like(out0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        moe.forward(cfg, x, inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws, out=out,
                    noise=inp.get("gumbel"), stream=s)
        grads = moe.backward(cfg, x, inp["Wg"], inp["bias"], inp["W1"], inp["W2"], dout,
                             fwd_ws=ws, ws=bws, noise=inp.get("gumbel"), stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out0)
    for n in g0:
        assert torch.equal(grads[n], g0[n]), n
    x2 = torch.flip(inp["x"], dims=[0]).contiguous()
    x.copy_(x2)
    graph.replay()
    torch.cuda.synchronize()
    out1, _, g1 = _fwd_bwd(cfg, dict(inp, x=x2), dout)
    assert torch.equal(out, out1)
    for n in g1:
        assert torch.equal(grads[n], g1[n]), n
    assert moe.get_device_error(bws) == moe.MOE_OK
    assert moe.get_device_error(ws) == moe.MOE_OK


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


@pytest.mark.parametrize("name", ["bwd_bf16_T129_d256_E8_k2_f320", "bwd_skew_T256_d128_E64_k8_f128_zipf",
                                  "bwd_ragged_T96_d192_E3_k2_f448"])
def test_backward_after_gathered_forward(cuda_ok, name):
    # a forward that gathers its rows leaves no packed rows behind: the
    # backward packs them itself and gives the same gradients, bit for bit
    base = SHAPES[name]
    grads = []
    for mode in (moe.MOE_XPERM_PACKED, moe.MOE_XPERM_GATHERED):
        _, _, _, g = _run(base.with_(x_perm_mode=mode))
        grads.append(g)
    for n in grads[0]:
        assert np.array_equal(grads[0][n], grads[1][n]), n
