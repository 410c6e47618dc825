"""GPU parity of the grouped expert FFN (tcgen05 for bf16, fp32 FMA for fp32)
and of the combine, each fed with oracle-derived inputs so errors do not
cascade from earlier stages."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_routed_gb300 as moe
from gpu_layers import (SMALL_NAMES, FULL_NAMES, layer, oracle_route, oracle_dispatch,
                        oracle_payload, sample_rows, tile_class_experts)
from parity_util import (assert_close, assert_close_bf16_stored, out_tolerance, to_np,
                         BF16_REL_L2, BF16_MAX_ABS)

pytestmark = pytest.mark.gpu
NAMES = SMALL_NAMES + FULL_NAMES


def _ffn_inputs(cfg, inp, host, src, name):
    """Packed rows in the oracle's order, and the fp64 rows the experts see."""
    src_t = torch.from_numpy(src.astype(np.int64)).cuda()
    if cfg.router == 3:
        # soft gating: every expert reads x itself
        return inp["x"], None, host["x"]
    if cfg.payload_fp8:
        q, s = oracle_payload(name)
        payload = torch.from_numpy(oracle.e4m3_encode(q[src])).cuda()
        scale = torch.from_numpy(s[src].astype(np.float32)).cuda()
        return payload, scale, q * s[:, None]
    return inp["x"][src_t].contiguous(), None, host["x"]


@pytest.mark.parametrize("name", NAMES)
def test_expert_ffn_parity(cuda_ok, name, gemm_tile_n=0):
    cfg, inp, host = layer(name)
    counts, offsets, pos, src = oracle_dispatch(name)
    x_perm, x_scale, x_hat = _ffn_inputs(cfg, inp, host, src, name)
    off_t = torch.from_numpy(offsets.astype(np.int32)).cuda()
    ws = moe.alloc_workspace(cfg, kind="scratch")
    h, y = moe.expert_ffn(cfg.with_(gemm_tile_n=gemm_tile_n), x_perm, x_scale, off_t, inp["W1"],
                          inp["W2"], ws=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK
    storage = "bf16" if cfg.dtype == "bf16" else "f32"
    rel, mabs = (BF16_REL_L2, BF16_MAX_ABS) if cfg.dtype == "bf16" else out_tolerance(cfg)
    full = cfg.R <= 4096
    rows = {e: list(range(int(offsets[e]), int(offsets[e + 1]))) for e in range(cfg.E)
            if offsets[e + 1] > offsets[e]} if full else sample_rows(offsets)
    if not full:
        # every row of one expert of each tile form (the heaviest; a merged,
        # a swapped and a one-row remainder), besides the sampled rows
        for e in tile_class_experts(offsets).values():
            rows[e] = list(range(int(offsets[e]), int(offsets[e + 1])))
    for e, rs in rows.items():
        rs = np.asarray(rs)
        W1e = oracle.moe_oracle._expert(inp["W1"], e)
        W2e = oracle.moe_oracle._expert(inp["W2"], e)
        y_ref, h_ref = oracle.expert_ffn_rows(x_hat[src[rs]], W1e, W2e, storage)
        rs_t = torch.from_numpy(rs).cuda()
        if storage == "bf16":
            assert_close_bf16_stored(to_np(h[rs_t]), h_ref, rel, mabs, f"{name} H expert {e}")
        else:
            assert_close(to_np(h[rs_t]), h_ref, rel, mabs, f"{name} H expert {e}")
        assert_close(to_np(y[rs_t]), y_ref, rel, mabs, f"{name} Y expert {e}")


@pytest.mark.parametrize("name", NAMES)
def test_combine_parity(cuda_ok, name):
    cfg, inp, host = layer(name)
    _, idx_o, w_o = oracle_route(name)
    counts, offsets, pos, src = oracle_dispatch(name)
    # any fixed fp32 rows stand in for Y: the combine is checked on its own
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    Y = torch.randn((cfg.R, cfg.d), generator=g, device="cuda", dtype=torch.float32)
    ws = moe.alloc_workspace(cfg, kind="scratch")
    out = moe.combine(cfg, Y, torch.from_numpy(pos.astype(np.int32)).cuda(),
                      torch.from_numpy(w_o.astype(np.float32)).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK
    toks = np.arange(cfg.T)
    if cfg.T * cfg.d > (1 << 24):
        toks = np.sort(np.random.default_rng(7).choice(cfg.T, 512, replace=False))
    # the oracle combine over the sampled tokens only (their k rows of Y)
    rows = pos.reshape(cfg.T, cfg.k)[toks].reshape(-1)
    Ys = to_np(Y[torch.from_numpy(rows).cuda()]).astype(np.float64)
    ref = oracle.combine(Ys, np.arange(rows.size), w_o[toks].astype(np.float32).astype(np.float64))
    out = out[torch.from_numpy(toks).cuda()]
    if cfg.dtype == "bf16":
        # fp32 accumulation then one bf16 rounding: within one bf16 ulp
        got = to_np(out).astype(np.float64)
        tol = np.abs(ref) * 2.0 ** -8 + 1e-6
        assert np.all(np.abs(got - ref) <= tol)
    else:
        assert_close(to_np(out), ref, 1e-6, 1e-5, name)


def test_combine_flags_bad_position(cuda_ok):
    name = SMALL_NAMES[0]
    cfg, inp, _ = layer(name)
    _, idx_o, w_o = oracle_route(name)
    _, _, pos, _ = oracle_dispatch(name)
    pos = pos.astype(np.int32).copy()
    pos[5] = cfg.R + 3
    ws = moe.alloc_workspace(cfg, kind="scratch")
    Y = torch.ones((cfg.R, cfg.d), dtype=torch.float32, device="cuda")
    out = moe.combine(cfg, Y, torch.from_numpy(pos).cuda(),
                      torch.from_numpy(w_o.astype(np.float32)).cuda(), ws=ws)
    assert moe.get_device_error(ws) == moe.MOE_ERR_BAD_INDEX
    t = 5 // cfg.k
    j = 5 % cfg.k
    expect = w_o[t].sum() - w_o[t, j]
    assert abs(float(out[t, 0].float()) - expect) < 1e-2


def test_ffn_skips_empty_experts_and_flags_bad_offsets(cuda_ok):
    name = SMALL_NAMES[0]
    cfg, inp, host = layer(name)
    counts, offsets, pos, src = oracle_dispatch(name)
    x_perm, x_scale, _ = _ffn_inputs(cfg, inp, host, src, name)
    ws = moe.alloc_workspace(cfg, kind="scratch")
    # NaN weights for an expert with no rows are never read
    W1 = inp["W1"].clone()
    off = offsets.astype(np.int32).copy()
    e_empty = 2
    shift = off[e_empty + 1] - off[e_empty]
    off[e_empty + 1] = off[e_empty]      # expert 2 now owns no rows; its rows go to nobody
    W1[e_empty] = float("nan")
    h, y = moe.expert_ffn(cfg, x_perm, x_scale, torch.from_numpy(off).cuda(), W1, inp["W2"], ws=ws)
    assert moe.get_device_error(ws) == moe.MOE_OK
    assert shift >= 0
    assert torch.isfinite(y[:int(off[-1])]).all()
    # decreasing offsets are rejected on the device, nothing is computed
    bad = off.copy()
    bad[1], bad[2] = bad[2] + 1, bad[1]
    y2 = torch.full_like(y, 7.0)
    moe.expert_ffn(cfg, x_perm, x_scale, torch.from_numpy(bad).cuda(), inp["W1"], inp["W2"],
                   ws=ws, y_perm=y2)
    assert moe.get_device_error(ws) == moe.MOE_ERR_BAD_INDEX


# both pair-tile widths on shapes whose default is the other one: 512-feature
# tiles (two MMAs per k-step, one accumulator) on small layers with swapped
# tails and ragged last feature blocks, 256-feature tiles on the one full
# layer that defaults to 512
WIDTH_CASES = [(n, w) for n in ("wide_tile_T300_d1024_E2_k2_f1600",
                                "wide_tile_fp8_T520_d1024_E4_k1_f1024",
                                "ragged_T129_d256_E8_k2_f320",
                                "gate_E192_T300_d320_k4_f128") for w in ("512", "256")]
WIDTH_CASES.append((FULL_NAMES[4], "256"))


@pytest.mark.parametrize("name,width", WIDTH_CASES)
def test_expert_ffn_tile_width(cuda_ok, name, width):
    test_expert_ffn_parity(cuda_ok, name, gemm_tile_n=int(width))
