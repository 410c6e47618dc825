"""GPU parity of the router and the dispatch against the oracle (through the
C ABI). Routing follows the near-tie protocol; dispatch is fed the oracle's
routing so its outputs must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_routed_gb300 as moe
from gpu_layers import (SMALL_NAMES, FULL_NAMES, VARIANT_NAMES, layer, oracle_route,
                        oracle_dispatch, payload_static)
from parity_util import check_route, bits, to_np

pytestmark = pytest.mark.gpu
NAMES = SMALL_NAMES + FULL_NAMES + VARIANT_NAMES


@pytest.mark.parametrize("name", NAMES)
def test_route_parity(cuda_ok, name):
    cfg, inp, host = layer(name)
    idx, w, logits = moe.route(cfg, inp["x"], inp["Wg"], inp["bias"], noise=inp.get("gumbel"),
                               want_logits=True)
    torch.cuda.synchronize()
    L, idx_o, w_o = oracle_route(name)
    n_tie = check_route(cfg, L, idx_o, w_o, to_np(logits), to_np(idx), to_np(w))
    print(f"{name}: near-tie tokens {n_tie}")
    if cfg.router in (0, 2, 3):   # weights that sum to one
        assert np.all(np.abs(to_np(w).sum(1) - 1.0) <= 1e-6)


@pytest.mark.parametrize("name", NAMES)
def test_route_without_bias_pointer_equals_zero_bias(cuda_ok, name):
    cfg, inp, _ = layer(name)
    if cfg.bias != "zero":
        pytest.skip("shape has a bias")
    a = moe.route(cfg, inp["x"], inp["Wg"], None, noise=inp.get("gumbel"))
    b = moe.route(cfg, inp["x"], inp["Wg"], inp["bias"], noise=inp.get("gumbel"))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("name", NAMES)
def test_dispatch_parity(cuda_ok, name):
    cfg, inp, host = layer(name)
    _, idx_o, _ = oracle_route(name)
    counts, offsets, pos, src = oracle_dispatch(name)
    ws = moe.alloc_workspace(cfg, kind="scratch")
    idx_t = torch.from_numpy(idx_o.astype(np.int32)).cuda()
    d = moe.dispatch(cfg, inp["x"], idx_t, ws=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK
    assert np.array_equal(to_np(d["counts"]), counts)
    assert np.array_equal(to_np(d["offsets"]), offsets)
    assert np.array_equal(to_np(d["pos"]), pos)
    assert np.array_equal(to_np(d["src"]), src)
    R = cfg.R
    rows = np.arange(R) if R <= 300000 else np.random.default_rng(0).choice(R, 8192, replace=False)
    if cfg.router == 3:
        assert d["x_perm"] is None      # soft gating packs no rows
    elif not cfg.payload_fp8:
        # packed row r is the bytes of token src[r]
        got = bits(d["x_perm"][torch.from_numpy(rows).cuda()])
        ref = bits(inp["x"][torch.from_numpy(src[rows]).cuda()])
        assert np.array_equal(got, ref)
    else:
        q, s = oracle.quantize_payload_fp8(host["x"], payload_static(cfg))
        ref_bytes = oracle.e4m3_encode(q[src[rows]])
        got_bytes = to_np(d["x_perm"])[rows]
        assert np.array_equal(got_bytes, ref_bytes), \
            f"{int((got_bytes != ref_bytes).sum())} payload bytes differ"
        got_s = to_np(d["x_scale"])[rows].astype(np.float32)
        assert np.array_equal(got_s.view(np.uint32), s[src[rows]].astype(np.float32).view(np.uint32))


def test_dispatch_flags_bad_index_without_faulting(cuda_ok):
    cfg, inp, _ = layer(SMALL_NAMES[0])
    _, idx_o, _ = oracle_route(SMALL_NAMES[0])
    idx = idx_o.astype(np.int32).copy()
    idx[3, 1] = cfg.E          # out of range
    idx[10, 0] = -7
    ws = moe.alloc_workspace(cfg, kind="scratch")
    d = moe.dispatch(cfg, inp["x"], torch.from_numpy(idx).cuda(), ws=ws)
    assert moe.get_device_error(ws) == moe.MOE_ERR_BAD_INDEX
    pos = to_np(d["pos"])
    assert pos[3 * cfg.k + 1] == -1 and pos[10 * cfg.k + 0] == -1
    assert to_np(d["offsets"])[-1] == cfg.R - 2
    # the error word was cleared by the read
    assert moe.get_device_error(ws) == moe.MOE_OK


def test_dispatch_empty_batch(cuda_ok):
    from workloads import MoEConfig
    cfg = MoEConfig("empty", T=0, d=128, E=4, k=2, f=128, dtype="bf16", pre_k=4)
    ws = moe.alloc_workspace(cfg, kind="scratch")
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    counts = torch.full((4,), 99, dtype=torch.int32, device="cuda")
    offsets = torch.full((5,), 99, dtype=torch.int32, device="cuda")
    d = moe.dispatch(cfg, x, idx, ws=ws, counts=counts, offsets=offsets)
    assert to_np(d["counts"]).tolist() == [0] * 4
    assert to_np(d["offsets"]).tolist() == [0] * 5
