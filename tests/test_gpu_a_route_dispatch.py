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


def _fp8_edge_rows(T, d, static_scale, seed):
    """bf16 rows whose quotients x / s sit where E4M3 rounding is delicate.
    Candidates are every positive bf16 value below the row's absmax (or
    below 1000 s with a static scale, so that some saturate); each row holds
    every candidate where x times the rounded reciprocal of s gives another
    E4M3 code than the IEEE quotient, up to 160 within 8 fp32 steps of a
    rounding midpoint, 40 in E4M3's subnormal range, two zeros and ordinary
    values, with random signs. A per-token row starts with its absmax, which
    fixes s = fp32(amax / 448); its absmax is the best of 8 draws for the
    number of such disagreements."""
    from oracle.numerics import e4m3_round_satfinite
    rng = np.random.default_rng(seed)
    pos_bf16 = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    pool = pos_bf16[(pos_bf16 > 1e-3) & (pos_bf16 < 1e3)]

    def classify(cand, s):
        y = (cand * np.float32(np.float32(1.0) / s)).astype(np.float32)
        q = (cand / s).astype(np.float32)
        wrong = e4m3_round_satfinite(y.astype(np.float64)) != e4m3_round_satfinite(q.astype(np.float64))
        low = (y.view(np.uint32) & 0xFFFFF).astype(np.int64)
        tiny = np.abs(q) < 2.0 ** -6
        near = (np.abs(low - 0x80000) <= 8) & ~tiny
        return wrong, near, tiny

    rows = np.zeros((T, d), np.float32)
    for t in range(T):
        if static_scale is None:
            best = None
            for amax in rng.choice(pool, 8):
                amax = np.float32(amax)
                s = np.float32(amax / np.float32(448.0))
                cand = pos_bf16[pos_bf16 <= amax]
                cls = classify(cand, s)
                if best is None or cls[0].sum() > best[3][0].sum():
                    best = (amax, s, cand, cls)
            amax, s, cand, (wrong, near, tiny) = best
        else:
            amax, s = None, np.float32(static_scale)
            cand = pos_bf16[pos_bf16 < np.float32(1000.0) * s]
            wrong, near, tiny = classify(cand, s)
        parts = [cand[wrong][:120]]
        for mask, n in ((near & ~wrong, 160), (tiny & ~wrong, 40)):
            c = cand[mask]
            parts.append(rng.choice(c, size=min(n, c.size), replace=False) if c.size else c)
        chosen = np.concatenate(parts)[: d - 3]
        row = rng.choice(cand[~tiny], size=d).astype(np.float32)
        row[3:3 + chosen.size] = chosen
        row[1:3] = 0.0
        row *= np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
        if amax is not None:
            row[0] = amax
        rows[t] = row
    return rows


# static scales 7 * 2^-9 and 13 * 2^-10: bf16 values exist whose product with
# 1/s takes another code than the quotient (30 and 1 of them)
def _every_bf16_rows(d, amax, rng):
    """Rows of width d that together hold every finite bf16 value of
    magnitude <= amax (all of them if amax is None), each with a random
    sign, zero-padded; with an amax each row starts with +amax, so a
    per-token scale is fp32(amax / 448) on every row."""
    mags = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    if amax is not None:
        mags = mags[mags <= np.float32(amax)]
    vals = mags * np.where(rng.random(mags.size) < 0.5, -1.0, 1.0).astype(np.float32)
    width = d if amax is None else d - 1
    n = -(-vals.size // width)
    body = np.zeros(n * width, np.float32)
    body[:vals.size] = vals
    body = body.reshape(n, width)
    if amax is None:
        return body
    return np.concatenate([np.full((n, 1), np.float32(amax), np.float32), body], 1)


# every bf16 value through the quantiser: static scales on both sides of the
# range where the quotient comes from a reciprocal and two corrections
# ([2^-64, 2^64]) and per-token scales from a few absmax values; rows held in
# registers (d <= 5120) and rows read twice (wider)
@pytest.mark.parametrize("d", [4096, 6144])
@pytest.mark.parametrize("static_scale", [None, 0.013671875, 0.02, 3.0, 2.0 ** -70, 2.0 ** 70])
def test_dispatch_fp8_every_bf16_value(cuda_ok, static_scale, d):
    from workloads import MoEConfig
    rng = np.random.default_rng(21)
    E, k = 4, 2
    if static_scale is None:
        rows = np.concatenate([_every_bf16_rows(d, a, rng)
                               for a in (20.0, 0.75, 448.0, 0.0029296875, 2.0 ** -100)])
    else:
        rows = _every_bf16_rows(d, None, rng)
    T = rows.shape[0]
    mode = True if static_scale is None else 2
    cfg = MoEConfig("fp8_every_bf16", T=T, d=d, E=E, k=k, f=128, dtype="bf16", pre_k=4,
                    payload_fp8=mode, payload_scale=static_scale or 0.0)
    x = torch.from_numpy(rows).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(rows))
    idx = np.stack([np.arange(T) % E, (np.arange(T) + 1) % E], 1).astype(np.int32)
    ws = moe.alloc_workspace(cfg, kind="scratch")
    dd = moe.dispatch(cfg, x.cuda(), torch.from_numpy(idx).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK
    _, _, _, src = oracle.dispatch(idx, E)
    q, s = oracle.quantize_payload_fp8(rows.astype(np.float64), static_scale)
    ref = oracle.e4m3_encode(q[src])
    got = to_np(dd["x_perm"])
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} payload bytes differ"
    got_s = to_np(dd["x_scale"]).astype(np.float32)
    assert np.array_equal(got_s.view(np.uint32), s[src].astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("static_scale", [None, 0.013671875, 0.0126953125])
def test_dispatch_fp8_payload_rounding_edges(cuda_ok, static_scale):
    # the payload bytes are those of the IEEE fp32 quotient on rows built
    # around the cases a shortcut (x times 1/s) would get wrong: E4M3
    # rounding midpoints, E4M3 subnormals, saturation
    from workloads import MoEConfig
    T, d, E, k = 96, 512, 4, 2
    mode = True if static_scale is None else 2
    cfg = MoEConfig("fp8_edges", T=T, d=d, E=E, k=k, f=128, dtype="bf16", pre_k=4,
                    payload_fp8=mode, payload_scale=static_scale or 0.0)
    rows = _fp8_edge_rows(T, d, static_scale, seed=11 if static_scale is None else 12)
    x = torch.from_numpy(rows).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(rows))      # the rows are bf16 values
    idx = np.stack([np.arange(T) % E, (np.arange(T) + 1 + np.arange(T) // E) % E], 1)
    idx[idx[:, 0] == idx[:, 1], 1] = (idx[idx[:, 0] == idx[:, 1], 1] + 1) % E
    ws = moe.alloc_workspace(cfg, kind="scratch")
    dd = moe.dispatch(cfg, x.cuda(), torch.from_numpy(idx.astype(np.int32)).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK
    _, _, _, src = oracle.dispatch(idx, E)
    q, s = oracle.quantize_payload_fp8(rows.astype(np.float64), static_scale)
    ref = oracle.e4m3_encode(q[src])
    got = to_np(dd["x_perm"])
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} payload bytes differ"
    got_s = to_np(dd["x_scale"]).astype(np.float32)
    assert np.array_equal(got_s.view(np.uint32), s[src].astype(np.float32).view(np.uint32))
