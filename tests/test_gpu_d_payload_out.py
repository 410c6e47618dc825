"""GPU parity of the FP8 expert-output payload stages (through the C ABI):
the per-row min/max affine quantiser must match the oracle's bytes, scales
and zero points bit for bit on the same fp32 rows; the FP8 combine must
match the oracle's combine of the decoded rows."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_routed_gb300 as moe
from gpu_layers import layer, oracle_route, oracle_dispatch
from parity_util import to_np

pytestmark = pytest.mark.gpu


def _rows(R, d, seed):
    """Seeded fp32 rows with varied offsets and ranges, a constant row, an
    all-zero row and a row with one huge outlier."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    y = torch.randn((R, d), generator=g, device="cuda", dtype=torch.float32)
    y.mul_(torch.rand((R, 1), generator=g, device="cuda") * 10 + 1e-3)
    y.add_(torch.randn((R, 1), generator=g, device="cuda") * 3)
    if R > 3:
        y[1] = 2.5
        y[2] = 0.0
        y[3, d // 2] = 1e4
    return y


# widths for each quantiser form: a warp per row (d <= 1024 or > 8192), a CTA
# per row holding 2, 4 or 8 float4 per thread (ragged last pass at 1088,
# 1536 and 5120)
@pytest.mark.parametrize("R,d", [(1, 64), (9, 128), (300, 512), (2049, 1024), (37, 1088),
                                 (300, 1536), (64, 4096), (33, 8192), (5, 8256),
                                 (32768, 5120)])
def test_quantize_output_bit_exact(cuda_ok, R, d):
    cfg = moe.make_config(T=R, d=d, E=1, k=1, f=64, pre_k=1, output_fp8=1)
    y = _rows(R, d, seed=R)
    yq, ys, yz = moe.quantize_output(cfg, y)
    torch.cuda.synchronize()
    rows = np.arange(R) if R <= 4096 else np.sort(
        np.random.default_rng(1).choice(R, 2048, replace=False))
    yh = to_np(y[torch.from_numpy(rows).cuda()]).astype(np.float64)
    q, s, z = oracle.quantize_output_fp8(yh)
    got = to_np(yq)[rows]
    ref = oracle.e4m3_encode(q)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"
    assert np.array_equal(to_np(ys)[rows].view(np.uint32), s.astype(np.float32).view(np.uint32))
    assert np.array_equal(to_np(yz)[rows].view(np.uint32), z.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("name", ["outfp8_T300_d512_E4_k2_f256", "outfp8_f32_T64_d128_E4_k3_f128",
                                  "outfp8_T100_d256_E16_k8_f128",
                                  "wide_fp8_T16384_d5120_E16_k2_f1536_outfp8"])
def test_combine_fp8_parity(cuda_ok, name):
    cfg, _, _ = layer(name)
    _, idx_o, w_o = oracle_route(name)
    _, _, pos, _ = oracle_dispatch(name)
    R = cfg.R
    # a seeded payload: every finite E4M3 byte (0x7f and 0xff, the NaN codes,
    # moved to their finite neighbours), scales and zero points per row
    rng = np.random.default_rng(5)
    qb = rng.integers(0, 256, size=(R, cfg.d), dtype=np.uint8)
    qb[(qb & 0x7F) == 0x7F] -= 1
    s = rng.uniform(1e-3, 0.1, size=R).astype(np.float32)
    z = rng.standard_normal(R).astype(np.float32)
    w32 = w_o.astype(np.float32)
    ws = moe.alloc_workspace(cfg, kind="scratch")
    out = moe.combine_fp8(cfg, torch.from_numpy(qb).cuda(), torch.from_numpy(s).cuda(),
                          torch.from_numpy(z).cuda(), torch.from_numpy(pos.astype(np.int32)).cuda(),
                          torch.from_numpy(w32).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK
    toks = np.arange(cfg.T) if cfg.T <= 4096 else np.sort(rng.choice(cfg.T, 512, replace=False))
    rows = pos.reshape(cfg.T, cfg.k)[toks].reshape(-1)
    yhat = oracle.dequantize_output_fp8(oracle.e4m3_decode(qb[rows]), s[rows].astype(np.float64),
                                        z[rows].astype(np.float64))
    ref = oracle.combine(yhat, np.arange(rows.size), w32[toks].astype(np.float64))
    got = to_np(out[torch.from_numpy(toks).cuda()]).astype(np.float64)
    # fp32 decode (one fma) and accumulation, then the output rounding
    mag = np.einsum("tj,tjc->tc", np.abs(w32[toks]), np.abs(yhat.reshape(len(toks), cfg.k, -1)))
    tol = 1e-6 * mag + 1e-7
    if cfg.dtype == "bf16":
        tol = tol + np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(got - ref) <= tol)


def test_combine_fp8_flags_bad_position(cuda_ok):
    name = "outfp8_T300_d512_E4_k2_f256"
    cfg, _, _ = layer(name)
    _, _, w_o = oracle_route(name)
    _, _, pos, _ = oracle_dispatch(name)
    pos = pos.astype(np.int32).copy()
    pos[5] = cfg.R + 3
    ws = moe.alloc_workspace(cfg, kind="scratch")
    yq = torch.zeros((cfg.R, cfg.d), dtype=torch.uint8, device="cuda")   # E4M3 zero
    ys = torch.ones(cfg.R, dtype=torch.float32, device="cuda")
    yz = torch.ones(cfg.R, dtype=torch.float32, device="cuda")          # every row decodes to 1
    out = moe.combine_fp8(cfg, yq, ys, yz, torch.from_numpy(pos).cuda(),
                          torch.from_numpy(w_o.astype(np.float32)).cuda(), ws=ws)
    assert moe.get_device_error(ws) == moe.MOE_ERR_BAD_INDEX
    t, j = 5 // cfg.k, 5 % cfg.k
    assert abs(float(out[t, 0].float()) - (w_o[t].sum() - w_o[t, j])) < 1e-2
    assert abs(float(out[t + 1, 0].float()) - w_o[t + 1].sum()) < 1e-2


def test_quantize_output_empty_batch(cuda_ok):
    cfg = moe.make_config(T=0, d=128, E=4, k=2, f=64, pre_k=4, output_fp8=1)
    y = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    yq, ys, yz = moe.quantize_output(cfg, y)
    torch.cuda.synchronize()
    assert yq.shape == (0, 128) and ys.numel() == 0
