"""Pins for the oracle's FP8 expert-output payload (CPU only).

The Deepseek-MoE sync-tax article (section 3.1) quantises each token's
expert output vector on its own, from its min and max, by an affine map.
The oracle's reading: zero = the midpoint of [min, max], s = half the range
/ 448, q = E4M3((y - zero) / s), decoded as q * s + zero. The pins use
hand-worked rows, torch's own float8_e4m3fn cast of the same fp32 division,
the E4M3 rounding bound, and the combine of the decoded rows."""
import numpy as np
import torch

import oracle
from oracle import quantize_output_fp8, dequantize_output_fp8


def test_worked_row():
    # min -1, max 3: zero 1, half-range 2, s = fp32(2/448);
    # (y - zero)/s = -448, 448, 0, -112 (all E4M3 values)
    y = np.array([[-1.0, 3.0, 1.0, 0.5]])
    q, s, z = quantize_output_fp8(y)
    assert z.tolist() == [1.0]
    assert s.tolist() == [float(np.float32(2.0) / np.float32(448.0))]
    assert q[0].tolist() == [-448.0, 448.0, 0.0, -112.0]
    yh = dequantize_output_fp8(q, s, z)
    assert np.max(np.abs(yh - y)) < 1e-6


def test_constant_rows_decode_exactly():
    y = np.array([[2.5] * 8, [0.0] * 8, [-7.0] * 8])
    q, s, z = quantize_output_fp8(y)
    assert np.all(q == 0.0) and np.all(s == 1.0)
    assert z.tolist() == [2.5, 0.0, -7.0]
    assert np.array_equal(dequantize_output_fp8(q, s, z), y)


def test_matches_torch_e4m3_cast_of_the_fp32_division():
    g = torch.Generator().manual_seed(3)
    y = (torch.randn(64, 256, generator=g) * torch.rand(64, 1, generator=g) * 5
         + torch.randn(64, 1, generator=g))
    q, s, z = quantize_output_fp8(y.double().numpy())
    mn, mx = y.min(1).values, y.max(1).values
    zt = mx * 0.5 + mn * 0.5
    ht = mx * 0.5 - mn * 0.5
    st = ht / 448.0
    assert np.array_equal(z, zt.double().numpy())
    assert np.array_equal(s, st.double().numpy())
    ref = ((y - zt[:, None]) / st[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(q, ref.double().numpy())


def test_extremes_map_to_the_ends_and_error_bound():
    rng = np.random.default_rng(4)
    y = (rng.standard_normal((50, 300)) * rng.uniform(0.01, 30, (50, 1))
         + rng.uniform(-5, 5, (50, 1))).astype(np.float32).astype(np.float64)
    q, s, z = quantize_output_fp8(y)
    assert np.all(np.abs(q).max(axis=1) == 448.0)
    r = (y - z[:, None]) / s[:, None]
    # E4M3: half an ulp is 2^-4 of the value for normals, 2^-10 below 2^-6
    bound = s[:, None] * (2.0 ** -4 * np.abs(r) + 2.0 ** -10) + 1e-6 * (np.abs(y) + np.abs(z)[:, None])
    assert np.all(np.abs(dequantize_output_fp8(q, s, z) - y) <= bound)


def test_forward_combines_the_decoded_outputs():
    from workloads import MoEConfig, make_inputs
    cfg = MoEConfig("t", T=24, d=64, E=4, k=2, f=64, dtype="bf16", pre_k=4, seed=9)
    inp = make_inputs(cfg)
    plain = oracle.forward(cfg, inp)
    fq = oracle.forward(cfg.with_(output_fp8=1), inp)
    # the payload is the quantisation of the fp32-rounded expert outputs
    q, s, z = quantize_output_fp8(plain["Y"])
    assert np.array_equal(fq["y_q"], q) and np.array_equal(fq["y_scale"], s)
    ref = oracle.combine(dequantize_output_fp8(q, s, z), plain["pos"], plain["topk_w"])
    assert np.array_equal(fq["out"], ref)
    # and it stays close to the unquantised layer (E4M3 keeps ~2^-4 relative)
    rel = np.linalg.norm(fq["out"] - plain["out"]) / np.linalg.norm(plain["out"])
    assert 0 < rel < 0.05
    # the per-token path agrees with the whole-layer one
    toks = np.array([0, 5, 23])
    ft = oracle.forward_tokens(cfg.with_(output_fp8=1), inp, toks)
    np.testing.assert_allclose(ft["out"], fq["out"][toks], rtol=0, atol=1e-12)
