"""Pins for the oracle's bf16 / FP8 E4M3 rounding and the FP8 payload.

The independent routines are torch's own dtype conversions (float32 ->
bfloat16, float32 -> float8_e4m3fn) and hand-worked values from the OCP E4M3
definition."""
import numpy as np
import pytest
import torch

from oracle import (round_to_bf16, e4m3_round_satfinite, e4m3_encode, e4m3_decode,
                    quantize_payload_fp8)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    # add exact ties: bf16 value plus half an ulp
    base = torch.randn(1000).to(torch.bfloat16).float().numpy()
    _, ex = np.frexp(base)
    ties = (base + np.ldexp(1.0, ex - 9)).astype(np.float32)
    v32 = np.concatenate([v32, ties])
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_to_bf16(v32.astype(np.float64))
    assert np.array_equal(got, ref)


def _all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


def test_e4m3_rounding_matches_torch_on_every_bf16_in_range():
    v = _all_bf16_values()
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_round_satfinite(v.astype(np.float64))
    assert np.array_equal(got, ref)
    # the sign of zero survives, as in the hardware conversion
    neg_tiny = v[(v < 0) & (np.abs(v) < 2.0 ** -10)].astype(np.float64)
    assert np.all(np.signbit(e4m3_round_satfinite(neg_tiny)))


def test_e4m3_rounding_matches_torch_on_fp32_grid():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-12, 6, 100000))).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(e4m3_round_satfinite(v.astype(np.float64)), ref)


def test_e4m3_handworked_values():
    cases = {
        448.0: 448.0, 449.0: 448.0, 464.0: 448.0, 1e9: 448.0, -500.0: -448.0,
        2.0 ** -9: 2.0 ** -9,            # smallest subnormal
        2.0 ** -10: 0.0,                 # tie between 0 and 2^-9 -> even (0)
        3 * 2.0 ** -11: 2.0 ** -9,       # 0.75 ulp rounds up
        2.0 ** -6: 2.0 ** -6,            # smallest normal
        1.0 + 1 / 16: 1.0,               # tie between 1 and 1.125 -> even (1)
        1.0 + 3 / 16: 1.25,              # tie between 1.125 and 1.25 -> even (1.25)
        240.0: 240.0, 248.0: 256.0,      # tie -> 256 (even mantissa)
        0.0: 0.0,
    }
    for v, q in cases.items():
        assert e4m3_round_satfinite(np.array([v]))[0] == q, v


def test_e4m3_encode_decode_match_torch_bit_patterns():
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = e4m3_decode(bits)
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    assert np.array_equal(dec[finite], ref[finite])
    assert np.array_equal(np.signbit(dec[finite]), np.signbit(ref[finite]))
    assert np.array_equal(e4m3_encode(dec[finite]), bits[finite])


def test_payload_scale_and_saturation():
    rng = np.random.default_rng(2)
    x = torch.randn(64, 256).to(torch.bfloat16).float().numpy().astype(np.float64)
    x[3] = 0.0
    x[5, 7] = 20.0
    q, s = quantize_payload_fp8(x)
    a = np.abs(x).max(1).astype(np.float32)
    exp_s = (a / np.float32(448.0)).astype(np.float32)
    exp_s[3] = 1.0
    assert np.array_equal(s, exp_s.astype(np.float64))
    assert np.all(q[3] == 0.0)
    nz = np.arange(64) != 3
    assert np.all(np.abs(q[nz]).max(1) == 448.0)
    # every payload value is an E4M3 value, and dequantisation is close
    assert np.array_equal(e4m3_round_satfinite(q), q)
    xh = q * s[:, None]
    rel = np.abs(xh[nz] - x[nz]).max(1) / np.abs(x[nz]).max(1)
    assert np.all(rel <= 2.0 ** -4)


def test_payload_quantisation_uses_fp32_division():
    """The payload value is E4M3(fp32(x / s)): check against torch doing the
    same fp32 division and its own E4M3 cast."""
    x = torch.randn(32, 128).to(torch.bfloat16).float()
    q, s = quantize_payload_fp8(x.numpy().astype(np.float64))
    st = torch.from_numpy(s.astype(np.float32))
    ref = (x / st[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(q, ref)


def test_payload_quotient_is_rounded_to_fp32_before_e4m3():
    """Rows whose second value lands, after the fp32 division, exactly on an
    E4M3 rounding midpoint, while the exact quotient lies just above it:
    s = fp32(1.875 / 448), 1.40625 / s = 336.0000107 exactly, fp32 336 (the
    midpoint of 320 and 352), which ties to the even code 320, where the
    exact quotient would round up to 352; likewise 168 between 160 and 176.
    (Rows found by searching bf16 pairs; the torch column repeats the fp32
    division and torch's own E4M3 cast.)"""
    x = np.array([[1.875, 1.40625], [4.3125, 1.6171875], [4.75, 1.78125]])
    q, s = quantize_payload_fp8(x)
    assert q.tolist() == [[448.0, 320.0], [448.0, 160.0], [448.0, 160.0]]
    exact = x[:, 1] / s                       # fp64: not on the midpoint
    assert np.all(exact > [336.0, 168.0, 168.0])
    xt = torch.from_numpy(x.astype(np.float32))
    st = torch.from_numpy(s.astype(np.float32))
    ref = (xt / st[:, None]).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(q, ref)


# ---- static global scale (the sync-tax article's "static global" FP8
# variant: one scale fixed ahead of time for the whole tensor)
def test_static_scale_equal_to_absmax_scale_reproduces_dynamic():
    x = torch.randn(1, 512).to(torch.bfloat16).float().numpy().astype(np.float64)
    qd, sd = quantize_payload_fp8(x)
    qs, ss = quantize_payload_fp8(x, static_scale=float(sd[0]))
    assert np.array_equal(qd, qs) and np.array_equal(sd, ss)


def test_static_scale_worked_values():
    # s = 0.5: 1 -> 2; 224 -> 448; 300 -> 600 saturates to 448; -2^-7 -> -2^-6
    # (exact: E4M3's smallest normal); 8.5 -> 17, halfway between 16 and 18
    # (spacing 2 at exponent 4) -> 16, the even mantissa; 9.5 -> 19 -> 20
    x = np.array([[1.0, 224.0, 300.0, -2.0 ** -7, 8.5, 9.5, -1000.0, 0.0]])
    q, s = quantize_payload_fp8(x, static_scale=0.5)
    assert s.tolist() == [0.5]
    assert q[0].tolist() == [2.0, 448.0, 448.0, -2.0 ** -6, 16.0, 20.0, -448.0, 0.0]


def test_static_scale_is_one_scale_for_every_row():
    rng = np.random.default_rng(5)
    x = torch.randn(16, 128).to(torch.bfloat16).float().numpy().astype(np.float64)
    x[2] = 0.0
    scale = float(np.float32(20.0 / 448.0))
    q, s = quantize_payload_fp8(x, static_scale=scale)
    assert np.all(s == np.float32(scale))            # the all-zero row too
    st = torch.full((16, 1), scale, dtype=torch.float32)
    ref = (torch.from_numpy(x).float() / st).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(q, ref.double().numpy())


@pytest.mark.parametrize("bad", [0.0, -1.0, float("inf"), float("nan")])
def test_static_scale_rejects_bad_values(bad):
    with pytest.raises(ValueError):
        quantize_payload_fp8(np.ones((2, 8)), static_scale=bad)
