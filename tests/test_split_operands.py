"""The backward's bf16 tensor-core GEMMs carry each fp32 operand v as two
bf16 parts: hi = bf16(v), lo = bf16(v - hi). For v in [2^e, 2^(e+1)) the
difference v - hi is exact in fp32 and below 2^(e-8) in magnitude, so its
own bf16 rounding is off by at most 2^(e-17): |v - hi - lo| <= 2^-17 |v|.
Checked here with torch's fp32 -> bf16 rounding (round to nearest even), on
random fp32 values across the exponent range and on values built to sit
at the bound."""
import numpy as np
import torch


def _split(v32: np.ndarray):
    t = torch.from_numpy(v32)
    hi = t.to(torch.bfloat16).float()
    r = t - hi                                # exact in fp32
    lo = r.to(torch.bfloat16).float()
    return hi.double().numpy(), lo.double().numpy(), r.double().numpy()


def test_difference_is_exact_and_split_error_within_two_to_minus_17():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(400000) * np.exp2(rng.uniform(-60, 60, 400000))).astype(np.float32)
    v = v[v != 0]
    hi, lo, r = _split(v)
    v64 = v.astype(np.float64)
    assert np.array_equal(r, v64 - hi)        # v - hi needs no rounding
    err = np.abs(v64 - hi - lo)
    assert np.all(err <= 2.0 ** -17 * np.abs(v64))
    # and the bound is nearly reached: a split is not a wider format
    assert np.max(err / np.abs(v64)) > 2.0 ** -18


def test_bound_is_reached_just_above_a_power_of_two():
    # v = 2^e + r with r = 2^(e-9) (1 + 2^-8): r is under half a bf16 ulp of
    # 2^e (2^(e-8)), so hi = 2^e; r has nine significant bits, so its bf16
    # rounding is a tie, off by half its ulp, 2^(e-17): the bound itself
    for e in (-20, 0, 13):
        hi = 2.0 ** e
        r = 2.0 ** (e - 9) * (1 + 2.0 ** -8)
        v = np.array([hi + r], dtype=np.float64)
        assert float(np.float32(v[0])) == v[0]          # exactly an fp32 value
        h, lo, rr = _split(v.astype(np.float32))
        assert h[0] == hi and rr[0] == r
        err = abs(v[0] - h[0] - lo[0])
        assert err == 2.0 ** (e - 17)
        assert err <= 2.0 ** -17 * v[0]
