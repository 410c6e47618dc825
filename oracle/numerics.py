"""Rounding to the storage formats the layer uses, written from the format
definitions (test infrastructure only; see oracle/__init__.py).

* bf16: IEEE-754 binary32 with the significand cut to 8 bits (1 implicit + 7
  stored), so a value v in [2^(e-1), 2^e) is a multiple of 2^(e-8).
* FP8 E4M3 "fn" from the OCP 8-bit floating point specification (v1.0): sign,
  4 exponent bits with bias 7, 3 mantissa bits; no infinities; the all-ones
  exponent with all-ones mantissa is NaN, so the largest finite value is
  1.75 * 2^8 = 448; subnormals are m/8 * 2^-6 (smallest 2^-9).

Rounding is to nearest, ties to even (numpy ``rint``); the FP8 cast saturates
to +-448 ("satfinite"), which is what the Deepseek-MoE sync-tax article's FP8
payload (section 3.1) needs since a per-token absmax scale maps every value
into range.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6   # 2^-6 is the smallest normal
E4M3_MANT_BITS = 3


def round_to_bf16(v) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    Valid for the normal range of bf16, which is all this layer produces."""
    v = np.asarray(v, dtype=np.float64)
    m, ex = np.frexp(v)            # v = m * 2^ex, 0.5 <= |m| < 1
    q = np.ldexp(np.rint(np.ldexp(m, 8)), ex - 8)
    return np.where(v == 0.0, v, q)


def round_to_f32(v) -> np.ndarray:
    """Round fp64 values to fp32 (IEEE round to nearest even), as fp64."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def e4m3_round_satfinite(v) -> np.ndarray:
    """Round fp64 values to E4M3 values (ties to even), saturating at +-448.

    Returns fp64 values that are exactly representable in E4M3; the sign of
    zero is kept (a negative input that rounds to zero gives -0.0)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)            # a in [2^(ex-1), 2^ex)
    # exponent of the value's binade, clamped at the subnormal range
    e = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, e - E4M3_MANT_BITS)
    r = np.rint(a / quantum) * quantum
    r = np.minimum(r, E4M3_MAX)
    r = np.where(a == 0.0, 0.0, r)
    return np.copysign(r, v)


def e4m3_encode(q) -> np.ndarray:
    """Bit patterns (uint8) of E4M3 values ``q`` (which must be representable)."""
    q = np.asarray(q, dtype=np.float64)
    sign = np.signbit(q).astype(np.uint8) << 7
    a = np.abs(q)
    _, ex = np.frexp(a)
    e = ex - 1                      # a in [2^e, 2^(e+1))
    normal = a >= np.ldexp(1.0, E4M3_MIN_NORMAL_EXP)
    # normal: a = (1 + m/8) 2^e, biased exponent e + 7
    m_norm = np.rint((np.ldexp(a, -np.where(normal, e, 0)) - 1.0) * 8.0)
    e_field = np.where(normal, e + 7, 0)
    # subnormal: a = m/8 * 2^-6 = m * 2^-9
    m_sub = np.rint(np.ldexp(a, 9))
    m_field = np.where(normal, m_norm, m_sub)
    bits = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    return (bits.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(b) -> np.ndarray:
    """Values (fp64) of E4M3 bit patterns ``b`` (uint8). 0x7f/0xff decode to NaN."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e_field = (b >> 3) & 0xF
    m_field = b & 0x7
    normal = np.ldexp(1.0 + m_field / 8.0, e_field - 7)
    sub = np.ldexp(m_field.astype(np.float64), -9)
    val = np.where(e_field == 0, sub, normal)
    val = np.where((e_field == 0xF) & (m_field == 0x7), np.nan, val)
    return s * val
