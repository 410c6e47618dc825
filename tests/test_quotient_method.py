"""The FP8 quantisers form x / s without a division per element: y = RN(1/s),
q = RN(x y), then two corrections q <- RN(q + RN(x - s q) y) with the
residual from an FMA (Markstein's theorem). This pins that claim on the CPU
with exact rational arithmetic (each fp32 operation rounded once, as the
hardware's FMA and multiply do): on quotients placed on and next to E4M3
rounding midpoints, and on random ones, for scales in the range the
kernels take this path for ([2^-64, 2^64]), the result is the IEEE fp32
quotient. The GPU tests check the kernels' payload bytes against the oracle
on every finite bf16 value; this checks the method they rely on."""
import random
import struct
from fractions import Fraction as F

import pytest


def rn32(v: F) -> F:
    """v rounded to the nearest fp32 value, ties to even (subnormals too)."""
    if v == 0:
        return F(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    if F(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    m = a / F(2) ** (e - 23)
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * F(fl) * F(2) ** (e - 23)


def f32(bits: int) -> F:
    return F(struct.unpack("<f", struct.pack("<I", bits))[0])


def bf16(bits: int) -> F:
    return f32(bits << 16)


def two_corrections(x: F, s: F) -> F:
    y = rn32(1 / s)
    q = rn32(x * y)
    for _ in range(2):
        r = rn32(x - s * q)
        q = rn32(q + r * y)
    return q


def test_rn32_against_struct():
    rng = random.Random(3)
    for _ in range(2000):
        v = rng.uniform(-1e30, 1e30) * 10 ** rng.randint(-40, 0)
        want = struct.unpack("<f", struct.pack("<f", v))[0]
        assert rn32(F(v)) == F(want)


# (x / s) near an E4M3 rounding midpoint: (m + 1/2) / 8 * 2^e for e in the
# E4M3 range, with s moved 0..3 fp32 steps either way
@pytest.mark.parametrize("seed", [0, 1])
def test_two_corrections_give_the_ieee_quotient_at_e4m3_midpoints(seed):
    rng = random.Random(seed)
    mids = [F(2 * m + 1, 16) * F(2) ** e for e in range(-9, 9) for m in range(8)]
    n = 0
    for _ in range(350):
        x = bf16(rng.randrange(0x2000, 0x7F80))     # positive normal bf16, x >= ~2^-64
        s0 = rn32(x / rng.choice(mids))
        e = s0.numerator.bit_length() - s0.denominator.bit_length()
        for k in range(-3, 4):
            s = s0 + k * F(2) ** (e - 24)
            if not (F(2) ** -64 <= s <= F(2) ** 64) or x / s > 1024 or x / s < F(2) ** -100:
                continue
            assert two_corrections(x, s) == rn32(x / s), (x, s)
            assert two_corrections(-x, s) == -rn32(x / s)
            n += 1
    assert n > 1000


def test_two_corrections_give_the_ieee_quotient_at_random():
    # every quotient that can decide an E4M3 code (2^-11 and above): exact
    rng = random.Random(7)
    n = 0
    for _ in range(3000):
        x = bf16(rng.randrange(0x3400, 0x4400))     # bf16 values from 2^-23 to 512
        s = rn32(F(rng.uniform(0.001, 30.0)) / 448)
        if x / s > 1024 or x / s < F(2) ** -11:
            continue
        assert two_corrections(x, s) == rn32(x / s), (x, s)
        n += 1
    assert n > 500


def test_tiny_quotients_stay_below_the_first_e4m3_boundary():
    # below 2^-11 the residual may underflow and the last bits differ, but
    # the result stays under 2^-10 (E4M3 code +-0) with the sign of x
    rng = random.Random(9)
    for _ in range(3000):
        x = bf16(rng.randrange(0x0001, 0x3000))    # down to bf16 subnormals
        s = rn32(F(rng.uniform(0.001, 30.0)) / 448)
        if x / s >= F(2) ** -11:
            continue
        q = two_corrections(x, s)
        assert 0 <= q < F(2) ** -10
        assert -F(2) ** -10 < two_corrections(-x, s) <= 0


def test_one_correction_is_not_enough():
    # the second correction matters: a single one leaves quotients one ulp
    # off the IEEE result
    rng = random.Random(11)
    mids = [F(2 * m + 1, 16) * F(2) ** e for e in range(-9, 9) for m in range(8)]
    off = 0
    for _ in range(3000):
        x = bf16(rng.randrange(0x2000, 0x7F80))
        s = rn32(x / rng.choice(mids))
        if not (F(2) ** -64 <= s <= F(2) ** 64) or x / s > 1024:
            continue
        y = rn32(1 / s)
        q = rn32(x * y)
        q1 = rn32(q + rn32(x - s * q) * y)
        off += q1 != rn32(x / s)
        off += q != rn32(x / s)
    assert off > 0
