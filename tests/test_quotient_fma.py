"""The quantizer's divide-free quotient, checked on the CPU with exact rational
arithmetic: for a divisor y with at most 11 significant bits (an fp16 scale, or
the constants 3 and 15), q0 = fl(d * fl(1/y)) corrected once,
q1 = fl(q0 + fl(d - q0 * y) * fl(1/y)) (each fl(. + . * .) a single rounding, as an
FMA), equals the IEEE fp32 quotient fl(d / y) for every fp32 d; and fl(q1 + 1.5 * 2^23)
holds rint(q1) (round half to even) in its low bits. The cases include quotients
built to lie on exact rounding ties and next to fp32 rounding midpoints."""
from fractions import Fraction

import numpy as np
import pytest


def rn32(x: Fraction) -> float:
    """x rounded to the nearest fp32 value, ties to even (normal range)."""
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    scaled = x / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return float(sign * Fraction(m) * Fraction(2) ** (e - 23))


def fma32(a: float, b: float, c: float) -> float:
    return rn32(Fraction(a) * Fraction(b) + Fraction(c))


def quotient(d: float, y: float) -> float:
    r = rn32(1 / Fraction(y))
    q0 = rn32(Fraction(d) * Fraction(r))
    return fma32(fma32(q0, -y, d), r, q0)


def ieee_div(d: float, y: float) -> float:
    return float(np.float32(d) / np.float32(y))


def fp16_divisors(rng, n):
    bits = rng.integers(0x0400, 0x7C00, size=n).astype(np.uint16)   # positive normal fp16
    return [float(v) for v in bits.view(np.float16).astype(np.float32)]


def test_against_ieee_division_random():
    rng = np.random.default_rng(7)
    ys = fp16_divisors(rng, 300) + [3.0, 15.0]
    for y in ys:
        qs = rng.uniform(-1.0, 17.0, size=20)
        for q in qs:
            d = float(np.float32(q * y))
            if d == 0.0:
                continue
            assert quotient(d, y) == ieee_div(d, y), (d, y)


def test_ties_and_near_midpoints():
    """d = fl(y * h) for half-integers h (exact ties when representable) and the fp32
    neighbours of such d: the quotients the tie check used to send to the divide."""
    rng = np.random.default_rng(11)
    for y in fp16_divisors(rng, 200) + [3.0, 15.0]:
        for h in (0.5, 1.5, 2.5, 3.5, 7.5, 14.5):
            d0 = np.float32(h * y)
            for d in (d0, np.nextafter(d0, np.float32(np.inf)), np.nextafter(d0, np.float32(0))):
                d = float(d)
                q1 = quotient(d, y)
                assert q1 == ieee_div(d, y), (d, y)
                # round half to even through the magic constant
                t = rn32(Fraction(q1) + Fraction(12582912))
                assert int(t) - 12582912 == int(np.rint(np.float32(q1))), (q1, t)


@pytest.mark.parametrize("top", [3.0, 15.0])
def test_scale_division_by_constant(top):
    """s32 = (hi - lo) / (2^b - 1) for ranges of bf16 extremes and arbitrary fp32 values."""
    rng = np.random.default_rng(int(top))
    vals = list(rng.standard_normal(400).astype(np.float32) * 10) + \
        list(rng.uniform(0, 1e4, 200).astype(np.float32))
    for v in vals:
        v = abs(float(v))
        if v == 0.0:
            continue
        assert quotient(v, top) == ieee_div(v, top), (v, top)
