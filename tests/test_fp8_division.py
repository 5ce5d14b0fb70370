"""The quotient x / s of the FP8 quantizer, checked in exact arithmetic (CPU).

The quantizer codes E4M3(RN32(x / s)) (oracle.fp8: an fp32 division).  The CUDA
kernel takes y = RN32(1/s) once per block and forms each quotient with one
multiply and four FMAs (two residual corrections; Markstein's theorem makes the
last one the rounded quotient).  This test runs that sequence with every
operation rounded exactly like fp32 (rational arithmetic, round to nearest even)
and requires RN32(x / s) on random and adversarial operands: quotients next to
fp32 rounding midpoints, scales with all-ones significands, and the ends of the
scale range the kernel takes this path for (2^-60 <= s <= 2^100).
"""
import math
import random
from fractions import Fraction

import numpy as np


def rn32(v: Fraction) -> Fraction:
    """v rounded to the nearest fp32 value, ties to even (no overflow handling)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length() - 24
    while a >= Fraction(2) ** (e + 24):
        e += 1
    while a < Fraction(2) ** (e + 23):
        e -= 1
    e = max(e, -149)                      # the subnormal grid
    m = a / Fraction(2) ** e
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * Fraction(2) ** e


def method(x: Fraction, s: Fraction) -> Fraction:
    y = rn32(1 / s)
    q0 = rn32(x * y)
    r0 = rn32(x - s * q0)                 # an FMA rounds the exact residual once
    q1 = rn32(q0 + r0 * y)
    r1 = rn32(x - s * q1)
    return rn32(q1 + r1 * y)


def f32(v: float) -> Fraction:
    return Fraction(float(np.float32(v)))


def test_rn32_matches_numpy_float32():
    """rn32 of exact fp64 values against numpy's fp64 -> fp32 conversion (round to
    nearest even), including exact ties and subnormal results."""
    rng = random.Random(1)
    vals = [rng.uniform(-1, 1) * 2.0 ** rng.randint(-150, 120) for _ in range(3000)]
    vals += [float((2 ** 24 + 2 * k + 1) * 2.0 ** -25) for k in range(50)]      # ties between fp32 neighbours
    vals += [2.0 ** -149 * 1.5, 2.0 ** -149 * 2.5, 2.0 ** -150, -3 * 2.0 ** -151]
    for v in vals:
        assert rn32(Fraction(v)) == Fraction(float(np.float32(v))), v


def test_corrected_reciprocal_quotient_is_the_rounded_quotient():
    rng = random.Random(7)
    cases = []
    for _ in range(3000):                 # random blocks: s = RN32(amax / 448), |x| <= amax
        amax = f32(abs(rng.gauss(0, 1)) * 2.0 ** rng.randint(-50, 90) + 1e-30)
        s = rn32(amax / 448)
        x = rn32(amax * Fraction(rng.random()) * rng.choice((-1, 1)))
        cases.append((x, s))
    for _ in range(3000):                 # quotients next to fp32 midpoints
        s = f32(2.0 ** rng.randint(-60, 100) * (1 + rng.random()))
        e = rng.randint(-10, 8)
        mid = (Fraction(rng.getrandbits(23) + 2 ** 23) + Fraction(1, 2)) * Fraction(2) ** (e - 23)
        x = rn32(mid * s)
        cases.append((x, s))
    for k in range(24):                   # all-ones significands, both ends of the range
        for s in (Fraction(2 ** 24 - 1) * Fraction(2) ** (-60 - 23 + k), Fraction(2 ** 24 - 1) * Fraction(2) ** (100 - 24)):
            s = rn32(s)
            for x in (s * 448, s * Fraction(2 ** 24 - 1, 2 ** 24), s / 1024, -s * Fraction(3, 7)):
                cases.append((rn32(x), s))
    bad = [(x, s) for x, s in cases if method(x, s) != rn32(x / s)]
    assert not bad, f"{len(bad)} of {len(cases)} quotients differ; first {bad[0]}"
    # the cases are hard: the uncorrected product x * RN32(1/s) misses hundreds of them
    assert sum(rn32(x * rn32(1 / s)) != rn32(x / s) for x, s in cases) > 100
