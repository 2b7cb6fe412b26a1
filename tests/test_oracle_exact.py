"""Pins for the oracle's exact fp32 summation and its order key.

The normaliser Z is the exact real sum of binary32 terms, rounded once to
the nearest binary32 (ties to even).  Python's exact rationals give that
value independently of the oracle's big-integer code.
"""
from fractions import Fraction
import math
import struct

import numpy as np


def _round_f32(x: Fraction) -> float:
    """Nearest binary32 to a non-negative rational, ties to even (Python ints only)."""
    if x == 0:
        return 0.0
    # binary32 values are integers times 2^-149; work in those units
    n = x * 2**149
    if n < 2**24:
        q, r = divmod(n.numerator, n.denominator)
        rem = Fraction(r, n.denominator)
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
            q += 1
        return math.ldexp(q, -149)
    e = 0
    while n >= 2**24:
        n /= 2
        e += 1
    q, r = divmod(n.numerator, n.denominator)
    rem = Fraction(r, n.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
        q += 1
    return math.ldexp(q, e - 149)


def _f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def test_exact_sum_random_wide_range(oracle_mod):
    rng = np.random.default_rng(0)
    for trial in range(40):
        n = int(rng.integers(1, 3000))
        expo = rng.uniform(-160, 0, size=n) if trial % 2 else rng.uniform(-30, 0, size=n)
        x = np.exp2(expo).astype(np.float32) * rng.uniform(0.5, 1, size=n).astype(np.float32)
        x[rng.random(n) < 0.05] = 0.0
        want = _round_f32(sum(Fraction(float(v)) for v in x))
        got = float(oracle_mod.exact_sum_f32(x))
        assert got == want, (trial, got, want)


def test_exact_sum_special_values(oracle_mod):
    tiny = np.float32(2.0**-149)
    cases = [
        [1.0],
        [0.0, 0.0],
        [tiny] * 7,
        [1.0] + [tiny] * 3,
        [1.0, 2.0**-24],                 # tie -> even (stays 1.0)
        [1.0 + 2.0**-23, 2.0**-24],      # tie -> even (rounds up)
        [1.0, 2.0**-24, tiny],           # just above the tie -> up
        [np.float32(0.1)] * 1000,
        [1.0] * 100000,
    ]
    for c in cases:
        x = np.array(c, np.float32)
        want = _round_f32(sum(Fraction(float(v)) for v in x))
        assert float(oracle_mod.exact_sum_f32(x)) == want, c


def test_exact_sum_is_order_independent_and_beats_naive(oracle_mod):
    rng = np.random.default_rng(5)
    x = np.exp(-rng.uniform(0, 40, size=20000)).astype(np.float32)
    a = float(oracle_mod.exact_sum_f32(x))
    b = float(oracle_mod.exact_sum_f32(x[::-1].copy()))
    c = float(oracle_mod.exact_sum_f32(rng.permutation(x)))
    assert a == b == c
    assert a == _f32(math.fsum(float(v) for v in x)) or abs(a - math.fsum(map(float, x))) <= 6e-8 * a


def test_orderkey_is_monotone(oracle_mod):
    vals = [-math.inf, -3.4e38, -1.0, -1e-30, -2.0**-149, -0.0, 0.0, 2.0**-149, 1e-30, 1.0,
            1.0000001, 3.4e38, math.inf]
    keys = [oracle_mod.orderkey(v) for v in vals]
    assert keys == sorted(keys) and len(set(keys)) == len(keys)
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(5000) * np.exp2(rng.integers(-60, 60, 5000))).astype(np.float32)
    k = np.array([oracle_mod.orderkey(float(v)) for v in x], np.uint64)
    order_k = np.argsort(k, kind="stable")
    assert np.all(np.diff(x[order_k]) >= 0)
