"""Pins of the oracle's integer primitives against properties that the
mathematics fixes (nearest-integer rounding, floor square root, the dyadic
normalisation) and against float64 for the shift-based exp (DetLLM README,
"Layout": intmath rounding rules, DI-Exp)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def test_rshr_is_nearest_ties_up_exhaustive_small():
    xs, ss = np.meshgrid(np.arange(-1024, 1025), np.arange(0, 13))
    xs, ss = xs.ravel(), ss.ravel()
    r = oracle.rshr(xs, ss)
    for x, s, v in zip(xs.tolist(), ss.tolist(), r.tolist()):
        exact = Fraction(x, 2 ** s)
        diff = exact - v
        assert abs(diff) <= Fraction(1, 2), (x, s, v)
        if abs(diff) == Fraction(1, 2):
            assert v > exact, (x, s, v)  # ties go toward +infinity


def test_rshr_random_wide():
    rng = np.random.default_rng(1)
    x = rng.integers(-(2 ** 61), 2 ** 61, size=4000, dtype=np.int64)
    s = rng.integers(0, 63, size=4000).astype(np.int32)
    r = oracle.rshr(x, s)
    for xi, si, v in zip(x.tolist(), s.tolist(), r.tolist()):
        exact = Fraction(xi, 2 ** si)
        assert abs(exact - v) <= Fraction(1, 2)
        if abs(exact - v) == Fraction(1, 2):
            assert v > exact


def test_isqrt_matches_math_isqrt_and_definition():
    rng = np.random.default_rng(2)
    vals = list(rng.integers(0, 2 ** 62, size=3000, dtype=np.int64).tolist())
    for k in [0, 1, 2, 3, 4, 2 ** 31 - 1, 2 ** 31, 3037000499]:
        vals += [k * k, max(0, k * k - 1), k * k + 1]
    vals += [2 ** 62 - 1, 2 ** 63 - 1, 2 ** 64 - 1]
    r = oracle.isqrt(np.array(vals, dtype=np.uint64))
    for n, v in zip(vals, r.tolist()):
        assert v == math.isqrt(n)
        assert v * v <= n < (v + 1) * (v + 1)


def test_dyadic_normalised_and_rounded():
    rng = np.random.default_rng(3)
    # the operand range the quantisers produce: N < 2^40, D < 2^32, and
    # N/D >= 2^-25 (every shift within [-40, 40])
    N = rng.integers(1, 2 ** 40, size=6000, dtype=np.int64)
    D = rng.integers(1, 2 ** 32, size=6000, dtype=np.int64)
    N[:10] = [1, 1, 127, 2 ** 40 - 1, 5, 2 ** 14, 2 ** 15, 3, 1, 2 ** 39]
    D[:10] = [1, 2 ** 20, 127, 1, 127 * 3000, 1, 1, 3, 127, 127]
    keep = np.array([d.bit_length() - n.bit_length() <= 24 for n, d in zip(N.tolist(), D.tolist())])
    N, D = N[keep], D[keep]
    m, k = oracle.dyadic(N, D)
    for n_, d_, mi, ki in zip(N.tolist(), D.tolist(), m.tolist(), k.tolist()):
        x = Fraction(n_, d_) * (Fraction(2) ** ki)
        assert Fraction(2 ** 14) <= x < Fraction(2 ** 15), (n_, d_, ki)
        assert abs(x - mi) <= Fraction(1, 2)
        if abs(x - mi) == Fraction(1, 2):
            assert mi > x
        assert 2 ** 14 <= mi <= 2 ** 15


def test_exp2q_against_float64_exhaustive():
    delta = np.arange(-26 * 1024, 1, dtype=np.int64)
    e = oracle.exp2q(delta).astype(np.float64)
    ref = 2.0 ** 15 * np.exp2(delta / 1024.0)
    # relative error of the cubic on [0,1) is below 2^-13; the final
    # rounding shift adds at most one unit
    assert np.all(np.abs(e - ref) <= ref * 2.0 ** -13 + 1.0)
    assert e[-1] == 2 ** 15                       # 2^0
    assert np.all(np.diff(e) >= 0)                # monotone non-decreasing
    assert np.all(e[delta <= -24 * 1024] == 0)
    assert np.all(e >= 0) and np.all(e <= 2 ** 15)


def test_exp2q_integer_points_are_exact_powers():
    for i in range(0, 16):
        assert oracle.exp2q(np.array([-1024 * i]))[0] == 2 ** (15 - i)


def test_requant_is_nearest_ties_up():
    rng = np.random.default_rng(4)
    n = 3000
    acc = rng.integers(-(127 * 127 * 8192), 127 * 127 * 8192, size=n, dtype=np.int64)
    mt = rng.integers(2 ** 14, 2 ** 15 + 1, size=n).astype(np.int32)
    kt = rng.integers(8, 40, size=n).astype(np.int32)
    mc = rng.integers(2 ** 14, 2 ** 15, size=n).astype(np.int32)
    out = oracle.requant(acc, mt, kt, mc, 12)
    for a, m1, k1, m2, y in zip(acc.tolist(), mt.tolist(), kt.tolist(), mc.tolist(), out.tolist()):
        exact = Fraction(a * m1 * m2, 2 ** (k1 + 22 - 12))
        assert abs(exact - y) <= Fraction(1, 2)
        if abs(exact - y) == Fraction(1, 2):
            assert y > exact


def test_bound_violation_is_reported():
    # a shift outside [0, 62] is a bound violation, reported, not a crash
    with pytest.raises(oracle.OracleError):
        oracle.rshr(np.array([5]), np.array([70]))
