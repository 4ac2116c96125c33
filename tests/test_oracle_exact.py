"""Pins for the exact double-double GEMM oracle (oracle.exact_dd_gemm).

The oracle is the plain definition: X = sum_k (a_hi + a_lo)(b_hi + b_lo)
formed exactly, rounded once to the nearest double double ("Multiple Double
Arithmetic on NVIDIA Tensor Cores", Definition 1.1 and Section 2, step 5).
It is pinned here to exact rational brute force (Python Fractions), to closed
forms, and to invariants that hold bit for bit.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.exact_ref import bits, exact_entry, nearest_dd, pow2, rne

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_rne_matches_python_float_conversion():
    # The Fraction rounding used below agrees with CPython's correctly rounded
    # int/int division on normal, subnormal and tie cases.
    rng = np.random.default_rng(7)
    cases = [Fraction(1) + pow2(-53), Fraction(1) + 3 * pow2(-53), pow2(-1075), 3 * pow2(-1076),
             pow2(-1074) * Fraction(5, 2), Fraction(-7, 3), Fraction(10**30, 7)]
    for _ in range(500):
        n = int(rng.integers(1, 2**62)) * int(rng.integers(1, 2**62))
        d = 1 << int(rng.integers(0, 1200))
        cases.append(Fraction(n, d) * (1 if rng.random() < 0.5 else -1))
    for x in cases:
        assert bits(rne(x)) == bits(float(x)), x


def _special_dd(rng):
    kind = rng.integers(0, 9)
    if kind == 0:
        hi = rng.uniform(-1, 1)
        lo = hi * 2.0**-53 * rng.uniform(-1, 1)
    elif kind == 1:
        hi = math.ldexp(1.0, int(rng.integers(-60, 60))) * (1 if rng.random() < .5 else -1)
        lo = hi * 2.0**-53 * (1 if rng.random() < .5 else -1)   # |lo| = ulp(hi)/2
    elif kind == 2:
        hi = math.ldexp(float(rng.integers(1, 2**40)), -1074)     # subnormal
        lo = 0.0
    elif kind == 3:
        hi, lo = 0.0, 0.0
    elif kind == 4:
        hi = rng.uniform(-1, 1) * 2.0**500
        lo = hi * 2.0**-53 * rng.uniform(-1, 1)
    elif kind == 5:
        hi = rng.uniform(-1, 1) * 2.0**-500
        lo = hi * 2.0**-53 * rng.uniform(-1, 1)
    elif kind == 6:
        hi = rng.uniform(0.5, 1)
        lo = -hi * 2.0**-54 * rng.uniform(0, 1)                   # opposite signs
    elif kind == 7:
        hi = float(rng.integers(-2**20, 2**20))
        lo = 0.0
    else:
        hi = rng.normal() * 2.0 ** int(rng.integers(-30, 30))
        lo = hi * 2.0**-53 * rng.normal()
    s = hi + lo
    bb = s - hi
    return s, (hi - (s - bb)) + (lo - bb)


def _dd_matrix(rng, r, c):
    hi = np.zeros((r, c))
    lo = np.zeros((r, c))
    for i in range(r):
        for j in range(c):
            hi[i, j], lo[i, j] = _special_dd(rng)
    return hi, lo


@pytest.mark.parametrize("seed", range(150))
def test_bruteforce_tiny(seed):
    rng = np.random.default_rng(1000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 7, 3))
    A_hi, A_lo = _dd_matrix(rng, M, K)
    B_hi, B_lo = _dd_matrix(rng, K, N)
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    for i in range(M):
        for j in range(N):
            h, l = nearest_dd(exact_entry(A_hi, A_lo, B_hi, B_lo, i, j))
            assert bits(C_hi[i, j]) == bits(h), (i, j, C_hi[i, j], h)
            assert bits(C_lo[i, j]) == bits(l), (i, j, C_lo[i, j], l)


@pytest.mark.parametrize("terms,expect", [
    # 1 + 2^-53: tie in hi, even -> 1; lo = 2^-53
    ([1.0, 2.0**-53], (1.0, 2.0**-53)),
    # 1 + 3*2^-53: tie in hi, even -> 1 + 2^-51; lo = -2^-53
    ([1.0, 3 * 2.0**-53], (1.0 + 2.0**-51, -2.0**-53)),
    # 1 + 2^-60 + 2^-113: tie in lo, even -> 2^-60
    ([1.0, 2.0**-60, 2.0**-113], (1.0, 2.0**-60)),
    # 1 + (2^-60 + 2^-112) + 2^-113: tie in lo, even -> 2^-60 + 2^-111
    ([1.0, 2.0**-60 + 2.0**-112, 2.0**-113], (1.0, 2.0**-60 + 2.0**-111)),
    # exact cancellation -> (+0, +0)
    ([0.75, -0.75], (0.0, 0.0)),
    # subnormal sum
    ([2.0**-1074, 2.0**-1074, 2.0**-1073], (2.0**-1072, 0.0)),
])
def test_ties_and_cancellation(terms, expect):
    K = len(terms)
    A_hi = np.array([terms])
    A_lo = np.zeros((1, K))
    B_hi = np.ones((K, 1))
    B_lo = np.zeros((K, 1))
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert bits(C_hi[0, 0]) == bits(expect[0])
    assert bits(C_lo[0, 0]) == bits(expect[1])


@pytest.mark.parametrize("K", [1, 3, 64, 1000, 4097])
def test_closed_form_constant(K):
    # (1 + 2^-60)^2 summed K times = K + K 2^-59 + K 2^-120, whose nearest dd is
    # (K, K 2^-59): K 2^-59 < ulp(K)/2 and K 2^-120 < ulp(K 2^-59)/2.
    A_hi = np.ones((3, K))
    A_lo = np.full((3, K), 2.0**-60)
    B_hi = np.ones((K, 2))
    B_lo = np.full((K, 2), 2.0**-60)
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.all(C_hi == K)
    assert np.all(C_lo == K * 2.0**-59)


def _random_dd(rng, r, c):
    hi = rng.uniform(-1, 1, (r, c)) * np.ldexp(1.0, rng.integers(-8, 8, (r, c)))
    lo = hi * 2.0**-53 * rng.uniform(-1, 1, (r, c))
    s = hi + lo
    bb = s - hi
    return s, (hi - (s - bb)) + (lo - bb)


def _same(x, y):
    return np.array_equal(x.view(np.int64), y.view(np.int64))


def test_identity_and_permutation():
    rng = np.random.default_rng(3)
    M, K = 13, 21
    A_hi, A_lo = _random_dd(rng, M, K)
    I = np.eye(K)
    Z = np.zeros((K, K))
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, I, Z)
    assert _same(C_hi, A_hi + 0.0) and _same(C_lo, A_lo + 0.0)
    Pm = np.eye(M)[rng.permutation(M)]
    C_hi, C_lo = oracle.exact_dd_gemm(Pm, np.zeros((M, M)), A_hi, A_lo)
    assert _same(C_hi, Pm @ A_hi + 0.0) and _same(C_lo, Pm @ A_lo + 0.0)


def test_invariants():
    rng = np.random.default_rng(4)
    M, N, K = 11, 9, 37
    A_hi, A_lo = _random_dd(rng, M, K)
    B_hi, B_lo = _random_dd(rng, K, N)
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    # transposition: (AB)^T = B^T A^T
    T_hi, T_lo = oracle.exact_dd_gemm(B_hi.T, B_lo.T, A_hi.T, A_lo.T)
    assert _same(T_hi, C_hi.T.copy()) and _same(T_lo, C_lo.T.copy())
    # power-of-two scaling and negation are exact
    S_hi, S_lo = oracle.exact_dd_gemm(A_hi * 2.0**37, A_lo * 2.0**37, -B_hi, -B_lo)
    assert _same(S_hi, -C_hi * 2.0**37 + 0.0) and _same(S_lo, -C_lo * 2.0**37 + 0.0)
    # order of k does not matter
    p = rng.permutation(K)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi[:, p], A_lo[:, p], B_hi[p], B_lo[p])
    assert _same(R_hi, C_hi) and _same(R_lo, C_lo)
    # row / column selection returns the same entries
    rows, cols = np.array([7, 0, 3]), np.array([8, 1])
    E_hi, E_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=rows, cols=cols)
    assert _same(E_hi, C_hi[np.ix_(rows, cols)]) and _same(E_lo, C_lo[np.ix_(rows, cols)])
    # thread count does not matter
    U_hi, U_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, threads=1)
    assert _same(U_hi, C_hi) and _same(U_lo, C_lo)


def test_output_is_normalised_and_close_to_float_product():
    rng = np.random.default_rng(5)
    A_hi, A_lo = _random_dd(rng, 16, 50)
    B_hi, B_lo = _random_dd(rng, 50, 12)
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.all(np.abs(C_lo) <= np.spacing(np.abs(C_hi)) / 2)
    ref = A_hi @ B_hi
    assert np.allclose(C_hi, ref, rtol=1e-12, atol=1e-12)


def test_empty_and_zero_k():
    z = np.zeros((3, 0))
    C_hi, C_lo = oracle.exact_dd_gemm(z, z, np.zeros((0, 4)), np.zeros((0, 4)))
    assert C_hi.shape == (3, 4) and np.all(C_hi == 0) and np.all(C_lo == 0)
    assert not np.signbit(C_hi).any()


def test_rejects_non_finite():
    A = np.array([[np.inf]])
    with pytest.raises(ValueError):
        oracle.exact_dd_gemm(A, np.zeros((1, 1)), np.ones((1, 1)), np.zeros((1, 1)))
