"""Pins for the comparator's model (oracle.simt_dd): exact product errors
against rational arithmetic, the error-free sum, accuracy against the exact
oracle, exactness on short integers, and planted mistakes."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from oracle import simt_dd

rng0 = np.random.default_rng(0)


def check_two_prod(err_fn):
    rng = np.random.default_rng(1)
    a = rng.normal(size=500) * np.ldexp(1.0, rng.integers(-400, 400, 500))
    b = rng.normal(size=500) * np.ldexp(1.0, rng.integers(-400, 400, 500))
    p = a * b
    e = err_fn(a, b, p)
    for x, y, pp, ee in zip(a, b, p, e):
        assert Fraction(float(pp)) + Fraction(float(ee)) == Fraction(float(x)) * Fraction(float(y))


def test_two_prod_error_is_exact():
    check_two_prod(simt_dd._two_prod_err)


def test_two_sum_is_error_free():
    rng = np.random.default_rng(2)
    a = rng.normal(size=500) * np.ldexp(1.0, rng.integers(-60, 60, 500))
    b = rng.normal(size=500) * np.ldexp(1.0, rng.integers(-60, 60, 500))
    s, t = simt_dd._two_sum(a, b)
    for x, y, ss, tt in zip(a, b, s, t):
        assert Fraction(float(ss)) + Fraction(float(tt)) == Fraction(float(x)) + Fraction(float(y))


def check_accuracy(fn):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(9, 11, 40, "normal_rowcol30", 3)
    C_hi, C_lo = fn(A_hi, A_lo, B_hi, B_lo)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    mag = np.abs(A_hi) @ np.abs(B_hi)
    err = np.abs((C_hi - R_hi) + (C_lo - R_lo))
    # a dd inner product of length K loses at most ~K ulps of 2^-104 of |A||B|
    assert np.all(err <= 40 * 2.0**-100 * mag)


def test_accuracy_against_exact_oracle():
    check_accuracy(simt_dd.simt_dd_gemm)


def test_exact_on_short_integers():
    rng = np.random.default_rng(4)
    A = rng.integers(-2**20, 2**20, (7, 13)).astype(np.float64)
    B = rng.integers(-2**20, 2**20, (13, 5)).astype(np.float64)
    C_hi, C_lo = simt_dd.simt_dd_gemm(A, np.zeros_like(A), B, np.zeros_like(B))
    assert np.array_equal(C_hi, A @ B) and not C_lo.any()


def test_workload0_normwise():
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(0)
    C_hi, C_lo = simt_dd.simt_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    d = (C_hi - R_hi) + (C_lo - R_lo)
    assert np.linalg.norm(d) / (np.linalg.norm(A_hi) * np.linalg.norm(B_hi)) <= 1e-26


def _err_plain(a, b, p):
    return a * b - p  # rounds to zero: not the product error


def _gemm_without_cross_terms(A_hi, A_lo, B_hi, B_lo):
    return simt_dd.simt_dd_gemm(A_hi, np.zeros_like(A_lo), B_hi, np.zeros_like(B_lo))


@pytest.mark.parametrize("check,bad", [
    (check_two_prod, _err_plain),
    (check_accuracy, _gemm_without_cross_terms),
])
def test_planted_mistakes_are_caught(check, bad):
    with pytest.raises(AssertionError):
        check(bad)
