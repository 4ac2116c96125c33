"""Pins for the multiple-double oracle (oracle.exact_md_gemm) and the
quad-double model of the method (oracle.slices_md): rational brute force,
consistency with the double-double oracle and model, reconstruction, index-sum
brute force, single-part weights, the exactness bound, and planted mistakes."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from oracle import slices, slices_md
from tests.exact_ref import bits, pow2, rne

QD_GATE = 1e-57


def _exact_parts(x: Fraction, n: int):
    out = []
    for _ in range(n):
        v = rne(x) + 0.0
        out.append(v)
        if v == 0.0 or not math.isfinite(v):
            out += [0.0] * (n - len(out))
            break
        x -= Fraction(v)
    return out


@pytest.mark.parametrize("seed", range(25))
def test_md_oracle_bruteforce(seed):
    rng = np.random.default_rng(500 + seed)
    M, N, K = (int(v) for v in rng.integers(1, 5, 3))
    A, B = workloads.make_md(M, N, K, ["uniform", "normal", "uniform_exp20"][seed % 3], seed, 4)
    if seed % 4 == 0:  # some exact cancellation and zeros
        A[0][0, :] = 0.0
        A[1][0, :] = A[2][0, :] = A[3][0, :] = 0.0
    C = oracle.exact_md_gemm(A, B)
    for i in range(M):
        for j in range(N):
            X = sum(sum(Fraction(float(a[i, k])) for a in A) * sum(Fraction(float(b[k, j])) for b in B)
                    for k in range(K))
            ref = _exact_parts(X, 4)
            for p in range(4):
                assert bits(C[p][i, j]) == bits(ref[p]), (i, j, p)


def test_md_oracle_two_parts_is_dd_oracle():
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(13, 9, 50, "normal_rowcol30", 9)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    C = oracle.exact_md_gemm([A_hi, A_lo], [B_hi, B_lo])
    assert np.array_equal(C[0], R_hi) and np.array_equal(C[1], R_lo)


def test_md_inputs_are_normalised():
    A, B = workloads.make_md(30, 20, 25, "normal_rowcol30", 4, 4)
    for X in (A, B):
        for p in range(3):
            assert np.all(np.abs(X[p + 1]) <= np.spacing(np.abs(X[p])) / 2)


def test_qd_exactness_bound():
    assert slices_md.max_k(16) == 2**23
    assert 16 * 2**23 * 8191**2 < 2**53 <= 16 * 2**24 * 8191**2
    assert slices_md.max_k(8) == 2**24


def check_digits(fn):
    rng = np.random.default_rng(5)
    A, _ = workloads.make_md(1, 1, 300, "normal", 6, 4)
    for k in range(300):
        parts = [float(a[0, k]) for a in A]
        e = int(slices.exponent_of(np.array([parts[0]]))[0]) + int(rng.integers(0, 20))
        D = fn(parts, e, 16)
        v = sum(Fraction(x) for x in parts) * pow2(-e)
        rec = sum(Fraction(d) * pow2(-13 * (s + 1)) for s, d in enumerate(D))
        r = v - rec
        assert abs(r) < pow2(-208) and (r == 0 or (r > 0) == (v > 0))
        assert all(abs(d) < 2**13 for d in D)


def test_qd_digits_reconstruct():
    check_digits(slices_md.digits_of)


def test_digits_agree_with_dd_model():
    A_hi, A_lo, _, _ = workloads.make_dd(5, 1, 40, "uniform_exp20", 7)
    e = slices.row_exponents(A_hi)
    for i in range(5):
        for k in range(40):
            assert slices_md.digits_of([A_hi[i, k], A_lo[i, k]], int(e[i]), 8) == \
                slices.digits_of(A_hi[i, k], A_lo[i, k], int(e[i]))


def check_products(fn):
    rng = np.random.default_rng(8)
    DA = rng.integers(-8191, 8192, (16, 2, 3))
    DB = rng.integers(-8191, 8192, (16, 3, 2))
    P = fn(DA, DB)
    for d in range(16):
        for i in range(2):
            for j in range(2):
                ref = sum(int(DA[s, i, k]) * int(DB[d - s, k, j]) for s in range(d + 1) for k in range(3))
                assert P[d, i, j] == ref


def test_qd_slice_products_bruteforce():
    check_products(slices_md.slice_products)


def check_recombine(fn):
    rng = np.random.default_rng(10)
    for d in range(16):      # each part alone: weight 2^(-13(d+2)) 2^(e+f)
        P = np.zeros((16, 1, 1))
        v = float(rng.integers(1, 2**53))
        P[d, 0, 0] = v
        C = fn(P, np.array([3]), np.array([-5]), 4)
        assert C[0][0, 0] == math.ldexp(v, -13 * (d + 2) - 2)
        assert C[1][0, 0] == 0.0
    for _ in range(100):     # against rational rounding
        P = np.array([float(rng.integers(-2**53 + 1, 2**53)) for _ in range(16)]).reshape(16, 1, 1)
        e, f = int(rng.integers(-40, 40)), int(rng.integers(-40, 40))
        C = fn(P, np.array([e]), np.array([f]), 4)
        X = sum(Fraction(float(P[d, 0, 0])) * pow2(-13 * (d + 2)) for d in range(16)) * pow2(e + f)
        ref = _exact_parts(X, 4)
        for p in range(4):
            assert bits(C[p][0, 0]) == bits(ref[p])


def test_qd_recombine_rounds_once():
    check_recombine(slices_md.recombine)


def _normwise(C, R, A, B):
    d = sum(C[p] - R[p] for p in range(len(C)))
    return np.linalg.norm(d) / (np.linalg.norm(sum(A)) * np.linalg.norm(sum(B)))


@pytest.mark.parametrize("dist", workloads.DISTS)
def test_qd_chain_vs_exact(dist):
    A, B = workloads.make_md(11, 9, 37, dist, 12, 4)
    C, *_ = slices_md.sliced_md_gemm(A, B, 16)
    R = oracle.exact_md_gemm(A, B)
    assert _normwise(C, R, A, B) <= QD_GATE


def test_qd_chain_exact_on_short_integers():
    rng = np.random.default_rng(13)
    A0 = rng.integers(-2**20, 2**20, (6, 9)).astype(np.float64)
    B0 = rng.integers(-2**20, 2**20, (9, 4)).astype(np.float64)
    Z = [np.zeros_like(A0)] * 3
    W = [np.zeros_like(B0)] * 3
    C, *_ = slices_md.sliced_md_gemm([A0] + Z, [B0] + W, 16)
    assert np.array_equal(C[0], A0 @ B0) and not any(c.any() for c in C[1:])


def _digits_drop_third_part(parts, e, S):
    return slices_md.digits_of(list(parts[:2]) + [0.0] * (len(parts) - 2), e, S)


def _products_off_by_one(DA, DB):
    return np.roll(slices_md.slice_products(DA, DB), 1, axis=0)


def _recombine_truncating(P, e, f, nout):
    C = slices_md.recombine(P, e, f, nout)
    C[1] = np.zeros_like(C[1])
    return C


@pytest.mark.parametrize("check,bad", [
    (check_digits, _digits_drop_third_part),
    (check_products, _products_off_by_one),
    (check_recombine, _recombine_truncating),
])
def test_planted_mistakes_are_caught(check, bad):
    with pytest.raises(AssertionError):
        check(bad)
