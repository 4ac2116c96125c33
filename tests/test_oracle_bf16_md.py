"""Pins for the 8-bit-part variant for multiple doubles (oracle.slices_bf16_md):
reconstruction and truncation toward zero of 27 quad-double parts, part ranges,
index-sum brute force, single-part weights and rational rounding into four
doubles, the chain within the quad-double gate of the exact multiple-double
oracle on every distribution and bit-exact to it on short integers, the
double-double case equal to oracle.slices_bf16, and planted mistakes."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from oracle import slices, slices_bf16, slices_bf16_md as bm
from tests.exact_ref import bits, pow2, rne

QD_GATE = 1e-57
S = bm.QD_PARTS


def check_digits(fn):
    A, _ = workloads.make_md(3, 1, 90, "uniform_exp20", 8, 4)
    A[0][0, :4] = 0.0        # zeros in the leading double: lower doubles zero too
    for p in range(1, 4):
        A[p][0, :4] = 0.0
    e = bm.row_exponents(A[0])
    for i in range(3):
        for k in range(90):
            parts = [float(a[i, k]) for a in A]
            D = fn(parts, int(e[i]), S)
            v = sum(Fraction(x) for x in parts) * pow2(-int(e[i]))
            assert abs(v) < Fraction(1, 2)
            rec = sum(Fraction(d) * pow2(-8 * (s + 1)) for s, d in enumerate(D))
            r = v - rec
            assert abs(r) < pow2(-8 * S) and (r == 0 or (r > 0) == (v > 0)), (i, k)
            assert -128 <= D[0] <= 128 and all(-128 <= d <= 127 for d in D[1:])


def test_qd_parts_reconstruct_and_truncate_toward_zero():
    check_digits(bm.digits_of)


def test_dd_case_is_the_dd_variant():
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(7, 5, 40, "normal_rowcol30", 3)
    C, e, f, DA, DB, P = bm.sliced_gemm([A_hi, A_lo], [B_hi, B_lo], slices_bf16.S)
    R = slices_bf16.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(e, R[2]) and np.array_equal(DA, R[4]) and np.array_equal(P, R[6])
    assert np.array_equal(C[0], R[0]) and np.array_equal(C[1], R[1])


def check_products(fn):
    rng = np.random.default_rng(9)
    DA = rng.integers(-128, 129, (S, 2, 3))
    DB = rng.integers(-128, 129, (S, 3, 2))
    P = fn(DA, DB)
    for d in range(S):
        for i in range(2):
            for j in range(2):
                ref = sum(int(DA[s, i, k]) * int(DB[d - s, k, j]) for s in range(d + 1) for k in range(3))
                assert P[d, i, j] == ref


def test_qd_slice_products_bruteforce():
    check_products(bm.slice_products)
    assert bm.pairs(S) == 378


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


def check_recombine(fn):
    rng = np.random.default_rng(11)
    for d in range(S):       # each part alone: weight 2^(-8(d+2)) 2^(e+f)
        P = np.zeros((S, 1, 1), dtype=np.int64)
        v = int(rng.integers(1, 2**40))
        P[d, 0, 0] = v
        C = fn(P, np.array([2]), np.array([-3]), 4)
        assert C[0][0, 0] == math.ldexp(float(v), -8 * (d + 2) - 1)
        assert C[1][0, 0] == 0.0
    for _ in range(60):      # against rational rounding
        P = rng.integers(-2**44, 2**44, (S, 1, 1))
        e, f = int(rng.integers(-30, 30)), int(rng.integers(-30, 30))
        C = fn(P, np.array([e]), np.array([f]), 4)
        X = sum(Fraction(int(P[d, 0, 0])) * pow2(-8 * (d + 2)) for d in range(S)) * pow2(e + f)
        ref = _exact_parts(X, 4)
        for p in range(4):
            assert bits(C[p][0, 0]) == bits(ref[p])


def test_qd_recombine_rounds_once():
    check_recombine(bm.recombine)


def _normwise(C, R, A, B):
    d = sum(C[p] - R[p] for p in range(len(C)))
    return np.linalg.norm(d) / (np.linalg.norm(sum(A)) * np.linalg.norm(sum(B)))


@pytest.mark.parametrize("dist", workloads.DISTS)
def test_qd_chain_vs_exact(dist):
    A, B = workloads.make_md(9, 7, 31, dist, 13, 4)
    C, *_ = bm.sliced_gemm(A, B)
    R = oracle.exact_md_gemm(A, B)
    assert _normwise(C, R, A, B) <= QD_GATE


def test_qd_chain_exact_on_short_integers():
    rng = np.random.default_rng(14)
    A0 = rng.integers(-2**20, 2**20, (5, 8)).astype(np.float64)
    B0 = rng.integers(-2**20, 2**20, (8, 3)).astype(np.float64)
    Z = [np.zeros_like(A0)] * 3
    W = [np.zeros_like(B0)] * 3
    C, *_ = bm.sliced_gemm([A0] + Z, [B0] + W)
    assert np.array_equal(C[0], A0 @ B0) and not any(c.any() for c in C[1:])


def _digits_drop_last_double(parts, e, S_):
    return bm.digits_of(list(parts[:3]) + [0.0], e, S_)


def _products_shifted(DA, DB):
    return np.roll(bm.slice_products(DA, DB), 1, axis=0)


def _recombine_three_parts(P, e, f, nout):
    C = bm.recombine(P, e, f, nout)
    C[3] = np.zeros_like(C[3])
    return C


@pytest.mark.parametrize("check,bad", [
    (check_digits, _digits_drop_last_double),
    (check_products, _products_shifted),
    (check_recombine, _recombine_three_parts),
])
def test_planted_mistakes_are_caught(check, bad):
    with pytest.raises(AssertionError):
        check(bad)


# ---- octo doubles (8 doubles, 54 parts) and hexa doubles (16 doubles, 107 parts) ----

OD_HD = [(8, 54, -404), (16, 107, -828)]  # doubles, parts, log2 of the normwise gate


def log2_normwise(C, R, A, B):
    """log2 of the normwise error, formed from exact rational differences (the
    errors of hexa doubles are far below the double range of their squares)."""
    import math
    tot = Fraction(0)
    for i in range(C[0].shape[0]):
        for j in range(C[0].shape[1]):
            d = sum(Fraction(float(C[p][i, j])) - Fraction(float(R[p][i, j])) for p in range(len(C)))
            tot += d * d
    if tot == 0:
        return -math.inf
    den = np.linalg.norm(sum(A)) * np.linalg.norm(sum(B))
    return (math.log2(tot.numerator) - math.log2(tot.denominator)) / 2 - math.log2(den)


@pytest.mark.parametrize("n,S_,gate", OD_HD)
def test_od_hd_parts_reconstruct(n, S_, gate):
    A, _ = workloads.make_md(2, 1, 12, "uniform_exp20", 8 + n, n)
    e = bm.row_exponents(A[0])
    for i in range(2):
        for k in range(12):
            parts = [float(a[i, k]) for a in A]
            D = bm.digits_of(parts, int(e[i]), S_)
            v = sum(Fraction(x) for x in parts) * pow2(-int(e[i]))
            r = v - sum(Fraction(d) * pow2(-8 * (s + 1)) for s, d in enumerate(D))
            assert abs(r) < pow2(-8 * S_) and (r == 0 or (r > 0) == (v > 0))
            assert -128 <= D[0] <= 128 and all(-128 <= d <= 127 for d in D[1:])


@pytest.mark.parametrize("n,S_,gate", OD_HD)
@pytest.mark.parametrize("dist", workloads.DISTS)
def test_od_hd_chain_vs_exact(n, S_, gate, dist):
    A, B = workloads.make_md(4, 3, 15, dist, 17, n)
    C, *_ = bm.sliced_gemm(A, B, S_)
    R = oracle.exact_md_gemm(A, B)
    assert log2_normwise(C, R, A, B) <= gate


@pytest.mark.parametrize("n,S_,gate", OD_HD)
def test_od_hd_chain_exact_on_short_integers(n, S_, gate):
    rng = np.random.default_rng(15)
    A0 = rng.integers(-2**20, 2**20, (3, 5)).astype(np.float64)
    B0 = rng.integers(-2**20, 2**20, (5, 2)).astype(np.float64)
    C, *_ = bm.sliced_gemm([A0] + [np.zeros_like(A0)] * (n - 1), [B0] + [np.zeros_like(B0)] * (n - 1), S_)
    assert np.array_equal(C[0], A0 @ B0) and not any(c.any() for c in C[1:])


@pytest.mark.parametrize("n", [8, 16])
def test_md_oracle_bruteforce_many_parts(n):
    A, B = workloads.make_md(2, 2, 3, ["uniform", "normal"][n // 16], 40 + n, n)
    C = oracle.exact_md_gemm(A, B)
    for i in range(2):
        for j in range(2):
            X = sum(sum(Fraction(float(a[i, k])) for a in A) * sum(Fraction(float(b[k, j])) for b in B)
                    for k in range(3))
            ref = _exact_parts(X, n)
            for p in range(n):
                assert bits(C[p][i, j]) == bits(ref[p]), (i, j, p)
