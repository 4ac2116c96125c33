"""Pins for the oracle's model of the method's steps (oracle.slices).

Each step is pinned to something other than itself: the worked quartering
example of Section 2 ("Multiple Double Arithmetic on NVIDIA Tensor Cores"),
exact rational reconstruction, the trailing-zero property of quarter products,
the bound of eq. (5), brute-force integer sums for the index-sum grouping of
eqs. (1)-(4), single-part closed forms for the recombination weights, and the
exact oracle for the whole chain.
"""
import math
import pathlib
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import slices
from tests.exact_ref import pow2
import workloads

GOLDEN = pathlib.Path(__file__).parent / "golden" / "quartering_example.txt"


def _read_golden():
    rows = {}
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        key, *rest = line.split()
        rows[key] = rest
    return rows


def check_worked_example(digits_fn):
    g = _read_golden()
    frac = "".join(g["fraction"])
    fields = ["".join(g[f"f{q}"]) for q in range(4)]
    assert len(frac) == 52 and all(len(f) == 52 for f in fields)
    # the fixture is self-consistent: the parts are disjoint 13-bit windows of f
    assert int(frac, 2) == sum(int(f, 2) for f in fields)
    for q, f in enumerate(fields):
        assert int(f, 2) >> (52 - 13 * (q + 1)) << (52 - 13 * (q + 1)) == int(f, 2)
        assert int(f, 2) < 1 << (52 - 13 * q)
    # the value 0.f (binary) has shared exponent 0 and digits f0..f3, then zeros
    y = math.ldexp(float(int(frac, 2)), -52)
    e = int(slices.exponent_of(np.array([y]))[0])
    assert e == 0
    D = digits_fn(y, 0.0, e)
    expect = [int(f, 2) >> (52 - 13 * (q + 1)) for q, f in enumerate(fields)]
    assert D[:4] == expect, (D, expect)
    assert D[4:] == [0, 0, 0, 0]
    # the quarters x_q = D_q * 2^(-13(q+1)) * 2 carry the printed significand
    # bits and the exponents 0, -13, -26, -39
    for q in range(4):
        lead, *mid, ex = g[f"x{q}"]
        x = math.ldexp(float(D[q]), -13 * (q + 1) + 1)
        m, E = math.frexp(x)
        assert E - 1 == int(ex)
        sig = int(m * 2**13)
        assert format(sig, "013b") == lead + "".join(mid)


def test_worked_quartering_example():
    check_worked_example(slices.digits_of)


def test_exponent_of_closed_forms():
    xs = np.array([1.0, 0.5, 0.75, 2.0**-1074, 0.0, -3.0, 2.0**1023, 1.0 - 2.0**-53, 2.0**-1022])
    ex = slices.exponent_of(xs)
    assert list(ex) == [1, 0, 0, -1073, 0, 2, 1024, 0, -1021]
    rng = np.random.default_rng(0)
    v = rng.normal(size=200) * np.ldexp(1.0, rng.integers(-1070, 1000, 200))
    for x, e in zip(v, slices.exponent_of(v)):
        a = abs(Fraction(float(x)))
        assert pow2(int(e) - 1) <= a < pow2(int(e))


def test_row_col_exponents():
    A = np.array([[0.0, 0.0, 0.0], [0.25, -0.9, 0.1], [-4.0, 1.0, 0.0]])
    assert list(slices.row_exponents(A)) == [0, 0, 3]
    assert list(slices.col_exponents(A)) == [3, 1, -3]


def check_reconstruction(digits_fn):
    rng = np.random.default_rng(1)
    for _ in range(400):
        hi = rng.normal() * 2.0 ** int(rng.integers(-40, 40))
        lo = hi * 2.0**-53 * rng.uniform(-1, 1)
        s = hi + lo
        bb = s - hi
        hi, lo = s, (hi - (s - bb)) + (lo - bb)
        e = int(slices.exponent_of(np.array([hi]))[0]) + int(rng.integers(0, 30))
        D = digits_fn(hi, lo, e)
        v = (Fraction(hi) + Fraction(lo)) * pow2(-e)
        rec = sum(Fraction(d) * pow2(-13 * (s_ + 1)) for s_, d in enumerate(D))
        r = v - rec
        # truncation toward zero: remainder has the sign of v and is < 2^-104
        assert abs(r) < pow2(-104)
        assert r == 0 or (r > 0) == (v > 0)
        assert all(abs(d) < 2**13 for d in D)
        assert all(d == 0 or (d > 0) == (v > 0) for d in D)
        # a plain double (lo = 0) whose 53 bits lie within the 104-bit window
        # is reproduced bit-exactly by its quarters
        e2 = int(slices.exponent_of(np.array([hi]))[0])
        D2 = digits_fn(hi, 0.0, e2)
        rec2 = sum(Fraction(d) * pow2(e2 - 13 * (s_ + 1)) for s_, d in enumerate(D2))
        assert rec2 == Fraction(hi)


def test_quarters_sum_back_exactly():
    check_reconstruction(slices.digits_of)


def test_opposite_sign_borrow():
    # hi > 0, lo < 0: the truncated digits are those of hi - |lo| (eq. (7) move)
    hi, lo = 0.75, -2.0**-60
    D = slices.digits_of(hi, lo, 0)
    X = sum(d << (13 * (7 - s)) for s, d in enumerate(D))
    assert X == (3 << 102) - (1 << 44) - 0  # floor((3/4 - 2^-60) 2^104)
    D = slices.digits_of(-hi, -lo, 0)
    assert all(d <= 0 for d in D)


def test_quarter_products_have_26_trailing_zero_bits():
    # "Multiplying two quarters leaves at least 26 zero bits at the end"
    rng = np.random.default_rng(2)
    for _ in range(2000):
        a = int(rng.integers(-(2**13) + 1, 2**13))
        b = int(rng.integers(-(2**13) + 1, 2**13))
        p = float(a * b)
        if p == 0:
            continue
        m, _ = math.frexp(abs(p))
        sig = int(m * 2**53)
        tz = (sig & -sig).bit_length() - 1
        assert tz >= 26
    assert float((2**13 - 1) ** 2) == (2**13 - 1) ** 2


def test_eq5_bound_and_exactness_limit():
    # eq. (5): N * (2^26 - 1) <= 2^52  =>  N <= 67,108,865
    B = sum(2**i for i in range(26))
    assert B == 2**26 - 1
    assert 2**52 // B == 67_108_865
    assert 67_108_865 * B <= 2**52 < 67_108_866 * B
    # index-sum grouping: part d sums (d+1) K products of 13-bit digits, so
    # every partial sum stays below 2^53 for K <= 2^24 (and not for 2^25)
    dmax = (1 << 13) - 1
    assert slices.S * slices.MAX_K * dmax**2 < 2**53
    assert slices.S * 2 * slices.MAX_K * dmax**2 >= 2**53


def check_slice_products(fn):
    rng = np.random.default_rng(3)
    M, N, K = 3, 4, 5
    DA = rng.integers(-(2**13) + 1, 2**13, (8, M, K))
    DB = rng.integers(-(2**13) + 1, 2**13, (8, K, N))
    P = fn(DA, DB)
    for d in range(8):
        for i in range(M):
            for j in range(N):
                ref = 0
                for s in range(8):
                    for t in range(8):
                        if s + t == d:
                            ref += sum(int(DA[s, i, k]) * int(DB[t, k, j]) for k in range(K))
                assert P[d, i, j] == ref


def test_slice_products_bruteforce():
    check_slice_products(slices.slice_products)
    check_slice_products(lambda a, b: slices.slice_products(a, b, exact_int=True))


def test_slice_products_float_matches_int_at_bound():
    # largest digits, K large: float64 matmul is still exact below 2^53
    rng = np.random.default_rng(4)
    K = 4096
    DA = np.full((8, 2, K), 8191, dtype=np.int64) * rng.choice([-1, 1], (8, 2, K))
    DB = np.full((8, K, 3), 8191, dtype=np.int64)
    Pf = slices.slice_products(DA, DB)
    Pi = slices.slice_products(DA, DB, exact_int=True)
    assert np.array_equal(Pf, Pi)


def check_recombine(fn):
    rng = np.random.default_rng(5)
    # each part alone carries weight 2^(-13 (d + 2)) times 2^(e + f)
    for d in range(8):
        P = np.zeros((8, 1, 1))
        val = float(rng.integers(1, 2**53))
        P[d, 0, 0] = val
        e, f = np.array([int(rng.integers(-30, 30))]), np.array([int(rng.integers(-30, 30))])
        h, l = fn(P, e, f)
        assert h[0, 0] == math.ldexp(val, -13 * (d + 2) + int(e[0] + f[0]))
        assert l[0, 0] == 0.0
    # sums of integer parts: within dd accuracy of the exact rational sum
    for _ in range(300):
        P = np.array([float(rng.integers(-(2**53) + 1, 2**53)) for _ in range(8)]).reshape(8, 1, 1)
        P[rng.integers(0, 8, rng.integers(0, 8))] = 0.0
        e, f = np.array([int(rng.integers(-40, 40))]), np.array([int(rng.integers(-40, 40))])
        h, l = fn(P, e, f)
        ex = sum(Fraction(float(P[d, 0, 0])) * pow2(-13 * (d + 2)) for d in range(8)) * pow2(int(e[0] + f[0]))
        mag = sum(abs(Fraction(float(P[d, 0, 0]))) * pow2(-13 * (d + 2)) for d in range(8)) * pow2(int(e[0] + f[0]))
        err = abs(Fraction(float(h[0, 0])) + Fraction(float(l[0, 0])) - ex)
        assert err <= mag * pow2(-103)
        assert abs(l[0, 0]) <= np.spacing(abs(h[0, 0])) / 2 or h[0, 0] == 0
    # two parts that fit one double are summed exactly
    P = np.zeros((8, 1, 1))
    P[0, 0, 0] = float(2**39 + 12345)
    P[1, 0, 0] = float(2**12 + 77)
    h, l = fn(P, np.array([0]), np.array([0]))
    assert Fraction(float(h[0, 0])) == Fraction(2**39 + 12345) * pow2(-26) + Fraction(2**12 + 77) * pow2(-39)
    assert l[0, 0] == 0.0


def test_recombine_weights_and_accuracy():
    check_recombine(slices.recombine)


def _normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo):
    d = (C_hi - R_hi) + (C_lo - R_lo)
    return np.linalg.norm(d) / (np.linalg.norm(A_hi + A_lo) * np.linalg.norm(B_hi + B_lo))


def test_sliced_chain_vs_exact_oracle_small_workload():
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(0)
    C_hi, C_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert _normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= 1e-26
    assert np.max(np.abs(C_hi - R_hi)) <= 1e-28 * np.max(np.abs(R_hi))


@pytest.mark.parametrize("dist", workloads.DISTS)
def test_sliced_chain_vs_exact_oracle_ragged(dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(7, 13, 29, dist, 11)
    C_hi, C_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert _normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= 1e-26


def test_sliced_chain_exact_on_short_integers():
    # integer inputs below 2^20: every digit product is kept, the sum fits one
    # double, so the chain equals the exact product bit for bit
    rng = np.random.default_rng(6)
    A_hi = rng.integers(-2**20, 2**20, (9, 17)).astype(np.float64)
    B_hi = rng.integers(-2**20, 2**20, (17, 5)).astype(np.float64)
    Z1, Z2 = np.zeros_like(A_hi), np.zeros_like(B_hi)
    C_hi, C_lo, *_ = slices.sliced_dd_gemm(A_hi, Z1, B_hi, Z2)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, Z1, B_hi, Z2)
    assert np.array_equal(C_hi, R_hi) and np.array_equal(C_lo, R_lo)
    assert np.array_equal(C_hi, A_hi @ B_hi)


# ---- planted mistakes: each plausible slip in the model fails one pin ----

def _digits_msd_last(hi, lo, e):
    return slices.digits_of(hi, lo, e)[::-1]


def _digits_dropping_lo(hi, lo, e):
    return slices.digits_of(hi, 0.0, e)


def _digits_rounding(hi, lo, e):
    v = (Fraction(hi) + Fraction(lo)) * pow2(104 - e)
    X = round(abs(v))
    sign = -1 if v < 0 else 1
    return [sign * ((X >> (13 * (7 - s))) & 8191) for s in range(8)]


def _products_transposed(DA, DB):
    return slices.slice_products(DA, DB[::-1])


def _products_all_pairs_index_off(DA, DB):
    P = slices.slice_products(DA, DB)
    return np.roll(P, 1, axis=0)


def _recombine_weight_off(P, e, f):
    return slices.recombine(np.roll(P, -1, axis=0), e, f)


def _recombine_sign(P, e, f):
    h, l = slices.recombine(P, e, f)
    return h, -l


@pytest.mark.parametrize("check,bad", [
    (check_worked_example, _digits_msd_last),
    (check_reconstruction, _digits_dropping_lo),
    (check_reconstruction, _digits_rounding),
    (check_slice_products, _products_transposed),
    (check_slice_products, _products_all_pairs_index_off),
    (check_recombine, _recombine_weight_off),
    (check_recombine, _recombine_sign),
])
def test_planted_mistakes_are_caught(check, bad):
    with pytest.raises(AssertionError):
        check(bad)
