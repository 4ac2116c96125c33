"""Pins for the 8-bit-part model (oracle.slices_bf16): balanced digits against
a second derivation (two's-complement bytes with carries), reconstruction and
truncation toward zero, bf16 representability of every part (torch's own
bf16 conversion), index-sum brute force, single-part weights and rational
rounding of the recombination, the exact oracle on short integers and within
the normwise gate, and planted mistakes."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import slices, slices_bf16 as sb
from tests.exact_ref import bits, pow2, rne

GATE = 1e-26


def _digits_by_bytes(X: int) -> list[int]:
    """Balanced digits by another route: the base-256 digits of |X| (most
    significant first), each digit >= 128 replaced by digit - 256 with a carry
    into the next higher digit, then the sign applied to every digit."""
    sign = -1 if X < 0 else 1
    m = abs(X)
    raw = [(m >> (8 * (sb.S - 1 - s))) & 255 for s in range(sb.S)]
    out = [0] * sb.S
    carry = 0
    for s in range(sb.S - 1, -1, -1):
        v = raw[s] + carry
        if s > 0 and v >= 128:
            out[s], carry = v - 256, 1
        else:
            out[s], carry = v, 0
    # for a negative X the digits of |X| are negated; a negated digit of
    # exactly -128 is +128, which is rebalanced (128 = 256 - 128) by the
    # same rule on the negated sequence
    out = [sign * d for d in out]
    carry = 0
    for s in range(sb.S - 1, -1, -1):
        v = out[s] + carry
        if s > 0 and v >= 128:
            out[s], carry = v - 256, 1
        elif s > 0 and v < -128:
            out[s], carry = v + 256, -1
        else:
            out[s], carry = v, 0
    return out


def _edge_values():
    top = (1 << (sb.FIX_BITS - 1)) - 1
    vals = [0, 1, -1, 127, 128, -128, -129, 255, 256, -256, top, -top, 128 << 96, -(128 << 96),
            (128 << 96) - 1, 0x80 * sum(1 << (8 * i) for i in range(12)),
            -0x80 * sum(1 << (8 * i) for i in range(12))]
    rng = np.random.default_rng(3)
    for _ in range(2000):
        v = int.from_bytes(rng.bytes(13), "little") >> (1 + int(rng.integers(0, 100)))
        vals.append(v if rng.integers(0, 2) else -v)
    return vals


def test_balanced_digits_two_derivations():
    for X in _edge_values():
        D = sb.balanced_digits(X)
        assert D == _digits_by_bytes(X), X
        assert sum(d << (8 * (sb.S - 1 - s)) for s, d in enumerate(D)) == X
        assert -128 <= D[0] <= 128 and all(-128 <= d <= 127 for d in D[1:])


def test_every_part_is_exact_in_bf16():
    D = torch.tensor(sorted({d for X in _edge_values() for d in sb.balanced_digits(X)}), dtype=torch.int64)
    assert D.min() >= -128 and D.max() <= 128
    assert torch.equal(D.to(torch.bfloat16).to(torch.int64), D)
    # the 8-bit significand holds every integer up to 256, and 257 is the first
    # it cannot hold: the check above is not vacuous
    assert torch.tensor([256.0]).to(torch.bfloat16).item() == 256.0
    assert torch.tensor([257.0]).to(torch.bfloat16).item() != 257.0


def check_digits(fn):
    A_hi, A_lo, _, _ = workloads.make_dd(6, 1, 120, "uniform_exp20", 21)
    A_lo[0, :5] = -np.sign(A_hi[0, :5]) * np.spacing(np.abs(A_hi[0, :5])) / 2  # opposite signs
    A_hi[1, 3] = 0.0
    A_lo[1, 3] = 0.0
    e = sb.row_exponents(A_hi)
    for i in range(6):
        for k in range(120):
            D = fn(A_hi[i, k], A_lo[i, k], int(e[i]))
            v = (Fraction(float(A_hi[i, k])) + Fraction(float(A_lo[i, k]))) * pow2(-int(e[i]))
            assert abs(v) < Fraction(1, 2)
            rec = sum(Fraction(d) * pow2(-8 * (s + 1)) for s, d in enumerate(D))
            r = v - rec
            assert abs(r) < pow2(-104) and (r == 0 or (r > 0) == (v > 0)), (i, k)
            assert -128 <= D[0] <= 128 and all(-128 <= d <= 127 for d in D[1:])


def test_digits_reconstruct_and_truncate_toward_zero():
    check_digits(sb.digits_of)


def test_exponents_have_one_bit_of_headroom():
    A_hi, _, B_hi, _ = workloads.make_dd(9, 7, 30, "normal_rowcol30", 4)
    A_hi[2, :] = 0.0
    e, f = sb.row_exponents(A_hi), sb.col_exponents(B_hi)
    assert np.array_equal(e, slices.row_exponents(A_hi) + 1)
    assert e[2] == 1
    for i in range(9):
        assert np.all(np.abs(A_hi[i]) < 2.0 ** (int(e[i]) - 1))
        if A_hi[i].any():
            assert np.max(np.abs(A_hi[i])) >= 2.0 ** (int(e[i]) - 2)
    for j in range(7):
        assert np.all(np.abs(B_hi[:, j]) < 2.0 ** (int(f[j]) - 1))
    assert sb.row_exponents(np.array([[0.5, -0.25]]))[0] == 1       # 0.5 < 2^0, not < 2^-1
    assert sb.row_exponents(np.array([[0.4999]]))[0] == 0


def check_products(fn):
    rng = np.random.default_rng(8)
    DA = rng.integers(-128, 129, (sb.S, 2, 3))
    DB = rng.integers(-128, 129, (sb.S, 3, 2))
    P = fn(DA, DB)
    for d in range(sb.S):
        for i in range(2):
            for j in range(2):
                ref = sum(int(DA[s, i, k]) * int(DB[d - s, k, j]) for s in range(d + 1) for k in range(3))
                assert P[d, i, j] == ref


def test_slice_products_bruteforce():
    check_products(sb.slice_products)


def test_pair_count_and_bound():
    assert sb.PAIRS == 91 == sum(1 for s in range(13) for t in range(13) if s + t <= 12)
    # parts of magnitude <= 128: a product is at most 2^14, so a chunk of 1024
    # products sums to at most 2^24, an integer an fp32 accumulator holds
    assert 128 * 128 == 2**14 and 1024 * 2**14 == 2**24


def check_recombine(fn):
    rng = np.random.default_rng(10)
    for d in range(sb.S):      # each part alone: weight 2^(-8(d+2)) 2^(e+f)
        P = np.zeros((sb.S, 1, 1), dtype=np.int64)
        v = int(rng.integers(1, 2**40))
        P[d, 0, 0] = v
        C_hi, C_lo = fn(P, np.array([3]), np.array([-5]))
        assert C_hi[0, 0] == math.ldexp(float(v), -8 * (d + 2) - 2)
        assert C_lo[0, 0] == 0.0
    for _ in range(150):       # against rational rounding
        P = rng.integers(-2**44, 2**44, (sb.S, 1, 1))
        e, f = int(rng.integers(-40, 40)), int(rng.integers(-40, 40))
        C_hi, C_lo = fn(P, np.array([e]), np.array([f]))
        X = sum(Fraction(int(P[d, 0, 0])) * pow2(-8 * (d + 2)) for d in range(sb.S)) * pow2(e + f)
        hi = rne(X) + 0.0
        lo = rne(X - Fraction(hi)) + 0.0
        assert bits(C_hi[0, 0]) == bits(hi) and bits(C_lo[0, 0]) == bits(lo)


def test_recombine_rounds_once():
    check_recombine(sb.recombine)


def _normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo):
    d = (C_hi - R_hi) + (C_lo - R_lo)
    return np.linalg.norm(d) / (np.linalg.norm(A_hi + A_lo) * np.linalg.norm(B_hi + B_lo))


@pytest.mark.parametrize("dist", workloads.DISTS)
def test_chain_vs_exact_oracle(dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(13, 11, 70, dist, 31)
    C_hi, C_lo, *_ = sb.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert _normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= GATE


def test_chain_exact_on_short_integers():
    # 21-bit integers fill the top three parts only, so no pair is dropped and
    # nothing is truncated: the result is the exact product
    rng = np.random.default_rng(13)
    A0 = rng.integers(-2**20, 2**20, (6, 9)).astype(np.float64)
    B0 = rng.integers(-2**20, 2**20, (9, 4)).astype(np.float64)
    C_hi, C_lo, *_ = sb.sliced_dd_gemm(A0, np.zeros_like(A0), B0, np.zeros_like(B0))
    R_hi, R_lo = oracle.exact_dd_gemm(A0, np.zeros_like(A0), B0, np.zeros_like(B0))
    assert np.array_equal(C_hi, R_hi) and np.array_equal(C_lo, R_lo)
    assert np.array_equal(C_hi, A0 @ B0)


def _digits_lose_lo(hi, lo, e):
    return sb.digits_of(hi, 0.0, e)


def _products_swapped(DA, DB):
    P = sb.slice_products(DA, DB)
    return P[::-1].copy()


def _recombine_weight_off(P, e, f):
    return sb.recombine(P, np.asarray(e) + 1, f)


@pytest.mark.parametrize("check,bad", [
    (check_digits, _digits_lose_lo),
    (check_products, _products_swapped),
    (check_recombine, _recombine_weight_off),
])
def test_planted_mistakes_are_caught(check, bad):
    with pytest.raises(AssertionError):
        check(bad)
