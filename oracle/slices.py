"""The method's steps, written plainly: shared exponents, 13-bit quarters,
slice-pair products grouped by index sum, double-double recombination.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Source of every step:
"Multiple Double Arithmetic on NVIDIA Tensor Cores" (page 1), Section 2 and
Section 3.  Where the page leaves a step open, the reading taken is stated at
the step.

Notation: S = 8 slices (four quarters of the high double and four of the low
double make "8 parts" of a double double, Section 2, steps 1-2).  A double
double x = hi + lo of a row i of A (column j of B) is written against the
shared exponent e of that row (column) as

    x * 2^-e = sum_{s=0}^{S-1} D_s * 2^(-13 (s+1)) + r,   |r| < 2^(-13 S),

where the D_s are the truncating base-2^13 digits of |x * 2^-e| carrying the
sign of x ("quarters" of 13 bits with exponents 0, -13, -26, -39, ... on one
grid, Section 2 and Problems 3.2 / 3.4).  The product of two such expansions
is a convolution of the digit sequences (eqs. (1)-(3)): the part of index d
collects the pairs with s + t = d, so

    P_d = sum_{s+t=d} A_s @ B_t,    d = 0 .. S-1,

which is the nonzero block structure of the stacked / block-Toeplitz rewrite
of eq. (4) with the pairs of index sum >= S dropped.  All P_d are integers of
magnitude < 2^53 for K <= 2^24, so they are exact in double precision
(the argument of eq. (5)).  Finally (steps 4-5) the parts are summed in
double-double arithmetic and scaled back:

    C = 2^(e_i + f_j) * sum_{d} P_d * 2^(-13 (d + 2)).
"""
from __future__ import annotations

import numpy as np

S = 8              # slices per double double: 4 quarters of hi + 4 of lo
DIGIT_BITS = 13    # bits per quarter
FIX_BITS = S * DIGIT_BITS  # 104 fraction bits kept by the digit expansion
MAX_K = 1 << 24    # largest K for which every P_d stays below 2^53


def exponent_of(x: np.ndarray) -> np.ndarray:
    """Smallest integer e with |x| < 2^e, elementwise (0 where x == 0)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, ex = np.frexp(x)  # x = m * 2^ex with 1/2 <= m < 1, exact
    return np.where(x == 0, 0, ex).astype(np.int64)


def row_exponents(A_hi: np.ndarray) -> np.ndarray:
    """Shared exponent e_i of each row of A: the smallest e with
    max_k |A_hi[i,k]| < 2^e; an all-zero row gets 0.  (The page groups elements
    by the exponent of their leading quarter, Section 3 Problem 3.2; here one
    exponent is shared by a whole row, so that all quarters of the row lie on
    one grid.)"""
    return exponent_of(np.max(np.abs(A_hi), axis=1)) if A_hi.shape[1] else np.zeros(A_hi.shape[0], np.int64)


def col_exponents(B_hi: np.ndarray) -> np.ndarray:
    """Shared exponent f_j of each column of B (as row_exponents, over k)."""
    return exponent_of(np.max(np.abs(B_hi), axis=0)) if B_hi.shape[0] else np.zeros(B_hi.shape[1], np.int64)


def digits_of(hi: float, lo: float, e: int) -> list[int]:
    """The S truncating base-2^13 digits of (hi + lo) * 2^-e, signed.

    Exact rational arithmetic on Python integers: X = floor(|hi + lo| *
    2^(104 - e)) and D_s = sign * (13-bit field s of X, most significant
    first).  When hi and lo have opposite signs, the truncation of the sum
    borrows from the high digits: this is the value-preserving move of
    Problem 3.3 (eq. (7)) carried out on the fixed-point value.
    """
    n1, d1 = float(hi).as_integer_ratio()
    n2, d2 = float(lo).as_integer_ratio()
    num = n1 * d2 + n2 * d1          # (hi + lo) = num / den exactly
    den = d1 * d2
    sign = -1 if num < 0 else 1
    num = abs(num)
    shift = FIX_BITS - e
    if shift >= 0:
        num <<= shift
    else:
        den <<= -shift
    X = num // den
    if X >= 1 << FIX_BITS:
        raise ValueError("element not below 2^e: shared exponent too small")
    mask = (1 << DIGIT_BITS) - 1
    return [sign * ((X >> (DIGIT_BITS * (S - 1 - s))) & mask) for s in range(S)]


def split_rows(A_hi: np.ndarray, A_lo: np.ndarray, e: np.ndarray) -> np.ndarray:
    """Digit planes of A: D[s, i, k] (int64) against the row exponents e."""
    M, K = A_hi.shape
    D = np.zeros((S, M, K), dtype=np.int64)
    for i in range(M):
        ei = int(e[i])
        for k in range(K):
            D[:, i, k] = digits_of(A_hi[i, k], A_lo[i, k], ei)
    return D


def split_cols(B_hi: np.ndarray, B_lo: np.ndarray, f: np.ndarray) -> np.ndarray:
    """Digit planes of B: D[t, k, j] (int64) against the column exponents f."""
    K, N = B_hi.shape
    D = np.zeros((S, K, N), dtype=np.int64)
    for j in range(N):
        fj = int(f[j])
        for k in range(K):
            D[:, k, j] = digits_of(B_hi[k, j], B_lo[k, j], fj)
    return D


def slice_products(DA: np.ndarray, DB: np.ndarray, exact_int: bool = False) -> np.ndarray:
    """P[d] = sum_{s+t=d} DA[s] @ DB[t] for d = 0..S-1 (the index-sum grouping of
    eqs. (1)-(3)), as float64 holding exact integers.

    The matrix products are taken with float64 matmul: every partial sum is an
    integer of magnitude < 2^53 (checked), so any summation order is exact.
    ``exact_int=True`` uses int64 matmul instead (slow; used by the pins).
    """
    _, M, K = DA.shape
    N = DB.shape[2]
    if K > MAX_K:
        raise ValueError("K beyond the exactness bound")
    bound = 0
    P = np.zeros((S, M, N), dtype=np.float64)
    for d in range(S):
        acc = np.zeros((M, N), dtype=np.int64 if exact_int else np.float64)
        for s in range(d + 1):
            t = d - s
            if exact_int:
                acc += DA[s] @ DB[t]
            else:
                acc += DA[s].astype(np.float64) @ DB[t].astype(np.float64)
        bound = max(bound, (d + 1) * K * ((1 << DIGIT_BITS) - 1) ** 2)
        P[d] = acc
    assert bound < 2 ** 53
    return P


def _two_sum(a, b):
    s = a + b
    bb = s - a
    return s, (a - (s - bb)) + (b - bb)


def _quick_two_sum(a, b):
    s = a + b
    return s, b - (s - a)


def recombine(P: np.ndarray, e: np.ndarray, f: np.ndarray):
    """Steps 4-5: sum the parts P_d * 2^(-13 (d+2)) into one double double,
    then scale by 2^(e_i + f_j).

    Reading: the parts are added from the smallest weight (d = S-1) to the
    largest (d = 0); each addition is a two_sum of the running high word and
    the part, its error is added to the running low word, and a quick_two_sum
    renormalises the pair.  All operations are float64 round-to-nearest; the
    scaling by 2^(-13 (d+2)) is exact; the final scaling by 2^(e_i + f_j) is a
    correctly rounded ldexp of each word.  Zero results are +0.
    """
    P = np.asarray(P, dtype=np.float64)
    h = np.ldexp(P[S - 1], -DIGIT_BITS * (S + 1))
    l = np.zeros_like(h)
    for d in range(S - 2, -1, -1):
        t = np.ldexp(P[d], -DIGIT_BITS * (d + 2))
        s, err = _two_sum(h, t)
        err = err + l
        h, l = _quick_two_sum(s, err)
    scale = (np.asarray(e, dtype=np.int64)[:, None] + np.asarray(f, dtype=np.int64)[None, :])
    C_hi = np.ldexp(h, scale) + 0.0
    C_lo = np.ldexp(l, scale) + 0.0
    return C_hi, C_lo


def sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo):
    """The whole method on the CPU: exponents, digits, P_d, recombination.
    Returns (C_hi, C_lo, e, f, DA, DB, P)."""
    A_hi, A_lo, B_hi, B_lo = (np.asarray(x, dtype=np.float64) for x in (A_hi, A_lo, B_hi, B_lo))
    e = row_exponents(A_hi)
    f = col_exponents(B_hi)
    DA = split_rows(A_hi, A_lo, e)
    DB = split_cols(B_hi, B_lo, f)
    P = slice_products(DA, DB)
    C_hi, C_lo = recombine(P, e, f)
    return C_hi, C_lo, e, f, DA, DB, P
