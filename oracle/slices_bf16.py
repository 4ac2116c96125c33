"""The method's steps with 8-bit parts for 16-bit tensor cores (the variant
that runs the slice-pair products on GB300's bf16 tensor cores).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 1, relates its
rewriting to the Ozaki scheme, where accurate products come out of lower
precision arithmetic, and Section 2 eqs. (1)-(5) show why the rewriting is
exact: parts on one shared grid have few nonzero bits, so their products and
the sums of those products are exact in the accumulator.  "Ozaki 2.5:
Engineering the Deconstruction Path of fp64-Emulated Dense Matrix
Multiplication on FP8 Tensor Cores" (summary) does the same on 8-bit tensor
pipes.  This module keeps the steps of oracle.slices and changes only the
width of a part, so that a part fits a bf16 significand:

* exponent: e = (the smallest e with max |hi| < 2^e over the row / column) + 1,
  so that |x| 2^-e < 1/2 (one bit of headroom for balanced digits);
* X = trunc((hi + lo) 2^(8 S - e)), truncation toward zero (as the 13-bit
  quarters), S = 13 parts, so |X| < 2^(8 S - 1);
* balanced base-256 digits of X, least significant first:
  D_s = ((X_s + 128) mod 256) - 128 for s = S-1 .. 1, X_(s-1) = (X_s - D_s)/256,
  and D_0 the remaining X_0.  Then D_s in [-128, 127] for s >= 1,
  D_0 in [-128, 128], X = sum_s D_s 256^(S-1-s) exactly, and every part is an
  integer of magnitude <= 128, exact in bf16 (8-bit significand);
* P_d = sum_{s+t=d} A_s @ B_t for d = 0 .. S-1 (91 pairs): exact integers,
  |P_d| <= (d+1) K 2^14;
* the parts of the product summed exactly, Z = sum_d P_d 256^(S-1-d), and
  rounded once to the nearest double double:
  C = RN_dd(Z 2^(e_i + f_j - 8 (S + 1))).

Readings (the pages fix none of these for 8-bit parts): truncation toward
zero of the fixed-point value; balanced digits (one sign bit per part is not
spent, so 8-bit parts carry 8 bits); S = 13 (103 bits of the grid, about the
104 of the 13-bit quarters); the pairs of index sum <= S - 1; one rounding at
the end, as for the multiple doubles of oracle.slices_md.
"""
from __future__ import annotations

import numpy as np

from . import slices, slices_md

S = 13             # parts per double double
DIGIT_BITS = 8     # bits per part
FIX_BITS = S * DIGIT_BITS   # 104 fraction bits of the fixed-point value
HALF = 1 << (DIGIT_BITS - 1)
PAIRS = S * (S + 1) // 2    # 91 pairs with s + t <= S - 1


def row_exponents(A_hi: np.ndarray) -> np.ndarray:
    """Shared exponent of each row of A: one more than the exponent of the
    13-bit method, so that |x| 2^-e < 1/2 for every element of the row."""
    return slices.row_exponents(A_hi) + 1


def col_exponents(B_hi: np.ndarray) -> np.ndarray:
    """Shared exponent of each column of B (as row_exponents, over k)."""
    return slices.col_exponents(B_hi) + 1


def fixed_point(hi: float, lo: float, e: int) -> int:
    """X = trunc((hi + lo) 2^(104 - e)) as a signed Python integer."""
    n1, d1 = float(hi).as_integer_ratio()
    n2, d2 = float(lo).as_integer_ratio()
    num = n1 * d2 + n2 * d1
    den = d1 * d2
    sign = -1 if num < 0 else 1
    num = abs(num)
    shift = FIX_BITS - e
    if shift >= 0:
        num <<= shift
    else:
        den <<= -shift
    X = num // den
    if X >= 1 << (FIX_BITS - 1):
        raise ValueError("element not below 2^(e-1): shared exponent too small")
    return sign * X


def balanced_digits(X: int) -> list[int]:
    """The S balanced base-256 digits of X (most significant first)."""
    D = [0] * S
    for s in range(S - 1, 0, -1):
        d = (X + HALF) % (1 << DIGIT_BITS) - HALF   # Python % is a floor mod
        D[s] = d
        X = (X - d) >> DIGIT_BITS                     # exact division
    D[0] = X
    return D


def digits_of(hi: float, lo: float, e: int) -> list[int]:
    return balanced_digits(fixed_point(hi, lo, e))


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


def slice_products(DA: np.ndarray, DB: np.ndarray) -> np.ndarray:
    """P[d] = sum_{s+t=d} DA[s] @ DB[t], d = 0 .. S-1, as exact int64."""
    _, M, K = DA.shape
    N = DB.shape[2]
    if S * K * HALF * HALF >= 2 ** 62:
        raise ValueError("K too large for int64 part sums")
    P = np.zeros((S, M, N), dtype=np.int64)
    for d in range(S):
        for s in range(d + 1):
            P[d] += DA[s] @ DB[d - s]
    return P


def recombine(P: np.ndarray, e, f):
    """Z = sum_d P_d 256^(S-1-d), exact; C = RN_dd(Z 2^(e_i + f_j - 8 (S+1)))."""
    _, M, N = P.shape
    C_hi = np.zeros((M, N))
    C_lo = np.zeros((M, N))
    base = -DIGIT_BITS * (S + 1)
    for i in range(M):
        for j in range(N):
            Z = 0
            for d in range(S):
                Z += int(P[d, i, j]) << (DIGIT_BITS * (S - 1 - d))
            q = base + int(e[i]) + int(f[j])
            hi = slices_md.round_scaled(Z, q)
            C_hi[i, j] = hi + 0.0
            if hi != 0.0 and np.isfinite(hi):
                C_lo[i, j] = slices_md.round_scaled(Z - slices_md._units(hi, q), q) + 0.0
    return C_hi, C_lo


def sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo):
    """The whole variant on the CPU.  Returns (C_hi, C_lo, e, f, DA, DB, P)."""
    A_hi, A_lo, B_hi, B_lo = (np.asarray(x, dtype=np.float64) for x in (A_hi, A_lo, B_hi, B_lo))
    e = row_exponents(A_hi)
    f = col_exponents(B_hi)
    DA = split_rows(A_hi, A_lo, e)
    DB = split_cols(B_hi, B_lo, f)
    P = slice_products(DA, DB)
    C_hi, C_lo = recombine(P, e, f)
    return C_hi, C_lo, e, f, DA, DB, P
