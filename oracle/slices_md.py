"""The method's steps for multiple doubles with more parts (quad double:
4 doubles, S = 16 parts of 13 bits, 136 pairs).

TEST INFRASTRUCTURE ONLY (see the package docstring).  "Multiple Double
Arithmetic on NVIDIA Tensor Cores": the algorithms of Section 2 work for
general multiple doubles; a quartered quad double has 16 times the size of a
double (Section 2), Table 2 lists the dimensions for qd, od and hd, and
Table 1 reports quad-double runs.  The steps are those of oracle.slices with
S parts: a shared exponent per row / column, the S truncating base-2^13
digits of |x| 2^-e (x the sum of the element's parts), part sums P_d over the
pairs s + t = d <= S - 1, and the parts of the product summed.

Reading for the last step (the page prescribes double-double summation only
for double doubles): the sum of the parts is formed exactly (all P_d are
integers, all weights powers of two) and rounded once into n non-overlapping
doubles, x_0 = RN(X), x_1 = RN(X - x_0), ...  For S = 16 every P_d stays below
2^53 when K <= 2^23 (16 K (2^13 - 1)^2 < 2^53).
"""
from __future__ import annotations

import math

import numpy as np

from . import slices

DIGIT_BITS = 13


def max_k(S: int) -> int:
    """Largest power-of-two K for which S K (2^13 - 1)^2 < 2^53."""
    k = 1
    while S * (2 * k) * ((1 << DIGIT_BITS) - 1) ** 2 < 2 ** 53:
        k *= 2
    return k


def digits_of(parts, e: int, S: int) -> list[int]:
    """The S truncating base-2^13 digits of (sum of parts) 2^-e, signed."""
    num, den = 0, 1
    for x in parts:
        n, d = float(x).as_integer_ratio()
        num, den = num * d + n * den, den * d
    sign = -1 if num < 0 else 1
    num = abs(num)
    shift = DIGIT_BITS * S - e
    if shift >= 0:
        num <<= shift
    else:
        den <<= -shift
    X = num // den
    if X >= 1 << (DIGIT_BITS * S):
        raise ValueError("element not below 2^e")
    mask = (1 << DIGIT_BITS) - 1
    return [sign * ((X >> (DIGIT_BITS * (S - 1 - s))) & mask) for s in range(S)]


def split_rows(A_parts, e, S: int) -> np.ndarray:
    M, K = A_parts[0].shape
    D = np.zeros((S, M, K), dtype=np.int64)
    for i in range(M):
        for k in range(K):
            D[:, i, k] = digits_of([a[i, k] for a in A_parts], int(e[i]), S)
    return D


def split_cols(B_parts, f, S: int) -> np.ndarray:
    K, N = B_parts[0].shape
    D = np.zeros((S, K, N), dtype=np.int64)
    for j in range(N):
        for k in range(K):
            D[:, k, j] = digits_of([b[k, j] for b in B_parts], int(f[j]), S)
    return D


def slice_products(DA: np.ndarray, DB: np.ndarray) -> np.ndarray:
    """P[d] = sum_{s+t=d} DA[s] @ DB[t], d = 0..S-1, as exact integers in
    float64 (every partial sum below 2^53, checked)."""
    S, M, K = DA.shape
    N = DB.shape[2]
    assert S * K * ((1 << DIGIT_BITS) - 1) ** 2 < 2 ** 53
    P = np.zeros((S, M, N))
    for d in range(S):
        acc = np.zeros((M, N))
        for s in range(d + 1):
            acc += DA[s].astype(np.float64) @ DB[d - s].astype(np.float64)
        P[d] = acc
    return P


def round_scaled(n: int, q: int) -> float:
    """n * 2^q rounded to the nearest double, ties to even, gradual underflow."""
    if n == 0:
        return 0.0
    sign = -1.0 if n < 0 else 1.0
    m = abs(n)
    top = m.bit_length() - 1 + q          # exponent of the leading bit
    lsb = max(top - 52, -1074)            # exponent of the last kept bit
    shift = lsb - q
    if shift <= 0:
        keep, lsb = m, q                  # representable as it is
    else:
        keep = m >> shift
        rem = m - (keep << shift)
        half = 1 << (shift - 1)
        if rem > half or (rem == half and keep & 1):
            keep += 1
    if keep.bit_length() + lsb > 1024:
        return sign * math.inf
    return sign * math.ldexp(float(keep), lsb)


def _units(v: float, q: int) -> int:
    """v / 2^q as an exact integer (v lies on the 2^q grid)."""
    n, d = v.as_integer_ratio()
    num, den = (n, d << q) if q >= 0 else (n << (-q), d)
    assert num % den == 0
    return num // den


def recombine(P: np.ndarray, e, f, nout: int):
    """Sum of P_d 2^(-13(d+2)) 2^(e_i + f_j), exact, rounded once into `nout`
    non-overlapping doubles (x_0 = RN(X), x_1 = RN(X - x_0), ...)."""
    S, M, N = P.shape
    outs = [np.zeros((M, N)) for _ in range(nout)]
    base = -DIGIT_BITS * (S + 1)          # weight of the last digit position
    for i in range(M):
        for j in range(N):
            X = 0
            for d in range(S):
                X += int(P[d, i, j]) << (DIGIT_BITS * (S - 1 - d))
            q = base + int(e[i]) + int(f[j])
            for p in range(nout):
                v = round_scaled(X, q)
                outs[p][i, j] = v + 0.0
                if v == 0.0 or not math.isfinite(v):
                    break
                X -= _units(v, q)
    return outs


def sliced_md_gemm(A_parts, B_parts, S: int = 16):
    """The whole method for multiple doubles; returns (C parts, e, f, DA, DB, P)."""
    A_parts = [np.asarray(a, dtype=np.float64) for a in A_parts]
    B_parts = [np.asarray(b, dtype=np.float64) for b in B_parts]
    e = slices.row_exponents(A_parts[0])
    f = slices.col_exponents(B_parts[0])
    DA = split_rows(A_parts, e, S)
    DB = split_cols(B_parts, f, S)
    P = slice_products(DA, DB)
    C = recombine(P, e, f, len(A_parts))
    return C, e, f, DA, DB, P
