"""The 8-bit-part variant for multiple doubles (quad double: 4 doubles, 27
parts of 8 bits, 378 pairs).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2: the rewriting
works for general multiple doubles (a quartered quad double has 16 times the
size of a double; Tables 1 and 2 cover quad doubles).  This module applies the
8-bit balanced parts of oracle.slices_bf16 to an element given as n doubles
(x = x_0 + ... + x_(n-1)):

* exponent e' = (the 13-bit method's exponent of the leading doubles) + 1;
* X = trunc(x 2^(8 S - e')) with |X| < 2^(8 S - 1);
* the S balanced base-256 digits of X (least significant first,
  D = ((X + 128) mod 256) - 128, the top digit the rest);
* P_d = sum_{s+t=d} A_s @ B_t for d = 0 .. S-1 (S (S+1) / 2 pairs);
* Z = sum_d P_d 256^(S-1-d) exactly, rounded once into n non-overlapping
  doubles of Z 2^(e'_i + f'_j - 8 (S+1)) (x_0 = RN(X), x_1 = RN(X - x_0), ...).

S = 13 for double doubles (104 bits) and S = 27 for quad doubles (216 bits, the
208 bits of the 16 13-bit quarters plus a part).  Readings as in
oracle.slices_bf16 and oracle.slices_md.
"""
from __future__ import annotations

import numpy as np

from . import slices, slices_md

DIGIT_BITS = 8
HALF = 1 << (DIGIT_BITS - 1)
QD_PARTS = 27


def pairs(S: int) -> int:
    return S * (S + 1) // 2


def row_exponents(A0: np.ndarray) -> np.ndarray:
    return slices.row_exponents(A0) + 1


def col_exponents(B0: np.ndarray) -> np.ndarray:
    return slices.col_exponents(B0) + 1


def fixed_point(parts, e: int, S: int) -> int:
    """X = trunc((sum of parts) 2^(8 S - e)) as a signed Python integer."""
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
    if X >= 1 << (DIGIT_BITS * S - 1):
        raise ValueError("element not below 2^(e-1): shared exponent too small")
    return sign * X


def balanced_digits(X: int, S: int) -> list[int]:
    D = [0] * S
    for s in range(S - 1, 0, -1):
        d = (X + HALF) % (1 << DIGIT_BITS) - HALF
        D[s] = d
        X = (X - d) >> DIGIT_BITS
    D[0] = X
    return D


def digits_of(parts, e: int, S: int) -> list[int]:
    return balanced_digits(fixed_point(parts, e, S), S)


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
    """P[d] = sum_{s+t=d} DA[s] @ DB[t], d = 0 .. S-1, as exact int64."""
    S, M, K = DA.shape
    N = DB.shape[2]
    if S * K * HALF * HALF >= 2 ** 62:
        raise ValueError("K too large for int64 part sums")
    P = np.zeros((S, M, N), dtype=np.int64)
    for d in range(S):
        for s in range(d + 1):
            P[d] += DA[s] @ DB[d - s]
    return P


def recombine(P: np.ndarray, e, f, nout: int):
    """Z = sum_d P_d 256^(S-1-d), exact, rounded once into nout doubles of
    Z 2^(e_i + f_j - 8 (S+1))."""
    S, M, N = P.shape
    outs = [np.zeros((M, N)) for _ in range(nout)]
    base = -DIGIT_BITS * (S + 1)
    for i in range(M):
        for j in range(N):
            Z = 0
            for d in range(S):
                Z += int(P[d, i, j]) << (DIGIT_BITS * (S - 1 - d))
            q = base + int(e[i]) + int(f[j])
            for p in range(nout):
                v = slices_md.round_scaled(Z, q)
                outs[p][i, j] = v + 0.0
                if v == 0.0 or not np.isfinite(v):
                    break
                Z -= slices_md._units(v, q)
    return outs


def sliced_gemm(A_parts, B_parts, S: int = QD_PARTS):
    """The whole variant; returns (C parts, e, f, DA, DB, P)."""
    A_parts = [np.asarray(a, dtype=np.float64) for a in A_parts]
    B_parts = [np.asarray(b, dtype=np.float64) for b in B_parts]
    e = row_exponents(A_parts[0])
    f = col_exponents(B_parts[0])
    DA = split_rows(A_parts, e, S)
    DB = split_cols(B_parts, f, S)
    P = slice_products(DA, DB)
    C = recombine(P, e, f, len(A_parts))
    return C, e, f, DA, DB, P
