"""Model of the comparator: a plain double-double GEMM, one accumulator per
output, k in order.

TEST INFRASTRUCTURE ONLY (see the package docstring).  "Multiple Double
Arithmetic on NVIDIA Tensor Cores", Section 4.2, second method: the product
of double-double matrices where one thread computes one inner product with
double-double additions and multiplications on the regular cores.  The page
does not spell out the double-double operations; the reading taken here is
the usual one (error-free transformations):

    for k = 0 .. K-1:
        p   = a_hi * b_hi                        (rounded)
        e   = a_hi * b_hi - p                    (exact: the product error)
        e   = e + (a_hi * b_lo + a_lo * b_hi)    (rounded, in this order)
        s, t = two_sum(c_hi, p)
        t   = (t + c_lo) + e
        c_hi, c_lo = quick_two_sum(s, t)

The product error is formed exactly with Dekker's splitting (Veltkamp split
by 2^27 + 1); it equals the fused multiply-add a_hi*b_hi - p of the GPU code
bit for bit whenever no intermediate over- or underflows.  Zero results are
+0.
"""
from __future__ import annotations

import numpy as np

_SPLIT = 134217729.0  # 2^27 + 1


def _two_prod_err(a, b, p):
    """Exact a*b - p for p = fl(a*b) (Dekker)."""
    ab = a * _SPLIT
    a1 = ab - (ab - a)
    a2 = a - a1
    bb = b * _SPLIT
    b1 = bb - (bb - b)
    b2 = b - b1
    return ((a1 * b1 - p) + a1 * b2 + a2 * b1) + a2 * b2


def _two_sum(a, b):
    s = a + b
    bb = s - a
    return s, (a - (s - bb)) + (b - bb)


def _quick_two_sum(a, b):
    s = a + b
    return s, b - (s - a)


def simt_dd_gemm(A_hi, A_lo, B_hi, B_lo):
    """(C_hi, C_lo) of the comparator's arithmetic, vectorised over outputs."""
    A_hi, A_lo, B_hi, B_lo = (np.asarray(x, dtype=np.float64) for x in (A_hi, A_lo, B_hi, B_lo))
    M, K = A_hi.shape
    N = B_hi.shape[1]
    c_hi = np.zeros((M, N))
    c_lo = np.zeros((M, N))
    for k in range(K):
        a_hi = A_hi[:, k:k + 1]
        a_lo = A_lo[:, k:k + 1]
        b_hi = B_hi[k:k + 1, :]
        b_lo = B_lo[k:k + 1, :]
        p = a_hi * b_hi
        e = _two_prod_err(a_hi, b_hi, p)
        e = e + (a_hi * b_lo + a_lo * b_hi)
        s, t = _two_sum(c_hi, p)
        t = (t + c_lo) + e
        c_hi, c_lo = _quick_two_sum(s, t)
    return c_hi + 0.0, c_lo + 0.0
