"""Exact rational reference used to pin the oracle: Python Fractions and a
round-to-nearest-even written from the IEEE 754 definition (binary64,
gradual underflow).  Independent of oracle/ and of the CUDA library."""
from __future__ import annotations

import math
from fractions import Fraction


def pow2(k: int) -> Fraction:
    return Fraction(1 << k) if k >= 0 else Fraction(1, 1 << -k)


def rne(x: Fraction) -> float:
    """x rounded to the nearest binary64 value, ties to even (+0 for 0)."""
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    a = abs(x)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    while pow2(E) > a:
        E -= 1
    while pow2(E + 1) <= a:
        E += 1
    q = max(E - 52, -1074)
    m = a / pow2(q)
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    if n * pow2(q) >= pow2(1024):
        return sign * math.inf
    return sign * math.ldexp(float(n), q)


def exact_entry(A_hi, A_lo, B_hi, B_lo, i: int, j: int) -> Fraction:
    K = A_hi.shape[1]
    return sum(((Fraction(float(A_hi[i, k])) + Fraction(float(A_lo[i, k])))
                * (Fraction(float(B_hi[k, j])) + Fraction(float(B_lo[k, j])))
                for k in range(K)), Fraction(0))


def nearest_dd(x: Fraction):
    """(RN(x), RN(x - RN(x))); a word that rounds to zero is +0 (the sign of
    an underflowed zero is not kept)."""
    hi = rne(x)
    lo = rne(x - Fraction(hi)) if math.isfinite(hi) else 0.0
    return hi + 0.0, lo + 0.0


def bits(x: float) -> int:
    import struct
    return struct.unpack("<q", struct.pack("<d", x))[0]
