"""The identities the GPU recombination kernels round with, checked against
exact greedy rounding (x_0 = RN(Z 2^q), x_1 = RN(Z 2^q - x_0), ...) on the
CPU.  The kernels read each part of the expansion straight off the bits of
|Z|: with L the lowest set bit of |Z|, every remainder keeps L as its lowest
set bit, and after an odd number of roundings up its bits above L are those
of |Z| inverted (2^p - T = ~(T - 1), whose bits at and below L are T's).
These tests restate that rule in Python and compare it with rounding done in
exact rational arithmetic; the kernels themselves are compared with the
oracle bit for bit in the GPU tests."""
import random
from fractions import Fraction

from tests.exact_ref import rne


def greedy(Z, q, nout):
    out, X = [], Fraction(Z) * Fraction(2) ** q
    for _ in range(nout):
        v = rne(X) + 0.0
        out.append(v)
        if v == 0.0:
            return out + [0.0] * (nout - len(out))
        X -= Fraction(v)
    return out


def bit_scan(Z, q, nout, invert=True, sticky=True):
    """The parts of Z 2^q from the bits of |Z| alone (no remainder formed).
    invert / sticky switch parts of the rule off, for the planted mistakes."""
    sign, m = (1, -Z) if Z < 0 else (0, Z)
    if m == 0:
        return [0.0] * nout
    L = (m & -m).bit_length() - 1
    bit = lambda j: (m >> j) & 1 if j >= 0 else 0
    pos, inv, out = m.bit_length(), False, []
    for _ in range(nout):
        if pos <= L:
            out.append(0.0)
            continue
        flip = inv and invert
        top = next((j for j in range(pos - 1, L, -1) if (1 - bit(j) if flip else bit(j))), L)
        lo = top - 53                                  # the round bit
        w = sum(((1 - bit(j) if flip and j > L else bit(j)) << (j - lo)) for j in range(lo, top + 1))
        keep = w >> 1
        if keep >> 52 != 1:
            return None                                # the rule broke down
        up = (w & 1) and ((sticky and L < lo) or (keep & 1))  # sticky: a set bit below the round bit
        v = float(Fraction(keep + up) * Fraction(2) ** (top - 52 + q))
        out.append(-v if sign else v)
        pos = top - 52
        if up:
            inv, sign = not inv, sign ^ 1
    return [v + 0.0 for v in out]


def _cases(rng, n):
    for _ in range(n):
        nb = rng.choice([54, 60, 120, 300, 500, 900])
        Z = rng.getrandbits(nb) | 1 << (nb - 1)
        if rng.random() < 0.3:                        # a run of ones at the bottom
            Z |= (1 << rng.randrange(nb)) - 1
        if rng.random() < 0.3:                        # a lone bit under a run of zeros: ties
            k = rng.randrange(1, nb)
            Z = (Z >> k << k) | 1 << (k - 1)
        yield -Z if rng.random() < 0.5 else Z


def test_bit_scan_equals_greedy_rounding():
    rng = random.Random(7)
    cases = list(_cases(rng, 600)) + [
        (2**52 + 1) * 2**300 + 2**299, 2**52 * 2**300 + 2**299,   # ties in the first part
        2**600 + (2**52 + 1) * 2**200 + 2**199,                    # a tie in the second
        2**900 - 1, -(2**900 - 1), 2**500 - 2**200 + 1, 1, 3, 2**53 + 1, 0]
    for Z in cases:
        nb = abs(Z).bit_length()
        q = rng.randint(-1022, max(-1022, 1022 - nb))
        for nout in (2, 4, 16):
            a, b = bit_scan(Z, q, nout), greedy(Z, q, nout)
            assert [x.hex() for x in a] == [x.hex() for x in b], (Z, q, nout)


def _all_agree(**kw):
    rng = random.Random(11)
    for Z in list(_cases(rng, 300)) + [(2**52 + 2) * 2**300 + 2**299 + 1, 2**600 - 2**200 + 1]:
        nb = abs(Z).bit_length()
        q = rng.randint(-1022, max(-1022, 1022 - nb))
        a = bit_scan(Z, q, 8, **kw)
        if a is None or [x.hex() for x in a] != [x.hex() for x in greedy(Z, q, 8)]:
            return False
    return True


def test_planted_mistakes_in_the_rule_are_caught():
    assert _all_agree()
    assert not _all_agree(invert=False)   # remainders after a rounding up left uninverted
    assert not _all_agree(sticky=False)   # bits below the round bit ignored
