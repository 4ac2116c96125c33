// exact_round.cuh -- the exact sum of part sums on a base-256 grid and its
// rounding into non-overlapping doubles, with 64-bit limbs (the bf16
// variants' recombination).
//
//   Z = sum_{d=0}^{NP-1} v_d 256^(NP-1-d),   |v_d| < 2^46,
//
// is formed exactly either in W 64-bit limbs (two's complement, least
// significant first) by Horner's rule over groups of three parts (a group
// v_a 2^16 + v_b 2^8 + v_c stays below 2^63), or as 64-bit column sums of its
// 32-bit words followed by one carry pass.  Z 2^q is rounded into NOUT
// doubles x_0 = RN(Z 2^q), x_1 = RN(Z 2^q - x_0), ... (ties to even) by the
// limb routines below (the fast ones need every part to be a normal double:
// q >= -1022, so that a nonzero remainder is at least 2^q, and the result
// below 2^1023), or by the general routine with gradual underflow.
#pragma once

#include <cstdint>

#include "wide_int.cuh"

namespace ddg {
namespace xr {

// Z = Z 2^SH + h for 0 < SH < 64 and a signed h (|h| < 2^63).
template <int W, int SH>
__device__ __forceinline__ void horner(uint64_t (&z)[W], long long h) {
#pragma unroll
    for (int i = W - 1; i > 0; --i) z[i] = (z[i] << SH) | (z[i - 1] >> (64 - SH));
    z[0] <<= SH;
    const uint64_t s = (uint64_t)(h >> 63);  // sign extension of h
    const uint64_t t0 = z[0] + (uint64_t)h;
    uint64_t c = t0 < z[0];
    z[0] = t0;
#pragma unroll
    for (int i = 1; i < W; ++i) {
        const uint64_t u = z[i] + s;
        const uint64_t c1 = u < z[i];
        const uint64_t u2 = u + c;
        c = c1 | (u2 < u);
        z[i] = u2;
    }
}

// v_a 256^(n-1) + ... + v_(a+n-1) for a group of n <= 3 parts.
template <int N>
__device__ __forceinline__ long long group(const long long* v) {
    long long g = v[0];
#pragma unroll
    for (int i = 1; i < N; ++i) g = g * 256 + v[i];
    return g;
}

// Z as W limbs from the NP part sums.
template <int NP, int W>
__device__ __forceinline__ void exact_sum(const long long (&v)[NP], uint64_t (&z)[W]) {
    constexpr int G = NP / 3, R = NP % 3;
    const long long h0 = group<3>(&v[0]);
    z[0] = (uint64_t)h0;
#pragma unroll
    for (int i = 1; i < W; ++i) z[i] = (uint64_t)(h0 >> 63);
#pragma unroll
    for (int g = 1; g < G; ++g) horner<W, 24>(z, group<3>(&v[3 * g]));
    if (R == 1) horner<W, 8>(z, v[NP - 1]);
    if (R == 2) horner<W, 16>(z, group<2>(&v[NP - 2]));
}

template <int W>
__device__ __forceinline__ bool is_zero(const uint64_t (&m)[W]) {
    uint64_t o = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) o |= m[i];
    return o == 0;
}

// Index of the leading 1 of a nonzero magnitude.
template <int W>
__device__ __forceinline__ int msb(const uint64_t (&m)[W]) {
    int t = -1;
#pragma unroll
    for (int i = 0; i < W; ++i)
        if (m[i] != 0) t = 64 * i + 63 - __clzll((long long)m[i]);
    return t;
}

template <int W>
__device__ __forceinline__ void negate(uint64_t (&m)[W]) {
    uint64_t c = 1;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const uint64_t u = ~m[i] + c;
        c = c && (u == 0);
        m[i] = u;
    }
}

// Bits [b, b + 64) of m (b >= 0).
template <int W>
__device__ __forceinline__ uint64_t window(const uint64_t (&m)[W], int b) {
    const int i = b >> 6, o = b & 63;
    uint64_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < W; ++j) {
        if (j == i) lo = m[j];
        if (j == i + 1) hi = m[j];
    }
    return o == 0 ? lo : (lo >> o) | (hi << (64 - o));
}

// Are any bits of m below position b set (b >= 0)?
template <int W>
__device__ __forceinline__ bool any_below(const uint64_t (&m)[W], int b) {
    uint64_t o = 0;
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const int lo = 64 * j;
        if (lo + 64 <= b) o |= m[j];
        else if (lo < b) o |= m[j] & ((1ULL << (b - lo)) - 1);
    }
    return o != 0;
}

// Keep only the bits of m below position p (p >= 0).
template <int W>
__device__ __forceinline__ void keep_below(uint64_t (&m)[W], int p) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const int lo = 64 * j;
        if (lo >= p) m[j] = 0;
        else if (lo + 64 > p) m[j] &= (1ULL << (p - lo)) - 1;
    }
}

// m = 2^p - m for 0 <= m < 2^p (p < 64 W).
template <int W>
__device__ __forceinline__ void complement_to(uint64_t (&m)[W], int p) {
    negate(m);
    uint64_t c = 0;
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const uint64_t add = (j == (p >> 6)) ? (1ULL << (p & 63)) : 0;
        const uint64_t u = m[j] + add;
        const uint64_t c1 = u < m[j];
        const uint64_t u2 = u + c;
        c = c1 | (u2 < u);
        m[j] = u2;
    }
}

// The fast path applies: every part of Z 2^q is a normal double or zero.
template <int W>
__device__ __forceinline__ bool fast_path_ok(const uint64_t (&z)[W], int q) {
    if (q < -1022) return false;
    uint64_t m[W];
#pragma unroll
    for (int i = 0; i < W; ++i) m[i] = z[i];
    if ((int64_t)m[W - 1] < 0) negate(m);
    return is_zero(m) || msb(m) + q <= 1022;
}

// Z 2^q rounded into NOUT doubles (fast path only; +0 for zeros).
template <int W, int NOUT>
__device__ __forceinline__ void round_parts(const uint64_t (&z)[W], int q, double (&out)[NOUT]) {
    uint64_t m[W];
#pragma unroll
    for (int i = 0; i < W; ++i) m[i] = z[i];
    uint64_t sign = (uint64_t)m[W - 1] >> 63;
    if (sign) negate(m);
#pragma unroll
    for (int p = 0; p < NOUT; ++p) {
        if (is_zero(m)) {
            out[p] = 0.0;
            continue;
        }
        const int t = msb(m);
        int pos = t - 52;  // exponent (relative to q) of the last kept bit
        uint64_t keep;
        bool up = false;
        if (pos <= 0) {
            keep = m[0];  // the whole value (< 2^53)
            pos = 0;
#pragma unroll
            for (int i = 0; i < W; ++i) m[i] = 0;
        } else {
            const uint64_t x = window(m, pos - 1);  // round bit, then the 53 kept bits
            keep = x >> 1;
            const bool rbit = x & 1;
            up = rbit && ((keep & 1) || any_below(m, pos - 1));
            keep_below(m, pos);  // the tail below the kept bits
            if (up) {
                complement_to(m, pos);  // |tail - 2^pos|
                keep += 1;
                if (keep >> 53) { keep >>= 1; pos += 1; }
            }
        }
        out[p] = wide::make_double(keep, pos + q, sign);
        if (up) sign ^= 1;  // the remainder has the opposite sign
    }
}


// ---- sums as 64-bit column sums of 32-bit words (deferred carries) ----

// Adds h (|h| < 2^63) at bit offset o (a compile-time constant after
// unrolling) of a number kept as column sums acc[w] of its 32-bit words.
template <int NC>
__device__ __forceinline__ void add_at(long long (&acc)[NC], long long h, int o) {
    const int w = o >> 5, r = o & 31;
    const __int128 G = (__int128)h << r;  // |G| < 2^87
    acc[w] += (long long)(uint32_t)G;
    acc[w + 1] += (long long)(uint32_t)(G >> 32);
    acc[w + 2] += (long long)(G >> 64);
}

// One carry pass over the column sums: the number in W 64-bit limbs (two's
// complement; the caller guarantees it fits).
template <int W, int NC>
__device__ __forceinline__ void carry_to_limbs(const long long (&acc)[NC], uint64_t (&z)[W]) {
    static_assert(NC >= 2 * W, "column sums cover the limbs");
    long long carry = 0;
#pragma unroll
    for (int w = 0; w < 2 * W; w += 2) {
        const long long t0 = acc[w] + carry;
        const long long t1 = acc[w + 1] + (t0 >> 32);
        carry = t1 >> 32;
        z[w / 2] = (uint64_t)(uint32_t)t0 | ((uint64_t)(uint32_t)t1 << 32);
    }
}

// ---- rounding by scanning the bits of |Z| ----
//
// With L the lowest set bit of |Z|, every remainder R of the expansion keeps
// L as its lowest set bit, and below the position reached so far its bits are
// either those of |Z| or, after an odd number of roundings up, those of |Z|
// inverted above L (2^p - T = ~(T - 1) for T with lowest set bit L, and the
// bits at and below L of ~(T - 1) are those of T).  So no remainder is ever
// formed: each part reads 54 bits of |Z| at its leading bit, inverts them
// above L when needed, and the sticky bit is simply L < (round-bit position).

// Bits [lo, lo + 64) of m (lo may be negative: zeros below bit 0; m is held
// in local memory for the dynamic limb index).
template <int W>
__device__ __forceinline__ uint64_t bits_from(const uint64_t* m, int lo) {
    if (lo < 0) return m[0] << (-lo);  // only used with lo > -64
    const int i = lo >> 6, o = lo & 63;
    const uint64_t a = m[i], b = i + 1 < W ? m[i + 1] : 0;
    return o ? (a >> o) | (b << (64 - o)) : a;
}

// Leading bit of the remainder below position pos: the highest set bit of m
// below pos, or with inv the highest clear bit of m in (L, pos), else L.
// -1 if the remainder is 0.
template <int W>
__device__ __forceinline__ int remainder_top(const uint64_t* m, int pos, bool inv, int L) {
    if (pos <= L) return -1;
    const int lL = L >> 6;
    int i = (pos - 1) >> 6;
    uint64_t v = inv ? ~m[i] : m[i];
    if (pos & 63) v &= (1ULL << (pos & 63)) - 1;
#pragma unroll 1
    for (;;) {
        if (i == lL) {
            v &= ~((2ULL << (L & 63)) - 1);  // only bits above L (the bit at L is always set)
            if (v) return 64 * i + 63 - __clzll((long long)v);
            return L;
        }
        if (v) return 64 * i + 63 - __clzll((long long)v);
        --i;
        v = inv ? ~m[i] : m[i];
    }
}

// Z 2^q rounded into nout doubles x_0 = RN(Z 2^q), x_1 = RN(Z 2^q - x_0), ...
// (ties to even; +0 for zeros) when every part is a normal double or zero:
// q >= -1022 and the leading bit of Z 2^q at most 2^1022; otherwise false.
template <int W>
__device__ __forceinline__ bool round_parts_scan(const uint64_t (&z)[W], int q, double* out, int nout) {
    uint64_t m[W];
#pragma unroll
    for (int i = 0; i < W; ++i) m[i] = z[i];
    uint64_t sign = m[W - 1] >> 63;
    if (sign) negate(m);
    int L = -1;
#pragma unroll
    for (int i = W - 1; i >= 0; --i)
        if (m[i] != 0) L = 64 * i + __ffsll((long long)m[i]) - 1;
    if (L < 0) {
        for (int p = 0; p < nout; ++p) out[p] = 0.0;
        return true;
    }
    const int t = msb(m);
    if (q < -1022 || t + q > 1022) return false;
    int pos = t + 1;  // the remainder is the part of |Z| below pos
    bool inv = false, zero = false;
#pragma unroll 1
    for (int p = 0; p < nout; ++p) {
        const int tr = zero ? -1 : remainder_top<W>(m, pos, inv, L);
        if (tr < 0) {
            zero = true;
            out[p] = 0.0;
            continue;
        }
        const int lo = tr - 53;  // round bit
        uint64_t w = bits_from<W>(m, lo) & ((1ULL << 54) - 1);
        if (inv) {  // invert the window above L
            const int b = L - lo;
            w ^= b < 0 ? ((1ULL << 54) - 1) : (((1ULL << 54) - 1) & ~((2ULL << b) - 1));
        }
        const uint64_t keep = w >> 1;  // 53 bits, leading bit set
        const bool up = (w & 1) && (L < lo || (keep & 1));
        out[p] = __longlong_as_double(
            (long long)((sign << 63) | (((uint64_t)(tr + q + 1022) << 52) + keep + (up ? 1 : 0))));
        pos = tr - 52;
        if (up) {
            inv = !inv;
            sign ^= 1;
        }
    }
    return true;
}

// Z 2^q rounded into nout doubles x_0 = RN(Z 2^q), x_1 = RN(Z 2^q - x_0), ...
// for any q: gradual underflow (a part below half the smallest subnormal is
// 0) and overflow (an infinite part) end the expansion, and the remaining
// parts are +0, as in the definition of the exact multiple-double product.
template <int W>
__device__ __forceinline__ void round_parts_general(const uint64_t (&z)[W], int q, double* out, int nout) {
    uint64_t m[W];
#pragma unroll
    for (int i = 0; i < W; ++i) m[i] = z[i];
    uint64_t sign = (uint64_t)m[W - 1] >> 63;
    if (sign) negate(m);
    bool stop = false;
#pragma unroll 1
    for (int p = 0; p < nout; ++p) {
        if (stop || is_zero(m)) {
            out[p] = 0.0;
            stop = true;
            continue;
        }
        const int t = msb(m);
        int pos = max(t - 52, -1074 - q);  // last kept bit, relative to q
        uint64_t keep = 0;
        bool up = false;
        if (pos <= 0) {
            keep = m[0];  // exact (t <= 52)
            pos = 0;
#pragma unroll
            for (int i = 0; i < W; ++i) m[i] = 0;
        } else if (pos - 1 <= t) {
            const uint64_t x = window(m, pos - 1);
            keep = x >> 1;
            up = (x & 1) && ((keep & 1) || any_below(m, pos - 1));
            keep_below(m, pos);
            if (up) {
                complement_to(m, pos);
                keep += 1;
                if (keep >> 53) { keep >>= 1; pos += 1; }
            }
        }  // else: below half the smallest subnormal, rounds to 0
        const double v = wide::make_double(keep, pos + q, sign);
        if (keep == 0 || isinf(v)) stop = true;
        out[p] = keep == 0 ? 0.0 : v;
        if (up) sign ^= 1;
    }
}

}  // namespace xr
}  // namespace ddg
