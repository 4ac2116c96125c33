// wide_int.cuh -- 256-bit two's-complement integers and the correctly rounded
// conversion of an exact integer times a power of two into non-overlapping
// doubles (used where the parts of a product are summed exactly and rounded
// once).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace ddg {
namespace wide {

typedef unsigned __int128 u128;

struct U256 {
    u128 lo, hi;
};

__device__ __forceinline__ U256 u256_zero() { return U256{0, 0}; }

__device__ __forceinline__ U256 u256_add(U256 a, U256 b) {
    U256 r;
    r.lo = a.lo + b.lo;
    r.hi = a.hi + b.hi + (r.lo < a.lo ? 1 : 0);
    return r;
}

__device__ __forceinline__ U256 u256_neg(U256 a) {
    U256 r;
    r.lo = ~a.lo + 1;
    r.hi = ~a.hi + (r.lo == 0 ? 1 : 0);
    return r;
}

__device__ __forceinline__ bool u256_is_neg(U256 a) { return (uint64_t)(a.hi >> 127) != 0; }
__device__ __forceinline__ bool u256_is_zero(U256 a) { return a.lo == 0 && a.hi == 0; }

// m * 2^sh for m < 2^64, 0 <= sh <= 190.
__device__ __forceinline__ U256 u256_shl(uint64_t m, int sh) {
    U256 r;
    if (sh >= 128) {
        r.lo = 0;
        r.hi = (u128)m << (sh - 128);
    } else if (sh == 0) {
        r.lo = m;
        r.hi = 0;
    } else {
        r.lo = (u128)m << sh;
        r.hi = (u128)m >> (128 - sh);
    }
    return r;
}

// v * 2^sh for a signed v (|v| < 2^63), 0 <= sh <= 190.
__device__ __forceinline__ U256 u256_from_signed(long long v, int sh) {
    const U256 t = u256_shl((uint64_t)(v < 0 ? -v : v), sh);
    return v < 0 ? u256_neg(t) : t;
}

// Bits [off, off + n) of a, n <= 32.
__device__ __forceinline__ uint32_t u256_bits(U256 a, int off, int n) {
    const uint32_t mask = (n == 32) ? 0xFFFFFFFFu : ((1u << n) - 1);
    if (off >= 128) return (uint32_t)(a.hi >> (off - 128)) & mask;
    if (off + n <= 128) return (uint32_t)(a.lo >> off) & mask;
    return (uint32_t)((a.lo >> off) | (a.hi << (128 - off))) & mask;
}

__device__ __forceinline__ int u256_msb(U256 a) {  // a != 0, non-negative
    if (a.hi != 0) {
        const uint64_t h1 = (uint64_t)(a.hi >> 64);
        return h1 ? 255 - __clzll((long long)h1) : 191 - __clzll((long long)(uint64_t)a.hi);
    }
    const uint64_t l1 = (uint64_t)(a.lo >> 64);
    return l1 ? 127 - __clzll((long long)l1) : 63 - __clzll((long long)(uint64_t)a.lo);
}

// a >> sh (logical), 0 < sh < 256.
__device__ __forceinline__ U256 u256_shr(U256 a, int sh) {
    U256 r;
    if (sh >= 128) {
        r.lo = a.hi >> (sh - 128);
        r.hi = 0;
    } else {
        r.lo = (a.lo >> sh) | (a.hi << (128 - sh));
        r.hi = a.hi >> sh;
    }
    return r;
}

// Are any of the bits below position `sh` set (sh >= 1)?
__device__ __forceinline__ bool u256_any_below(U256 a, int sh) {
    if (sh >= 256) return !u256_is_zero(a);
    if (sh >= 128) return a.lo != 0 || (sh > 128 && (a.hi << (256 - sh)) != 0);
    return (a.lo << (128 - sh)) != 0;
}

// keep * 2^lsb as a double (keep <= 2^53, exact when representable);
// +-inf when it reaches 2^1024.  IEEE 754 binary64 layout.
__device__ __forceinline__ double make_double(uint64_t keep, int lsb, uint64_t sign) {
    if (keep == 0) return __longlong_as_double((long long)(sign << 63));
    const int t = 63 - __clzll((long long)keep);
    const int E = lsb + t;  // exponent of the leading bit
    uint64_t bits;
    if (E > 1023) {
        bits = 0x7FF0000000000000ULL;
    } else if (E >= -1022) {
        const uint64_t mant = (keep << (52 - t)) & ((1ULL << 52) - 1);
        bits = ((uint64_t)(E + 1023) << 52) | mant;
    } else {
        bits = keep << (lsb + 1074);  // subnormal: lsb >= -1074 by construction
    }
    return __longlong_as_double((long long)((sign << 63) | bits));
}

// X * 2^q rounded into NOUT non-overlapping doubles: x_0 = RN(X 2^q),
// x_1 = RN(X 2^q - x_0), ... (round to nearest, ties to even, gradual
// underflow).  After a zero or an infinite part the remaining parts are +0.
// Zeros are written as +0.
template <int NOUT>
__device__ __forceinline__ void round_into_doubles(U256 X, int q, double (&out)[NOUT]) {
    bool stop = false;
#pragma unroll
    for (int p = 0; p < NOUT; ++p) {
        double v = 0.0;
        if (!stop && !u256_is_zero(X)) {
            const uint64_t sign = u256_is_neg(X) ? 1ULL : 0ULL;
            const U256 mag = sign ? u256_neg(X) : X;
            const int t = u256_msb(mag);
            const int top = q + t;
            const int lsb = max(top - 52, -1074);
            const int shift = lsb - q;
            uint64_t keep;
            int klsb;
            U256 used;  // the rounded magnitude in units of 2^q
            if (shift <= 0) {
                keep = (uint64_t)mag.lo;
                klsb = q;
                used = mag;
            } else {
                keep = (uint64_t)u256_shr(mag, shift).lo;
                const bool rbit = u256_bits(mag, shift - 1, 1) != 0;
                const bool sticky = shift >= 2 && u256_any_below(mag, shift - 1);
                if (rbit && (sticky || (keep & 1))) keep += 1;
                klsb = lsb;
                used = u256_shl(keep, shift);
                if (keep >> 53) { keep >>= 1; klsb += 1; }  // rounded up to 2^53
            }
            v = make_double(keep, klsb, sign);
            if (isinf(v)) stop = true;
            else X = u256_add(X, sign ? used : u256_neg(used));
        } else {
            stop = true;
        }
        // +0 for a zero of either sign (integer test: no FP64 operation)
        out[p] = (f64_bits(v) << 1) == 0 ? 0.0 : v;
    }
}

}  // namespace wide
}  // namespace ddg
