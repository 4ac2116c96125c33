// fixed_point.cuh -- the exact fixed-point value of a double double against
// a shared exponent: X = floor(|hi + lo| 2^(104 - e)) in 128-bit integer
// arithmetic, and the sign of the element.
//
// With |hi| = mh 2^Eh (mh < 2^53) and a normalised lo (|lo| <= ulp(hi)/2),
// put a = |hi| 2^(104-e) = mh 2^sh and b = |lo| 2^(104-e) <= 2^(sh-1):
//   same signs:      floor(a + b) = floor(a) + floor(b)
//                    (sh >= 0: a is an integer; sh < 0: b < 1/2 and
//                     frac(a) + b < 1)
//   opposite signs:  floor(a - b) = floor(a) - floor(b) - borrow, where
//                    borrow = [frac(b) > 0] when sh >= 0 (frac(a) = 0), and
//                    borrow = [frac(a) == 0] when sh < 0 (then 0 < b < 2^sh
//                    and frac(a) is 0 or >= 2^sh).
// The borrow is the move of "Multiple Double Arithmetic on NVIDIA Tensor
// Cores", Problem 3.3, eq. (7): the low double's opposite sign is taken from
// the high digits without changing the value.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace ddg {
namespace fxp {

constexpr int FIX_BITS = 104;
constexpr uint64_t ABS_MASK = 0x7FFFFFFFFFFFFFFFULL;

struct Unpacked {
    uint64_t m;  // integer significand (< 2^53)
    int E;       // |x| = m * 2^E
};

__device__ __forceinline__ Unpacked unpack_abs(uint64_t bits) {
    uint64_t a = bits & ABS_MASK;
    int biased = (int)(a >> 52);
    uint64_t frac = a & ((1ULL << 52) - 1);
    Unpacked u;
    if (biased == 0) { u.m = frac; u.E = -1074; }
    else { u.m = frac | (1ULL << 52); u.E = biased - 1075; }
    return u;
}

// floor(m * 2^sh) for m < 2^53 (shifts beyond the 104-bit window are clamped
// so that out-of-contract inputs cannot shift by >= 128).
__device__ __forceinline__ unsigned __int128 scaled_floor(uint64_t m, int sh) {
    if (sh >= 0) return (unsigned __int128)m << (sh > 74 ? 74 : sh);
    if (sh <= -64) return 0;
    return (unsigned __int128)(m >> (-sh));
}

__device__ __forceinline__ bool scaled_frac_zero(uint64_t m, int sh) {
    if (sh >= 0) return true;
    if (sh <= -64) return m == 0;
    return (m & ((1ULL << (-sh)) - 1)) == 0;
}

// X = floor(|hi + lo| * 2^(104 - e)) and the sign of the element.
__device__ __forceinline__ unsigned __int128 fixed_point(double hi, double lo, int e, uint64_t& sign_out) {
    uint64_t hb = f64_bits(hi);
    uint64_t lb = f64_bits(lo);
    if ((hb & ABS_MASK) == 0) { hb = lb; lb = 0; }  // hi = 0: the element is lo alone
    const uint64_t sign = hb >> 63;
    unsigned __int128 X = 0;
    if ((hb & ABS_MASK) != 0) {
        Unpacked h = unpack_abs(hb);
        int sh = h.E + FIX_BITS - e;
        X = scaled_floor(h.m, sh);
        if ((lb & ABS_MASK) != 0) {
            Unpacked l = unpack_abs(lb);
            int sl = l.E + FIX_BITS - e;
            unsigned __int128 bint = scaled_floor(l.m, sl);
            if ((lb >> 63) == sign) {
                X += bint;
            } else {
                bool borrow = (sh >= 0) ? !scaled_frac_zero(l.m, sl) : scaled_frac_zero(h.m, sh);
                X -= bint + (borrow ? 1 : 0);
            }
        }
    }
    sign_out = sign;
    return X;
}

}  // namespace fxp
}  // namespace ddg
