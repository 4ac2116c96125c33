// fixed_point_md.cuh -- the exact fixed-point value of a quad double (four
// non-overlapping doubles) against a shared exponent, in 256-bit integer
// arithmetic: X = floor(|x0 + x1 + x2 + x3| 2^(FIXB - e)) and the sign.
#pragma once

#include <cstdint>

#include "wide_int.cuh"

namespace ddg {
namespace fxp {

using wide::U256;
using wide::u256_add;
using wide::u256_neg;
using wide::u256_shl;
using wide::u256_zero;

struct UnpQ {
    uint64_t m;
    int E;  // |x| = m 2^E
};

__device__ __forceinline__ UnpQ unpack_abs_q(uint64_t bits) {
    const uint64_t a = bits & 0x7FFFFFFFFFFFFFFFULL;
    const int biased = (int)(a >> 52);
    UnpQ u;
    if (biased == 0) { u.m = a & ((1ULL << 52) - 1); u.E = -1074; }
    else { u.m = (a & ((1ULL << 52) - 1)) | (1ULL << 52); u.E = biased - 1075; }
    return u;
}

// X = floor(|x0 + x1 + x2 + x3| 2^(FIXB - e)) for a normalised quad double
// (|x_{p+1}| <= ulp(x_p) / 2) and the sign of the element.  With every part
// signed relative to the leading one, the parts that are integers at this
// scale add exactly; at the first part j with a fraction, floor(a_j + rest)
// = floor(a_j) when a_j has a nonzero fraction (the rest is below half its
// last bit), else floor(a_j) - 1 when the first nonzero later part is
// negative (the borrow of Problem 3.3, eq. (7)).
template <int FIXB>
__device__ __forceinline__ U256 fixed_point_qd(const double (&x)[4], int e, uint64_t& sign_out) {
    int lead = -1;
#pragma unroll
    for (int p = 3; p >= 0; --p)
        if ((f64_bits(x[p]) & 0x7FFFFFFFFFFFFFFFULL) != 0) lead = p;
    sign_out = 0;
    if (lead < 0) return u256_zero();
    const uint64_t sign = f64_bits(x[lead]) >> 63;
    sign_out = sign;
    U256 X = u256_zero();
    bool done = false;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint64_t b = f64_bits(x[p]);
        if (done || (b & 0x7FFFFFFFFFFFFFFFULL) == 0) continue;
        const bool negp = ((b >> 63) != sign);  // part sign relative to the element
        const UnpQ u = unpack_abs_q(b);
        const int sh = u.E + FIXB - e;
        if (sh >= 0) {
            U256 t = u256_shl(u.m, sh > 190 ? 190 : sh);
            X = u256_add(X, negp ? u256_neg(t) : t);
            continue;
        }
        // first part with a fraction: its floor, and the borrow
        const int rs = -sh;
        const uint64_t ip = rs >= 64 ? 0 : (u.m >> rs);
        const bool frac = rs >= 64 ? (u.m != 0) : ((u.m & ((1ULL << rs) - 1)) != 0);
        int64_t F;
        if (!negp) F = (int64_t)ip;
        else F = -(int64_t)(ip + (frac ? 1 : 0));
        if (!frac) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r <= p) continue;
                const uint64_t c = f64_bits(x[r]);
                if ((c & 0x7FFFFFFFFFFFFFFFULL) != 0) {
                    if ((c >> 63) != sign) F -= 1;
                    break;
                }
            }
        }
        U256 t = u256_shl((uint64_t)(F < 0 ? -F : F), 0);
        X = u256_add(X, F < 0 ? u256_neg(t) : t);
        done = true;
    }
    return X;
}

}  // namespace fxp
}  // namespace ddg
