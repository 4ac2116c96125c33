// dd_arith.cuh -- the recombination of the part sums into one double double
// ("Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2, steps 4-5),
// shared by the recombine kernel and by the slice GEMM that recombines in its
// epilogue, so that both give the same bits.
//
// Every addition is an explicit round-to-nearest FP64 operation (the
// error-free transformations must not be contracted or reassociated); the
// exact steps (k-split sums, power-of-two scalings, the sign of zero) use
// integer instructions, which give the same bits as the FP64 operations they
// replace on GB300's narrow FP64 pipe.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace ddg {

__device__ __forceinline__ void two_sum(double a, double b, double& s, double& e) {
    s = __dadd_rn(a, b);
    double bb = __dsub_rn(s, a);
    e = __dadd_rn(__dsub_rn(a, __dsub_rn(s, bb)), __dsub_rn(b, bb));
}

__device__ __forceinline__ void quick_two_sum(double a, double b, double& s, double& e) {
    s = __dadd_rn(a, b);
    e = __dsub_rn(b, __dsub_rn(s, a));
}

// Exact operations done with integer instructions (the FP64 pipe is the
// narrowest unit of GB300; these give the same bits as the FP64 operations
// they replace):

// An integer-valued double of magnitude below 2^53 as int64.
__device__ __forceinline__ long long to_int(double v) {
    const uint64_t b = f64_bits(v);
    const uint64_t a = b & 0x7FFFFFFFFFFFFFFFULL;
    if (a == 0) return 0;
    const int E = (int)(a >> 52) - 1075;
    const uint64_t m = (a & ((1ULL << 52) - 1)) | (1ULL << 52);
    const uint64_t mag = E >= 0 ? (m << E) : (m >> (-E));
    return (b >> 63) ? -(long long)mag : (long long)mag;
}

// An integer below 2^53 in magnitude as a double.
__device__ __forceinline__ double to_double(long long x) {
    if (x == 0) return 0.0;
    const uint64_t sign = x < 0 ? 1ULL : 0ULL;
    const uint64_t m = sign ? (uint64_t)(-x) : (uint64_t)x;
    const int p = 63 - __clzll((long long)m);
    const uint64_t mant = (m << (52 - p)) & ((1ULL << 52) - 1);
    return __longlong_as_double((long long)((sign << 63) | ((uint64_t)(1023 + p) << 52) | mant));
}

// x * 2^k for x = 0 or 1 <= |x| < 2^53 and -117 <= k <= 0: the result is a
// normal double (or 0), so only the exponent field changes.
__device__ __forceinline__ double scale_part(double x, int k) {
    const long long b = (long long)f64_bits(x);
    if ((b & 0x7FFFFFFFFFFFFFFFLL) == 0) return 0.0;
    return __longlong_as_double(b + ((long long)k << 52));
}

// ldexp(x, k), correctly rounded: an exponent-field add when x and the
// result are normal, the library ldexp otherwise (zero, subnormal, overflow).
__device__ __forceinline__ double scale_result(double x, int k) {
    const long long b = (long long)f64_bits(x);
    const int biased = (int)((b >> 52) & 0x7FF);
    if (biased != 0 && biased != 0x7FF && biased + k >= 1 && biased + k <= 2046)
        return __longlong_as_double(b + ((long long)k << 52));
    return ldexp(x, k);
}

// +0 for a zero of either sign.
__device__ __forceinline__ double plus_zero(double x) {
    return (f64_bits(x) << 1) == 0 ? 0.0 : x;
}

// (c_hi, c_lo) from the 8 part sums of one output: from d = 7 down to 0,
// (s, err) = two_sum(h, P_d 2^(-13 (d + 2))); err += l; (h, l) =
// quick_two_sum(s, err), starting from h = P_7 2^-117, l = 0; then both
// scaled by 2^sc (sc = e_i + f_j) and zeros made +0.
__device__ __forceinline__ void recombine_parts(const double (&part)[S], int sc, double& c_hi, double& c_lo) {
    // weight of part d: 2^(-13 (d + 2))
    double h = scale_part(part[S - 1], -DIGIT * (S + 1)), l = 0.0;
#pragma unroll
    for (int d = S - 2; d >= 0; --d) {
        double s, err;
        two_sum(h, scale_part(part[d], -DIGIT * (d + 2)), s, err);
        err = __dadd_rn(err, l);
        quick_two_sum(s, err, h, l);
    }
    c_hi = plus_zero(scale_result(h, sc));
    c_lo = plus_zero(scale_result(l, sc));
}

}  // namespace ddg
