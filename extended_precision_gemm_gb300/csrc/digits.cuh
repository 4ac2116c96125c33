// digits.cuh -- the 13-bit parts of a double double against a shared
// exponent, as used by the split kernels and by the slice GEMM that forms its
// parts from hi/lo tiles.
//
// X = floor(|hi + lo| * 2^(104 - e)) < 2^104 (fixed_point.cuh); the parts are
// its 13-bit fields, most significant first, with the sign of the element
// ("Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2: the
// quarters of a double, here on the grid the row / column shares).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "fixed_point.cuh"

namespace ddg {

// 13-bit field s of X, most significant first.
__device__ __forceinline__ uint32_t digit_field(unsigned __int128 X, int s) {
    return (uint32_t)(X >> (DIGIT * (S - 1 - s))) & ((1u << DIGIT) - 1);
}

// The 8 parts as doubles (exact small integers).
__device__ __forceinline__ void split_digits(double hi, double lo, int e, double out[S]) {
    uint64_t sign;
    const unsigned __int128 X = fxp::fixed_point(hi, lo, e, sign);
#pragma unroll
    for (int s = 0; s < S; ++s) out[s] = small_int_to_double(digit_field(X, s), sign);
}

}  // namespace ddg
