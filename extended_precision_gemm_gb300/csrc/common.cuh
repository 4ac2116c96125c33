// common.cuh -- constants and device helpers shared by the dd GEMM kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ddgemm.h"

namespace ddg {

constexpr int S = DDGEMM_SLICES;           // 8 parts per double double
constexpr int DIGIT = DDGEMM_DIGIT_BITS;   // 13 bits per part
constexpr int FIX = S * DIGIT;             // 104 fraction bits kept
constexpr int TM = DDGEMM_TILE_M;          // 32
constexpr int TN = DDGEMM_TILE_N;          // 32
constexpr int BK = DDGEMM_CHUNK_K;         // 8
constexpr int CHUNK_DOUBLES = S * BK * TM; // one (tile, k-chunk) block of all 8 planes: 2048 doubles
constexpr int EXP_NONE = DDGEMM_EXP_NONE;  // "no nonzero element seen" exponent sentinel

static_assert(TM == TN, "tiles of A and B share one layout");
static_assert(BK % 4 == 0, "k-chunk holds whole k4 groups of the m8n8k4 fragments");

__host__ __device__ inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Smallest integer e with |x| < 2^e for the magnitude bits of a finite double
// (sign bit cleared); EXP_NONE for zero.  IEEE 754 binary64 layout.
__device__ __forceinline__ int exponent_from_abs_bits(uint64_t a) {
    if (a == 0) return EXP_NONE;
    int biased = (int)(a >> 52);
    if (biased != 0) return biased - 1022;           // 1.f * 2^(b-1023) < 2^(b-1022)
    int msb = 63 - __clzll((long long)a);            // subnormal: f * 2^-1074
    return msb - 1074 + 1;
}

// The exponent a row / column uses: EXP_NONE (all zero) reads as 0.
__device__ __forceinline__ int effective_exponent(int e) { return e == EXP_NONE ? 0 : e; }

// A double holding the small integer v (|v| < 2^13, sign given separately),
// built from the IEEE 754 bit layout with integer instructions only.
__device__ __forceinline__ double small_int_to_double(uint32_t v, uint64_t sign) {
    if (v == 0) return 0.0;
    int p = 31 - __clz((int)v);                      // leading bit position
    uint64_t mant = ((uint64_t)v << (52 - p)) & ((1ULL << 52) - 1);
    uint64_t bits = (sign << 63) | ((uint64_t)(1023 + p) << 52) | mant;
    return __longlong_as_double((long long)bits);
}

}  // namespace ddg
