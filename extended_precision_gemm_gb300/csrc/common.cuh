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

// The IEEE 754 bits of x, moved through an opaque instruction.  Masked tests
// and maxima of the bits then stay integer instructions: a compiler may
// otherwise fold a test of the magnitude bits back into a floating-point
// comparison or absolute value, which runs on the FP64 pipe (the narrowest
// unit of GB300).
__device__ __forceinline__ uint64_t f64_bits(double x) {
    uint64_t b;
    asm("mov.b64 %0, %1;" : "=l"(b) : "d"(x));
    return b;
}

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

// Bounds-checked build.  Compiled with -DDDGEMM_CHECKED (libddgemm_checked.so),
// every global access the kernels guard with in_bounds() is tested against
// the extent of its buffer first; a failing access is skipped, never trapped,
// and the first failure of the translation unit is recorded (check site,
// offending index) with a count of all failures.  dd_check_report reads and
// clears the records.  In the normal build in_bounds() is the constant true
// and the checks compile to nothing.
struct CheckRecord {
    unsigned int count;  // failures since the last read
    unsigned int site;   // check site of the first failure
    long long index;     // its index (element offset into the buffer)
};

#ifdef DDGEMM_CHECKED
static __device__ CheckRecord g_check_record;  // one per translation unit

__device__ __forceinline__ bool in_bounds(int64_t index, int64_t extent, unsigned int site) {
    if (index >= 0 && index < extent) return true;
    if (atomicAdd(&g_check_record.count, 1u) == 0) {
        g_check_record.site = site;
        g_check_record.index = (long long)index;
    }
    return false;
}

// Host function reading and clearing this translation unit's record.
#define DDG_DEFINE_CHECK_READER(name)                                                          \
    cudaError_t name(CheckRecord* out) {                                                       \
        cudaError_t err_ = cudaDeviceSynchronize();                                            \
        if (err_ == cudaSuccess) err_ = cudaMemcpyFromSymbol(out, g_check_record, sizeof(*out)); \
        const CheckRecord zero_ = {0u, 0u, 0};                                                 \
        if (err_ == cudaSuccess) err_ = cudaMemcpyToSymbol(g_check_record, &zero_, sizeof(zero_)); \
        return err_;                                                                           \
    }
#else
__device__ __forceinline__ constexpr bool in_bounds(int64_t, int64_t, unsigned int) { return true; }

#define DDG_DEFINE_CHECK_READER(name)         \
    cudaError_t name(CheckRecord* out) {      \
        *out = CheckRecord{0u, 0u, 0};        \
        return cudaSuccess;                   \
    }
#endif

// Check sites (the site number a failure records).
enum CheckSite : unsigned int {
    kSiteSplitLoadA = 101, kSiteSplitLoadB = 102, kSiteSplitStore = 103,
    kSiteGemmCopyA = 201, kSiteGemmCopyB = 202, kSiteGemmStoreP = 203, kSiteGemmStoreC = 204,
    kSiteRecombineLoadP = 301, kSiteRecombineStoreC = 302,
    kSiteFusedLoadA = 401, kSiteFusedLoadB = 402, kSiteFusedExp = 403,
    kSiteTcSplitLoadA = 501, kSiteTcSplitLoadB = 502, kSiteTcSplitStore = 503,
    kSiteTcRecombineLoadP = 601, kSiteTcRecombineStoreC = 602,
    kSiteTcGemmStoreP = 701,
    kSiteExpLoadA = 801, kSiteExpLoadB = 802,
};

// Programmatic dependent launch: a kernel launched with launch_pdl may be
// scheduled while the work before it on the stream drains.  pdl_wait()
// returns once the grids it depends on have completed and their writes are
// visible: every such kernel calls it before its first access to global
// memory (a no-op for an ordinary launch).  pdl_launch_dependents() lets the
// next grid on the stream be scheduled as this one's blocks retire.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace ddg
