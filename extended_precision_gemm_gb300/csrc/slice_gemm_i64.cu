// slice_gemm_i64.cu -- step 2 of the dd GEMM on GB300's integer pipe.
//
// The same slice-pair products as slice_gemm.cu ("Multiple Double Arithmetic
// on NVIDIA Tensor Cores", eqs. (1)-(4), grouped by index sum,
//     P_d = sum_{s+t=d} A_s B_t,   d = 0..7,  36 pairs),
// from the same 13-bit parts, but each product is a 32-bit integer
// multiply-add into an int32 partial sum that is added into an exact int64
// total before it could overflow.  The sums are the same
// integers the FP64 kernel forms (|P_d| < 2^53), so P -- and the recombined C
// -- are identical bit for bit.  On GB300 the FP64 pipe (which also executes
// mma.sync f64) issues ~1.7 operations per clock per SM, the integer pipe 64:
// the exactness argument of eq. (5) needs only integers, not FP64.
//
// Mapping: one 128-thread block per 32 x 16 half tile of P and k-split;
// thread (tr, tc) = (tid / 8, tid % 8) owns rows {tr, tr+16} x columns
// {tc, tc+8} of the half for all 8 index sums.  The products go into int32
// partial sums (plain 32-bit multiply-adds, the cheapest integer operation)
// that are added into int64 totals every 4 or 8 k-steps, before they could
// overflow.  Parts arrive as int16 planes whose 8 parts per element are 16
// contiguous bytes; a 4-stage ring of bulk asynchronous copies (4 KB of A +
// 4 KB of B per k-chunk) with bounded mbarrier waits feeds shared memory;
// each k costs four 128-bit shared loads (broadcast inside the warp), 32
// unpacks and 144 multiply-adds per thread.
#include <atomic>
#include "async_copy.cuh"
#include "common.cuh"
#include "launch.cuh"

namespace ddg {
namespace {

constexpr int THREADS = 128;
constexpr int STAGES = 4;
constexpr int CHUNK_I16 = BK * TM * S;                            // 2048 int16 = 4 KB
constexpr uint32_t COPY_BYTES = CHUNK_I16 * sizeof(int16_t);
constexpr int STAGE_I16 = 2 * CHUNK_I16;
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_I16 * sizeof(int16_t) + 64;
constexpr unsigned long long WAIT_BUDGET_NS = 2000000000ULL;    // 2 s per wait
constexpr int64_t TILE_GROUP = 16;

static_assert(COPY_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");

__device__ unsigned int g_wait_timeouts_i64 = 0;

// Sign-extend the two int16 halves of a word.
__device__ __forceinline__ int lo16(uint32_t w) { return (int)(int16_t)(w & 0xFFFFu); }
__device__ __forceinline__ int hi16(uint32_t w) { return (int)w >> 16; }

__device__ __forceinline__ void unpack8(uint4 v, int (&d)[S]) {
    d[0] = lo16(v.x); d[1] = hi16(v.x); d[2] = lo16(v.y); d[3] = hi16(v.y);
    d[4] = lo16(v.z); d[5] = hi16(v.z); d[6] = lo16(v.w); d[7] = hi16(v.w);
}

// An integer of magnitude below 2^53 as a double, from the IEEE 754 layout
// with integer instructions only (exact).
__device__ __forceinline__ double exact_int_to_double(long long x) {
    if (x == 0) return 0.0;
    const uint64_t sign = x < 0 ? 1ULL : 0ULL;
    const uint64_t m = sign ? (uint64_t)(-x) : (uint64_t)x;
    const int p = 63 - __clzll((long long)m);
    const uint64_t mant = (m << (52 - p)) & ((1ULL << 52) - 1);
    return __longlong_as_double((long long)((sign << 63) | ((uint64_t)(1023 + p) << 52) | mant));
}

// Flushes: index sum d gets d+1 products of |D_s D_t| <= 8191^2 < 2^26 per
// k, so an int32 partial sum takes 32 / (d+1) k-steps exactly: 4 for
// d = 4..7, 8 for d = 0..3 (at most 32 * 8191^2 = 2146959392 < 2^31).
__device__ __forceinline__ void flush(uint32_t (&acc32)[S][2][2], long long (&acc64)[S][2][2], int d0, int d1) {
#pragma unroll
    for (int d = 0; d < S; ++d) {
        if (d < d0 || d >= d1) continue;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                acc64[d][i][j] += (long long)(int32_t)acc32[d][i][j];
                acc32[d][i][j] = 0u;
            }
    }
}

__global__ void __launch_bounds__(THREADS, 3)
    slice_gemm_i64_kernel(const int16_t* __restrict__ planesA, const int16_t* __restrict__ planesB,
                          int64_t KC, int splits, double* __restrict__ P, int64_t Mp, int64_t Np) {
    extern __shared__ __align__(128) int16_t smem16[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem16 + STAGES * STAGE_I16);

    const int tid = threadIdx.x, tr = tid >> 3, tc = tid & 7;
    // blocks cover half tiles: 32 rows x 16 columns (h = which half)
    const int64_t MT = Mp / TM, NT2 = (Np / TN) * 2;
    const int64_t t = blockIdx.x;
    const int64_t group = t / (TILE_GROUP * NT2);
    const int64_t first = group * TILE_GROUP;
    const int64_t rows = min((int64_t)TILE_GROUP, MT - first);
    const int64_t local = t - group * TILE_GROUP * NT2;
    const int64_t mt = first + local % rows, nt2 = local / rows;
    const int64_t nt = nt2 >> 1;
    const int h = (int)(nt2 & 1);
    const int z = blockIdx.y;
    const int64_t kc0 = (int64_t)z * KC / splits, kc1 = (int64_t)(z + 1) * KC / splits;
    const int nk = (int)(kc1 - kc0);
    const int16_t* srcA = planesA + (mt * KC + kc0) * CHUNK_I16;
    const int16_t* srcB = planesB + (nt * KC + kc0) * CHUNK_I16;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < STAGES && i < nk; ++i) {
            const uint32_t bar = smem_addr(&bars[i]);
            mbar_expect_tx(bar, 2u * COPY_BYTES);
            bulk_load(smem16 + i * STAGE_I16, srcA + (int64_t)i * CHUNK_I16, COPY_BYTES, bar);
            bulk_load(smem16 + i * STAGE_I16 + CHUNK_I16, srcB + (int64_t)i * CHUNK_I16, COPY_BYTES, bar);
        }

    uint32_t acc32[S][2][2];
    long long acc64[S][2][2];
#pragma unroll
    for (int d = 0; d < S; ++d)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) { acc32[d][i][j] = 0u; acc64[d][i][j] = 0; }

    const int col0 = h * 16 + tc;
    for (int it = 0; it < nk; ++it) {
        const int st = it % STAGES;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[st]), (uint32_t)(it / STAGES) & 1u, WAIT_BUDGET_NS);
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                atomicAdd(&g_wait_timeouts_i64, 1u);
                const int issued = min(nk, max(it - 1, 0) + STAGES);
                for (int j = it; j < issued; ++j)
                    mbar_wait_bounded(smem_addr(&bars[j % STAGES]), (uint32_t)(j / STAGES) & 1u, WAIT_BUDGET_NS);
            }
            return;
        }
        if (tid == 0 && it >= 1 && it - 1 + STAGES < nk) {
            const int nxt = it - 1 + STAGES, ns = (it - 1) % STAGES;
            const uint32_t bar = smem_addr(&bars[ns]);
            mbar_expect_tx(bar, 2u * COPY_BYTES);
            bulk_load(smem16 + ns * STAGE_I16, srcA + (int64_t)nxt * CHUNK_I16, COPY_BYTES, bar);
            bulk_load(smem16 + ns * STAGE_I16 + CHUNK_I16, srcB + (int64_t)nxt * CHUNK_I16, COPY_BYTES, bar);
        }
        const uint4* As = reinterpret_cast<const uint4*>(smem16 + st * STAGE_I16);
        const uint4* Bs = reinterpret_cast<const uint4*>(smem16 + st * STAGE_I16 + CHUNK_I16);
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            int a[2][S], b[2][S];
#pragma unroll
            for (int i = 0; i < 2; ++i) unpack8(As[k * TM + tr + 16 * i], a[i]);
#pragma unroll
            for (int j = 0; j < 2; ++j) unpack8(Bs[k * TN + col0 + 8 * j], b[j]);
#pragma unroll
            for (int s = 0; s < S; ++s)
#pragma unroll
                for (int u = 0; u + s < S; ++u)
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            acc32[s + u][i][j] += (uint32_t)a[i][s] * (uint32_t)b[j][u];
            if (k == BK / 2 - 1) flush(acc32, acc64, 4, S);  // after 4 k-steps
        }
        flush(acc32, acc64, 0, S);                          // after 8 k-steps
    }

    const int64_t plane = Mp * Np;
#pragma unroll
    for (int d = 0; d < S; ++d) {
        double* out = P + ((int64_t)z * S + d) * plane;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int64_t row = mt * TM + tr + 16 * i;
#pragma unroll
            for (int j = 0; j < 2; ++j) out[row * Np + nt * TN + col0 + 8 * j] = exact_int_to_double(acc64[d][i][j]);
        }
    }
}

}  // namespace

int slice_gemm_i64_ctas_per_sm() {
    static std::atomic<int> cached{0};  // per-SM count of this kernel (the same on every device)
    if (const int c = cached.load(std::memory_order_relaxed); c > 0) return c;
    int n = 0;
    if (cudaFuncSetAttribute(slice_gemm_i64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, slice_gemm_i64_kernel, THREADS, SMEM_BYTES) !=
            cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return 1;
    }
    cached.store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_slice_gemm_i64(const int16_t* planesA, const int16_t* planesB, int64_t Mp,
                                  int64_t Np, int64_t Kp, int splits, double* P, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(slice_gemm_i64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)((Mp / TM) * (Np / TN) * 2), (unsigned)splits);
    slice_gemm_i64_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(planesA, planesB, Kp / BK, splits, P, Mp, Np);
    return cudaGetLastError();
}

cudaError_t read_and_reset_wait_timeouts_i64(unsigned int* count) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(count, g_wait_timeouts_i64, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_timeouts_i64, &zero, sizeof(unsigned int));
}

}  // namespace ddg
