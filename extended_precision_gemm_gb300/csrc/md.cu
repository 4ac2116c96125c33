// md.cu -- the method for quad doubles (4 doubles per number, 16 parts of 13
// bits, 136 index-sum pairs) on GB300's integer pipe.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores": the rewriting of
// Section 2 works for general multiple doubles (a quartered quad double has
// 16 times the size of a double; Table 1 reports quad-double runs, Table 2
// the dimensions for qd).  Steps, as for double doubles:
//  1. shared exponents e_i, f_j from the leading parts; the 16 truncating
//     base-2^13 digits of |x| 2^-e of x = x0 + x1 + x2 + x3, formed exactly in
//     256-bit integer arithmetic, stored as int16 ([tile][k-chunk][k][row]
//     [part], 32 contiguous bytes per element);
//  2. P_d = sum_{s+t=d} A_s B_t, d = 0..15, as 32-bit integer multiply-adds
//     into int32 partial sums flushed into exact int64 totals (every 2, 4 or
//     8 k-steps, before (d+1) k 8191^2 could reach 2^31); every P_d < 2^53
//     for K <= 2^23;
//  3. the parts summed exactly (a 256-bit integer) and rounded once into four
//     non-overlapping doubles, x_0 = RN(X), x_1 = RN(X - x_0), ... (the page
//     fixes double-double summation only for double doubles; the exact sum
//     rounded once is the plain reading for more parts).
#include <atomic>
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "wide_int.cuh"
#include "fixed_point_md.cuh"
#include "launch.cuh"

namespace ddg {
namespace {

constexpr int SQ = 16;                      // parts per quad double
constexpr int NPQ = 4;                      // doubles per quad double
constexpr int FIXQ = SQ * DIGIT;            // 208 fraction bits
constexpr uint64_t ABS_MASK = 0x7FFFFFFFFFFFFFFFULL;
using namespace wide;

// ---------------------------------------------------------------------------
// Step 1: exponents come from the double-double exponent kernel on the
// leading parts; this kernel writes the 16 int16 parts.
// ---------------------------------------------------------------------------

struct QdOperand {
    const double* p[NPQ];
    int64_t ld, rows;
    const int32_t* exp;
};

__device__ __forceinline__ int64_t qd_offset(int64_t tile, int64_t KC, int64_t k, int ti) {
    return (((tile * KC + k / BK) * BK + k % BK) * TM + ti) * SQ;
}

// Items: one 32-row tile of A (32-column tile of B) x 32 k; lane = row
// (column), warp = 4 consecutive k.  Items [0, a_items) are A's.
__global__ void __launch_bounds__(256) split_qd_kernel(QdOperand A, QdOperand B, int64_t K, int64_t Kp,
                                                       int64_t KT, int64_t a_items, int64_t items,
                                                       int16_t* __restrict__ planesA, int16_t* __restrict__ planesB) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t KC = Kp / BK;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const bool is_a = item < a_items;
        const int64_t local = is_a ? item : item - a_items;
        const int64_t tile = local / KT, kt = local % KT;
        const int64_t k0 = kt * 32 + 4 * w;
        if (k0 >= Kp) continue;
        const QdOperand& op = is_a ? A : B;
        const int64_t r = tile * TM + lane;
        const int ex = r < op.rows ? effective_exponent(op.exp[r]) : 0;
        int16_t* planes = is_a ? planesA : planesB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int64_t k = k0 + kk;
            double x[NPQ] = {0, 0, 0, 0};
            if (r < op.rows && k < K) {
                const int64_t off = is_a ? r * op.ld + k : k * op.ld + r;
#pragma unroll
                for (int p = 0; p < NPQ; ++p) x[p] = __ldg(op.p[p] + off);
            }
            uint64_t sign;
            const U256 X = fxp::fixed_point_qd<FIXQ>(x, ex, sign);
            uint32_t wd[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t d0 = u256_bits(X, DIGIT * (SQ - 1 - 2 * j), DIGIT);
                uint32_t d1 = u256_bits(X, DIGIT * (SQ - 2 - 2 * j), DIGIT);
                if (sign) { d0 = (uint32_t)(-(int32_t)d0); d1 = (uint32_t)(-(int32_t)d1); }
                wd[j] = (d0 & 0xFFFFu) | (d1 << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(planes + qd_offset(tile, KC, k, lane));
            dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
        }
    }
}

// ---------------------------------------------------------------------------
// Step 2: P_d for d = 0..15 on the integer pipe.  A 128-thread block takes
// 32 rows x 8 columns of a 32 x 32 tile; thread (tr, tc) = (tid / 4, tid % 4)
// owns row tr and columns {tc, tc + 4} of its quarter.
// ---------------------------------------------------------------------------

constexpr int QTHREADS = 128;
constexpr int QSTAGES = 4;
constexpr int QCHUNK = BK * TM * SQ;                         // 4096 int16 = 8 KB
constexpr uint32_t QCOPY = QCHUNK * sizeof(int16_t);
constexpr int QSTAGE = 2 * QCHUNK;
constexpr size_t QSMEM = (size_t)QSTAGES * QSTAGE * sizeof(int16_t) + 64;
constexpr unsigned long long QWAIT_NS = 2000000000ULL;
constexpr int64_t QGROUP = 16;

__device__ unsigned int g_wait_timeouts_qd = 0;

__device__ __forceinline__ int lo16(uint32_t w) { return (int)(int16_t)(w & 0xFFFFu); }
__device__ __forceinline__ int hi16(uint32_t w) { return (int)w >> 16; }

__device__ __forceinline__ void unpack16(const uint4* src, int (&d)[SQ]) {
    const uint4 v0 = src[0], v1 = src[1];
    d[0] = lo16(v0.x); d[1] = hi16(v0.x); d[2] = lo16(v0.y); d[3] = hi16(v0.y);
    d[4] = lo16(v0.z); d[5] = hi16(v0.z); d[6] = lo16(v0.w); d[7] = hi16(v0.w);
    d[8] = lo16(v1.x); d[9] = hi16(v1.x); d[10] = lo16(v1.y); d[11] = hi16(v1.y);
    d[12] = lo16(v1.z); d[13] = hi16(v1.z); d[14] = lo16(v1.w); d[15] = hi16(v1.w);
}

// Index sum d collects d+1 products below 8191^2 < 2^26 per k: an int32
// partial sum takes floor(32 / (d+1)) k-steps, so d >= 8 are flushed every 2
// k, d = 4..7 every 4, d <= 3 every 8 (the k-chunk).
__device__ __forceinline__ void qflush(uint32_t (&a32)[SQ][2], long long (&a64)[SQ][2], int d0, int d1) {
#pragma unroll
    for (int d = 0; d < SQ; ++d) {
        if (d < d0 || d >= d1) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            a64[d][j] += (long long)(int32_t)a32[d][j];
            a32[d][j] = 0u;
        }
    }
}

__device__ __forceinline__ double exact_int_to_double(long long x) {
    if (x == 0) return 0.0;
    const uint64_t sign = x < 0 ? 1ULL : 0ULL;
    const uint64_t m = sign ? (uint64_t)(-x) : (uint64_t)x;
    const int p = 63 - __clzll((long long)m);
    const uint64_t mant = (m << (52 - p)) & ((1ULL << 52) - 1);
    return __longlong_as_double((long long)((sign << 63) | ((uint64_t)(1023 + p) << 52) | mant));
}

__global__ void __launch_bounds__(QTHREADS, 3)
    slice_gemm_qd_kernel(const int16_t* __restrict__ planesA, const int16_t* __restrict__ planesB, int64_t KC,
                         int splits, double* __restrict__ P, int64_t Mp, int64_t Np) {
    extern __shared__ __align__(128) int16_t sq[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(sq + QSTAGES * QSTAGE);
    const int tid = threadIdx.x, tr = tid >> 2, tc = tid & 3;
    const int64_t MT = Mp / TM, NT4 = (Np / TN) * 4;
    const int64_t t = blockIdx.x;
    const int64_t group = t / (QGROUP * NT4);
    const int64_t first = group * QGROUP;
    const int64_t rows = min((int64_t)QGROUP, MT - first);
    const int64_t local = t - group * QGROUP * NT4;
    const int64_t mt = first + local % rows, nt4 = local / rows;
    const int64_t nt = nt4 >> 2;
    const int quarter = (int)(nt4 & 3);
    const int z = blockIdx.y;
    const int64_t kc0 = (int64_t)z * KC / splits, kc1 = (int64_t)(z + 1) * KC / splits;
    const int nk = (int)(kc1 - kc0);
    const int16_t* srcA = planesA + (mt * KC + kc0) * QCHUNK;
    const int16_t* srcB = planesB + (nt * KC + kc0) * QCHUNK;

    if (tid == 0) {
        for (int i = 0; i < QSTAGES; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < QSTAGES && i < nk; ++i) {
            const uint32_t bar = smem_addr(&bars[i]);
            mbar_expect_tx(bar, 2u * QCOPY);
            bulk_load(sq + i * QSTAGE, srcA + (int64_t)i * QCHUNK, QCOPY, bar);
            bulk_load(sq + i * QSTAGE + QCHUNK, srcB + (int64_t)i * QCHUNK, QCOPY, bar);
        }

    uint32_t a32[SQ][2];
    long long a64[SQ][2];
#pragma unroll
    for (int d = 0; d < SQ; ++d)
#pragma unroll
        for (int j = 0; j < 2; ++j) { a32[d][j] = 0u; a64[d][j] = 0; }

    const int col0 = quarter * 8 + tc;
    for (int it = 0; it < nk; ++it) {
        const int st = it % QSTAGES;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[st]), (uint32_t)(it / QSTAGES) & 1u, QWAIT_NS);
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                atomicAdd(&g_wait_timeouts_qd, 1u);
                const int issued = min(nk, max(it - 1, 0) + QSTAGES);
                for (int j = it; j < issued; ++j)
                    mbar_wait_bounded(smem_addr(&bars[j % QSTAGES]), (uint32_t)(j / QSTAGES) & 1u, QWAIT_NS);
            }
            return;
        }
        if (tid == 0 && it >= 1 && it - 1 + QSTAGES < nk) {
            const int nxt = it - 1 + QSTAGES, ns = (it - 1) % QSTAGES;
            const uint32_t bar = smem_addr(&bars[ns]);
            mbar_expect_tx(bar, 2u * QCOPY);
            bulk_load(sq + ns * QSTAGE, srcA + (int64_t)nxt * QCHUNK, QCOPY, bar);
            bulk_load(sq + ns * QSTAGE + QCHUNK, srcB + (int64_t)nxt * QCHUNK, QCOPY, bar);
        }
        const uint4* As = reinterpret_cast<const uint4*>(sq + st * QSTAGE);
        const uint4* Bs = reinterpret_cast<const uint4*>(sq + st * QSTAGE + QCHUNK);
#pragma unroll 1
        for (int k = 0; k < BK; ++k) {
            int a[SQ], b[2][SQ];
            unpack16(As + (k * TM + tr) * 2, a);
#pragma unroll
            for (int j = 0; j < 2; ++j) unpack16(Bs + (k * TN + col0 + 4 * j) * 2, b[j]);
#pragma unroll
            for (int s = 0; s < SQ; ++s)
#pragma unroll
                for (int u = 0; u + s < SQ; ++u)
#pragma unroll
                    for (int j = 0; j < 2; ++j) a32[s + u][j] += (uint32_t)a[s] * (uint32_t)b[j][u];
            if ((k & 1) == 1) qflush(a32, a64, 8, SQ);
            if ((k & 3) == 3) qflush(a32, a64, 4, 8);
        }
        qflush(a32, a64, 0, 4);
    }

    const int64_t plane = Mp * Np;
    const int64_t row = mt * TM + tr;
#pragma unroll
    for (int d = 0; d < SQ; ++d) {
        double* out = P + ((int64_t)z * SQ + d) * plane;
#pragma unroll
        for (int j = 0; j < 2; ++j) out[row * Np + nt * TN + col0 + 4 * j] = exact_int_to_double(a64[d][j]);
    }
}

// ---------------------------------------------------------------------------
// Step 3: X = sum_d P_d 2^(13 (15 - d)) exactly (256 bits), value X 2^q with
// q = e_i + f_j - 13 * 17, rounded once into 4 doubles.
// ---------------------------------------------------------------------------

// An integer-valued double of magnitude below 2^63 as int64 (exact).
__device__ __forceinline__ long long exact_double_to_int(double v) {
    const uint64_t b = f64_bits(v);
    const uint64_t a = b & ABS_MASK;
    if (a == 0) return 0;
    const int E = (int)(a >> 52) - 1075;  // v = m 2^E, E >= -52 for integers >= 1
    const uint64_t m = (a & ((1ULL << 52) - 1)) | (1ULL << 52);
    const uint64_t mag = E >= 0 ? (m << E) : (m >> (-E));
    return (b >> 63) ? -(long long)mag : (long long)mag;
}

__global__ void __launch_bounds__(256) recombine_qd_kernel(const double* __restrict__ P, int splits, int64_t Mp,
                                                           int64_t Np, const int32_t* __restrict__ e,
                                                           const int32_t* __restrict__ f, int64_t M, int64_t N,
                                                           double* C0, double* C1, double* C2, double* C3,
                                                           int64_t ldc) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const int64_t plane = Mp * Np;
    const int fj = effective_exponent(f[j]);
    double* Cs[NPQ] = {C0, C1, C2, C3};
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        U256 X = u256_zero();
#pragma unroll
        for (int d = 0; d < SQ; ++d) {
            long long v = 0;
            for (int z = 0; z < splits; ++z) v += exact_double_to_int(__ldg(P + ((int64_t)z * SQ + d) * plane + i * Np + j));
            const uint64_t mag = (uint64_t)(v < 0 ? -v : v);
            const U256 t = u256_shl(mag, DIGIT * (SQ - 1 - d));
            X = u256_add(X, v < 0 ? u256_neg(t) : t);
        }
        const int q = effective_exponent(e[i]) + fj - DIGIT * (SQ + 1);
        double out[NPQ];
        round_into_doubles<NPQ>(X, q, out);
#pragma unroll
        for (int p = 0; p < NPQ; ++p) Cs[p][i * ldc + j] = out[p];
    }
}

}  // namespace

cudaError_t launch_split_qd(const double* const* A, int64_t lda, int64_t M, const int32_t* e,
                            const double* const* B, int64_t ldb, int64_t N, const int32_t* f, int64_t K,
                            int64_t Kp, int16_t* planesA, int16_t* planesB, cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    QdOperand a{}, b{};
    for (int p = 0; p < NPQ; ++p) { a.p[p] = A ? A[p] : nullptr; b.p[p] = B ? B[p] : nullptr; }
    a.ld = lda; a.rows = A ? M : 0; a.exp = e;
    b.ld = ldb; b.rows = B ? N : 0; b.exp = f;
    const int64_t KT = (Kp + 31) / 32;
    const int64_t a_items = ((a.rows + TM - 1) / TM) * KT;
    const int64_t items = a_items + ((b.rows + TN - 1) / TN) * KT;
    if (items == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>(items, 0x7FFFFFFF);  // one item per block
    split_qd_kernel<<<blocks, 256, 0, st>>>(a, b, K, Kp, KT, a_items, items, planesA, planesB);
    return cudaGetLastError();
}

int slice_gemm_qd_ctas_per_sm() {
    static std::atomic<int> cached{0};  // per-SM count of this kernel (the same on every device)
    if (const int c = cached.load(std::memory_order_relaxed); c > 0) return c;
    int n = 0;
    if (cudaFuncSetAttribute(slice_gemm_qd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QSMEM) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, slice_gemm_qd_kernel, QTHREADS, QSMEM) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return 1;
    }
    cached.store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_slice_gemm_qd(const int16_t* planesA, const int16_t* planesB, int64_t Mp, int64_t Np,
                                 int64_t Kp, int splits, double* P, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(slice_gemm_qd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QSMEM);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)((Mp / TM) * (Np / TN) * 4), (unsigned)splits);
    slice_gemm_qd_kernel<<<grid, QTHREADS, QSMEM, st>>>(planesA, planesB, Kp / BK, splits, P, Mp, Np);
    return cudaGetLastError();
}

cudaError_t launch_recombine_qd(const double* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                const int32_t* f, int64_t M, int64_t N, double* const* C, int64_t ldc,
                                cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    const unsigned gx = (unsigned)((N + 255) / 256);
    const unsigned gy = (unsigned)(M < 65535 ? M : 65535);
    recombine_qd_kernel<<<dim3(gx, gy), 256, 0, st>>>(P, splits, Mp, Np, e, f, M, N, C[0], C[1], C[2], C[3], ldc);
    return cudaGetLastError();
}

cudaError_t read_and_reset_wait_timeouts_qd(unsigned int* count) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(count, g_wait_timeouts_qd, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_timeouts_qd, &zero, sizeof(unsigned int));
}

}  // namespace ddg
