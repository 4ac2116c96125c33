// simt.cu -- the comparator: a double-double GEMM on the FP64 ALUs.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 4.2, second
// method: one thread computes one inner product of double doubles with
// double-double multiplications and additions on the regular cores (no
// splitting).  Per k, in order:
//     p = a_hi b_hi;  e = fma(a_hi, b_hi, -p)                (exact error)
//     e = e + (a_hi b_lo + a_lo b_hi)
//     (s, t) = two_sum(c_hi, p);  t = (t + c_lo) + e
//     (c_hi, c_lo) = quick_two_sum(s, t)
// 17 FP64 operations per k; on GB300 the FP64 pipe executes about 1.7 of them
// per clock per SM, so this kernel is bound by that pipe, like the mma.sync
// slice GEMM, but needs half as many FP64 operations per double-double flop.
// Every operation is an explicit round-to-nearest intrinsic (no contraction).
//
// Mapping: 16 x 16 threads per block, each thread a 2 x 2 block of outputs
// (rows ty + 16 i, columns tx + 16 j) of a 32 x 32 tile; A and B (hi, lo)
// pass through shared memory in k-slabs of 16.
#include "common.cuh"
#include "launch.cuh"

namespace ddg {
namespace {

constexpr int T = 32;   // output tile
constexpr int KS = 16;  // k-slab

__device__ __forceinline__ void dd_fma(double& c_hi, double& c_lo, double a_hi, double a_lo, double b_hi,
                                       double b_lo) {
    const double p = __dmul_rn(a_hi, b_hi);
    double e = __fma_rn(a_hi, b_hi, -p);
    e = __dadd_rn(e, __dadd_rn(__dmul_rn(a_hi, b_lo), __dmul_rn(a_lo, b_hi)));
    const double s = __dadd_rn(c_hi, p);
    const double bb = __dsub_rn(s, c_hi);
    double t = __dadd_rn(__dsub_rn(c_hi, __dsub_rn(s, bb)), __dsub_rn(p, bb));
    t = __dadd_rn(__dadd_rn(t, c_lo), e);
    c_hi = __dadd_rn(s, t);
    c_lo = __dsub_rn(t, __dsub_rn(c_hi, s));
}

__global__ void __launch_bounds__(256) simt_dd_gemm_kernel(const double* __restrict__ A_hi,
                                                           const double* __restrict__ A_lo, int64_t lda,
                                                           const double* __restrict__ B_hi,
                                                           const double* __restrict__ B_lo, int64_t ldb,
                                                           double* __restrict__ C_hi, double* __restrict__ C_lo,
                                                           int64_t ldc, int64_t M, int64_t N, int64_t K) {
    __shared__ double sa_hi[KS][T + 1], sa_lo[KS][T + 1], sb_hi[KS][T + 1], sb_lo[KS][T + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int64_t row0 = (int64_t)blockIdx.y * T, col0 = (int64_t)blockIdx.x * T;
    double c_hi[2][2] = {{0, 0}, {0, 0}}, c_lo[2][2] = {{0, 0}, {0, 0}};
    for (int64_t k0 = 0; k0 < K; k0 += KS) {
        // A slab: 32 rows x 16 k; B slab: 16 k x 32 columns (zeros outside)
        for (int idx = threadIdx.x; idx < T * KS; idx += 256) {
            const int r = idx / KS, kk = idx % KS;
            const int64_t gr = row0 + r, gk = k0 + kk;
            const bool in = gr < M && gk < K;
            sa_hi[kk][r] = in ? A_hi[gr * lda + gk] : 0.0;
            sa_lo[kk][r] = in ? A_lo[gr * lda + gk] : 0.0;
            const int kb = idx / T, c = idx % T;
            const int64_t gkb = k0 + kb, gc = col0 + c;
            const bool inb = gkb < K && gc < N;
            sb_hi[kb][c] = inb ? B_hi[gkb * ldb + gc] : 0.0;
            sb_lo[kb][c] = inb ? B_lo[gkb * ldb + gc] : 0.0;
        }
        __syncthreads();
        const int kn = (int)min((int64_t)KS, K - k0);
        for (int kk = 0; kk < kn; ++kk) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const double ah = sa_hi[kk][ty + 16 * i], al = sa_lo[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    dd_fma(c_hi[i][j], c_lo[i][j], ah, al, sb_hi[kk][tx + 16 * j], sb_lo[kk][tx + 16 * j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t r = row0 + ty + 16 * i, c = col0 + tx + 16 * j;
            if (r < M && c < N) {
                C_hi[r * ldc + c] = __dadd_rn(c_hi[i][j], 0.0);
                C_lo[r * ldc + c] = __dadd_rn(c_lo[i][j], 0.0);
            }
        }
}

}  // namespace

cudaError_t launch_simt_dd_gemm(const double* A_hi, const double* A_lo, int64_t lda, const double* B_hi,
                                const double* B_lo, int64_t ldb, double* C_hi, double* C_lo, int64_t ldc,
                                int64_t M, int64_t N, int64_t K, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    const int64_t gy = (M + T - 1) / T, gx = (N + T - 1) / T;
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    simt_dd_gemm_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, st>>>(A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi,
                                                                          C_lo, ldc, M, N, K);
    return cudaGetLastError();
}

}  // namespace ddg
