// recombine.cu -- step 3 of the dd GEMM: the parts of the product summed into
// one double double and scaled back.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2, steps 4-5:
// extract the parts of the product and add them in double-double arithmetic
// (massively parallel, on the regular cores).  For output (i, j):
//     P_d   = sum over k-splits (exact: integers below 2^53)
//     (h,l) = P_7 2^-117, then for d = 6 .. 0:
//             (s, err) = two_sum(h, P_d 2^(-13(d+2)));  err += l;
//             (h, l)   = quick_two_sum(s, err)
//     C_hi  = ldexp(h, e_i + f_j),  C_lo = ldexp(l, e_i + f_j)   (+0 for zero)
// The weights 2^(-13(d+2)) are exact powers of two: part d of the product of
// two digit expansions x = sum_s D_s 2^(-13(s+1)) carries 2^(-13(d+2)).
// Every addition is an explicit round-to-nearest FP64 operation (the
// error-free transformations must not be contracted or reassociated); the
// exact steps (k-split sums, power-of-two scalings, the sign of zero) use
// integer instructions.
#include "common.cuh"
#include "dd_arith.cuh"
#include "launch.cuh"

namespace ddg {
namespace {

__global__ void __launch_bounds__(256) recombine_kernel(const double* __restrict__ P, int splits,
                                                        int64_t Mp, int64_t Np,
                                                        const int32_t* __restrict__ e,
                                                        const int32_t* __restrict__ f, int64_t M,
                                                        int64_t N, double* __restrict__ C_hi,
                                                        double* __restrict__ C_lo, int64_t ldc) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const int64_t plane = Mp * Np;
    const int fj = effective_exponent(f[j]);
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        const double* p = P + i * Np + j;
        if (!in_bounds((int64_t)(splits * S - 1) * plane + i * Np + j, (int64_t)splits * S * plane, kSiteRecombineLoadP) ||
            !in_bounds(i * ldc + j, (M - 1) * ldc + N, kSiteRecombineStoreC))
            continue;
        double part[S];
#pragma unroll
        for (int d = 0; d < S; ++d) part[d] = __ldg(p + d * plane);
        if (splits > 1) {  // exact integer sums of the k-split partials
#pragma unroll
            for (int d = 0; d < S; ++d) {
                long long v = to_int(part[d]);
                for (int z = 1; z < splits; ++z) v += to_int(__ldg(p + ((int64_t)z * S + d) * plane));
                part[d] = to_double(v);
            }
        }
        double c_hi, c_lo;
        recombine_parts(part, effective_exponent(e[i]) + fj, c_hi, c_lo);
        C_hi[i * ldc + j] = c_hi;
        C_lo[i * ldc + j] = c_lo;
    }
}

}  // namespace

DDG_DEFINE_CHECK_READER(check_record_recombine)

cudaError_t launch_recombine(const double* P, int splits, int64_t Mp, int64_t Np,
                             const int32_t* e, const int32_t* f, int64_t M, int64_t N,
                             double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    const unsigned gx = (unsigned)((N + 255) / 256);
    const unsigned gy = (unsigned)(M < 65535 ? M : 65535);
    return launch_pdl(recombine_kernel, dim3(gx, gy), dim3(256), 0, st, P, splits, Mp, Np, e, f, M, N, C_hi, C_lo,
                      ldc);
}

}  // namespace ddg
