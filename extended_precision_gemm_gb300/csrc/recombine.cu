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
#include "launch.cuh"

namespace ddg {
namespace {

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
    const uint64_t b = (uint64_t)__double_as_longlong(v);
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
    const long long b = __double_as_longlong(x);
    if ((b & 0x7FFFFFFFFFFFFFFFLL) == 0) return 0.0;
    return __longlong_as_double(b + ((long long)k << 52));
}

// ldexp(x, k), correctly rounded: an exponent-field add when x and the
// result are normal, the library ldexp otherwise (zero, subnormal, overflow).
__device__ __forceinline__ double scale_result(double x, int k) {
    const long long b = __double_as_longlong(x);
    const int biased = (int)((b >> 52) & 0x7FF);
    if (biased != 0 && biased != 0x7FF && biased + k >= 1 && biased + k <= 2046)
        return __longlong_as_double(b + ((long long)k << 52));
    return ldexp(x, k);
}

// +0 for a zero of either sign.
__device__ __forceinline__ double plus_zero(double x) {
    return (__double_as_longlong(x) << 1) == 0 ? 0.0 : x;
}

__global__ void __launch_bounds__(256) recombine_kernel(const double* __restrict__ P, int splits,
                                                        int64_t Mp, int64_t Np,
                                                        const int32_t* __restrict__ e,
                                                        const int32_t* __restrict__ f, int64_t M,
                                                        int64_t N, double* __restrict__ C_hi,
                                                        double* __restrict__ C_lo, int64_t ldc) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const int64_t plane = Mp * Np;
    const int fj = effective_exponent(f[j]);
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        const double* p = P + i * Np + j;
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
        // weight of part d: 2^(-13 (d + 2))
        double h = scale_part(part[S - 1], -DIGIT * (S + 1)), l = 0.0;
#pragma unroll
        for (int d = S - 2; d >= 0; --d) {
            double s, err;
            two_sum(h, scale_part(part[d], -DIGIT * (d + 2)), s, err);
            err = __dadd_rn(err, l);
            quick_two_sum(s, err, h, l);
        }
        const int sc = effective_exponent(e[i]) + fj;
        C_hi[i * ldc + j] = plus_zero(scale_result(h, sc));
        C_lo[i * ldc + j] = plus_zero(scale_result(l, sc));
    }
}

}  // namespace

cudaError_t launch_recombine(const double* P, int splits, int64_t Mp, int64_t Np,
                             const int32_t* e, const int32_t* f, int64_t M, int64_t N,
                             double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    const unsigned gx = (unsigned)((N + 255) / 256);
    const unsigned gy = (unsigned)(M < 65535 ? M : 65535);
    recombine_kernel<<<dim3(gx, gy), 256, 0, st>>>(P, splits, Mp, Np, e, f, M, N, C_hi, C_lo, ldc);
    return cudaGetLastError();
}

}  // namespace ddg
