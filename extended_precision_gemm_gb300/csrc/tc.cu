// tc.cu -- the double-double GEMM with 8-bit parts on GB300's bf16 tensor
// cores (tcgen05 MMA, accumulators in tensor memory).
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 1, relates the
// rewriting to the Ozaki scheme, where accurate products are computed by
// lower precision arithmetic, and Section 2 eqs. (1)-(5) rest on one fact:
// parts on a shared grid have few nonzero bits, so their products and sums of
// products are exact in the accumulator.  "Ozaki 2.5: Engineering the
// Deconstruction Path of fp64-Emulated Dense Matrix Multiplication on FP8
// Tensor Cores" (summary) applies the same idea to 8-bit tensor pipes.  Here
// the parts are 8 bits wide, so that each is exact in bf16:
//
//  1. split: e' = e + 1 (e the shared exponent of the 13-bit method), X =
//     trunc((hi + lo) 2^(104 - e')) (|X| < 2^103), and the 13 balanced
//     base-256 digits of X, least significant first: D_s = ((X + 128) mod 256)
//     - 128, X <- (X - D_s) / 256, D_0 the rest; every |D_s| <= 128.  Parts
//     are stored as bf16 in blocks of 128 (A) or 256 (B) rows x 64 k, each
//     block in the 128-byte swizzled K-major layout the tensor core reads;
//  2. P_d = sum_{s+t=d} A_s B_t^T, d = 0..12 (91 pairs), on the tensor cores:
//     each product is at most 2^14, so 1024 of them sum to at most 2^24, and
//     every partial sum is an integer that f32 holds exactly; every 1024
//     products per output ("a chunk") the accumulator is read from tensor
//     memory and added into an exact int32
//     total (|P_d| <= 13 K 2^14 < 2^31 for K <= 8192 per k-split);
//  3. Z = sum_d P_d 2^(8 (12 - d)) exactly (256-bit), rounded once to the
//     nearest double double of Z 2^(e'_i + f'_j - 112).
#include <algorithm>

#include "tc_gemm.cuh"
#include "fixed_point.cuh"
#include "fixed_point_md.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"
#include "wide_int.cuh"
#include "exact_round.cuh"

namespace ddg {
namespace {

constexpr int TS = DDGEMM_TC_SLICES;        // 13 parts
constexpr int QS = DDGEMM_TC_QD_SLICES;     // 27 parts of a quad double
constexpr int QFIX = QS * TD;               // 216 fraction bits
static_assert(TS * TD == fxp::FIX_BITS, "13 parts of 8 bits cover the 104-bit fixed-point value");
static_assert((long long)TS * ksplit_max(TS) * 128 * 128 < (1LL << 31), "int32 totals per k-split");
static_assert((long long)QS * ksplit_max(QS) * 128 * 128 < (1LL << 31), "int32 totals per k-split");
static_assert(QS % 3 == 0, "quad-double parts come in groups of three");

// ---------------------------------------------------------------------------
// Step 1: bf16 parts.
// ---------------------------------------------------------------------------

// The 13 balanced base-256 digits of the element (hi, lo) against exponent
// e' (most significant first), each as the bit pattern of an f32 whose upper
// half is the digit's bf16 (every digit has at most 8 significant bits).
// With C = 128 (256^11 + ... + 256 + 1), the base-256 digits of X + C below
// 256^12 are D_s + 128 (s = 12 .. 1, least significant first), and
// (X + C) / 256^12 rounded down is D_0: the balanced digits are read off one
// addition.  A byte E placed under the exponent field of 2^23 (bits
// 0x4B0000EE) is the f32 2^23 + E, and subtracting 2^23 + 128 leaves E - 128
// exactly.
__device__ __forceinline__ void balanced_parts(double hi, double lo, int ep, uint32_t (&f32)[TS]) {
    uint64_t sign;
    const unsigned __int128 mag = fxp::fixed_point(hi, lo, ep, sign);
    const unsigned __int128 C = ((unsigned __int128)0x80808080u << 64) | 0x8080808080808080ULL;
    const unsigned __int128 Y = (sign ? (unsigned __int128)0 - mag : mag) + C;
    const uint32_t w[4] = {(uint32_t)Y, (uint32_t)(Y >> 32), (uint32_t)(Y >> 64), (uint32_t)(Y >> 96)};
#pragma unroll
    for (int s = 1; s < TS; ++s) {
        const int b = TS - 1 - s;  // byte of Y, least significant = 0
        const uint32_t bits = __byte_perm(w[b >> 2], 0x4B000000u, 0x7440u | (uint32_t)(b & 3));
        f32[s] = __float_as_uint(__fsub_rn(__uint_as_float(bits), 8388736.0f));
    }
    f32[0] = __float_as_uint(__int2float_rn((int)w[3]));
}

struct TcSplitGrid {
    const double* A_hi; const double* A_lo; int64_t lda, M; int32_t* e; int64_t a_tasks;
    const double* B_hi; const double* B_lo; int64_t ldb, N; int32_t* f; int64_t b_tasks;
    int64_t K, KB;  // KB = k-blocks of 64
    uint16_t* planesA; uint16_t* planesB;
    bool a_vec;     // A_hi, A_lo 16-byte aligned and lda even: 128-bit loads
    bool a_given, b_given;  // exponents supplied by the caller: never written
};

// One warp per task, 256 elements each: 4 rows of A, or 4 columns of B, x
// one k-block (lane = row or column (lane/8), 8 consecutive k (lane%8)).  An
// A lane reads 64 contiguous bytes of hi and of lo; for B each load
// instruction reads eight whole 32-byte sectors (4 columns of 8 rows of B).
// Each lane writes one 16-byte chunk of each part, so a warp writes whole
// 128-byte part rows: 512 contiguous bytes per part.  Rows / k beyond the
// matrix are written as 0.
__global__ void __launch_bounds__(256, 4) split_bf16_kernel(TcSplitGrid g) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * 8;
    const int64_t tasks = g.a_tasks + g.b_tasks;
    for (int64_t task = gw; task < tasks; task += nw) {
        if (task < g.a_tasks) {
            const int64_t rg = task / g.KB, kb = task % g.KB;
            const int64_t r = rg * 4 + (lane >> 3);
            const int kc = lane & 7;
            const int64_t k0 = kb * TBK + kc * 8;
            double hi[8], lo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) hi[j] = lo[j] = 0.0;
            int ep = 1;
            if (r < g.M && in_bounds(r * g.lda + min(k0 + 7, g.K - 1), (g.M - 1) * g.lda + g.K, kSiteTcSplitLoadA)) {
                const int32_t er = g.e[r];
                if (!g.a_given && kb == 0 && kc == 0 && er == EXP_NONE) g.e[r] = 0;
                ep = effective_exponent(er) + 1;
                const double* ph = g.A_hi + r * g.lda + k0;
                const double* pl = g.A_lo + r * g.lda + k0;
                if (g.a_vec && k0 + 8 <= g.K) {
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        const double2 h2 = __ldg(reinterpret_cast<const double2*>(ph + j));
                        const double2 l2 = __ldg(reinterpret_cast<const double2*>(pl + j));
                        hi[j] = h2.x; hi[j + 1] = h2.y; lo[j] = l2.x; lo[j + 1] = l2.y;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (k0 + j < g.K) { hi[j] = __ldg(ph + j); lo[j] = __ldg(pl + j); }
                }
            }
            uint32_t w[TS][4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t p0[TS], p1[TS];
                balanced_parts(hi[j], lo[j], ep, p0);
                balanced_parts(hi[j + 1], lo[j + 1], ep, p1);
#pragma unroll
                for (int s = 0; s < TS; ++s) w[s][j >> 1] = pack_bf16(p0[s], p1[s]);
            }
            const int64_t mt = r / TBM;
            const int rin = (int)(r % TBM);
            const int64_t a_extent = (int64_t)TS * round_up(g.M, PAIR_M) * g.KB * TBK;  // bf16 elements of planesA
            if (in_bounds(((mt * TS + TS - 1) * g.KB + kb) * (TBM * TBK) + (swizzled(rin, kc) + 15) / 2, a_extent,
                          kSiteTcSplitStore)) {
#pragma unroll
                for (int s = 0; s < TS; ++s) {
                    uint8_t* blk = reinterpret_cast<uint8_t*>(g.planesA + ((mt * TS + s) * g.KB + kb) * (TBM * TBK));
                    *reinterpret_cast<uint4*>(blk + swizzled(rin, kc)) = make_uint4(w[s][0], w[s][1], w[s][2], w[s][3]);
                }
            }
        } else {
            // B task: 4 columns x one k-block (lane = column (lane/8), 8
            // consecutive k (lane%8)), consecutive tasks on neighbouring columns
            const int64_t local = task - g.a_tasks;
            const int64_t groups = g.b_tasks / g.KB;
            const int64_t kb = local / groups, cg = local % groups;
            const int64_t n = cg * 4 + (lane >> 3);
            const int kc = lane & 7;
            int ep = 1;
            if (n < g.N) {
                const int32_t fr = g.f[n];
                if (!g.b_given && kb == 0 && kc == 0 && fr == EXP_NONE) g.f[n] = 0;
                ep = effective_exponent(fr) + 1;
            }
            const int64_t k0 = kb * TBK + kc * 8;
            double hi[8], lo[8];
            const bool n_ok = n < g.N && in_bounds(min(k0 + 7, g.K - 1) * g.ldb + n, (g.K - 1) * g.ldb + g.N,
                                                   kSiteTcSplitLoadB);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool in = n_ok && k0 + j < g.K;
                hi[j] = in ? __ldg(g.B_hi + (k0 + j) * g.ldb + n) : 0.0;
                lo[j] = in ? __ldg(g.B_lo + (k0 + j) * g.ldb + n) : 0.0;
            }
            uint32_t w[TS][4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t p0[TS], p1[TS];
                balanced_parts(hi[j], lo[j], ep, p0);
                balanced_parts(hi[j + 1], lo[j + 1], ep, p1);
#pragma unroll
                for (int s = 0; s < TS; ++s) w[s][j >> 1] = pack_bf16(p0[s], p1[s]);
            }
            const int64_t nt = n / TBN;
            const int nin = (int)(n % TBN);
            const int64_t b_extent = (int64_t)TS * round_up(g.N, TBN) * g.KB * TBK;  // bf16 elements of planesB
            if (in_bounds(((nt * TS + TS - 1) * g.KB + kb) * (TBN * TBK) + (swizzled(nin, kc) + 15) / 2, b_extent,
                          kSiteTcSplitStore)) {
#pragma unroll
                for (int s = 0; s < TS; ++s) {
                    uint8_t* blk = reinterpret_cast<uint8_t*>(g.planesB + ((nt * TS + s) * g.KB + kb) * (TBN * TBK));
                    *reinterpret_cast<uint4*>(blk + swizzled(nin, kc)) = make_uint4(w[s][0], w[s][1], w[s][2], w[s][3]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Step 3: exact sum of the parts and one rounding into a double double.
// ---------------------------------------------------------------------------

// Bits [75, 128) of a 128-bit magnitude normalised to bit 127, rounded to
// nearest (ties to even) into a double with leading-bit exponent E; the
// tail below the kept bits, or 2^75 minus it after rounding up, goes to rem.
__device__ __forceinline__ uint64_t round_top53(wide::u128 nrm, int E, uint64_t sign, wide::u128& rem, bool& up) {
    const uint64_t H = (uint64_t)(nrm >> 64), L = (uint64_t)nrm;
    const uint64_t keep = H >> 11;
    const bool rbit = (H >> 10) & 1;
    up = rbit && ((keep & 1) || (H & 0x3FF) != 0 || L != 0);
    const wide::u128 tail = nrm & ((((wide::u128)1) << 75) - 1);
    rem = up ? (((wide::u128)1) << 75) - tail : tail;
    // keep + up lies in [2^52, 2^53]: adding it to the biased exponent field
    // minus one carries into the exponent when it reaches 2^53
    return (sign << 63) | (((uint64_t)(E + 1022) << 52) + keep + (up ? 1 : 0));
}

__device__ __forceinline__ int msb128(wide::u128 m) {
    const uint64_t hi = (uint64_t)(m >> 64), lo = (uint64_t)m;
    return hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)lo);
}

// One k-split: |v_d| <= (d + 1) K 2^14 with 13 K 2^14 < 2^31, so the exact sum
// Z = sum_d v_d 256^(12 - d) is below 2^124 in magnitude (below 2^127 for any
// int32 v_d with |v_0| <= 2^30) and is formed in 128 bits from four groups (v_0; v_1..v_4; v_5..v_8; v_9..v_12: each group below
// 2^56).  Z 2^q rounded into (hi, lo) when both are normal doubles or zero
// (q >= -1022 and the leading bit of Z 2^q at most 2^1022); otherwise false.
__device__ __forceinline__ bool round_dd_one_split(const long long (&v)[TS], int q, double& hi, double& lo) {
    const long long g1 = ((v[1] * 256 + v[2]) * 256 + v[3]) * 256 + v[4];
    const long long g2 = ((v[5] * 256 + v[6]) * 256 + v[7]) * 256 + v[8];
    const long long g3 = ((v[9] * 256 + v[10]) * 256 + v[11]) * 256 + v[12];
    const wide::u128 Z = ((wide::u128)(__int128)v[0] << 96) + ((wide::u128)(__int128)g1 << 64) +
                         ((wide::u128)(__int128)g2 << 32) + (wide::u128)(__int128)g3;
    const uint64_t sign = (uint64_t)(Z >> 127);
    const wide::u128 M = sign ? (wide::u128)0 - Z : Z;
    if (M == 0) {
        hi = lo = 0.0;
        return true;
    }
    const int t = msb128(M);
    if (q < -1022 || t + q > 1022) return false;
    const int n = 127 - t;
    wide::u128 R;
    bool up;
    hi = __longlong_as_double((long long)round_top53(M << n, t + q, sign, R, up));
    if (R == 0) {
        lo = 0.0;
        return true;
    }
    // R is a multiple of 2^n below 2^75: its leading bit is at t1 >= n
    const int t1 = msb128(R);
    wide::u128 R2;
    bool up2;
    lo = __longlong_as_double((long long)round_top53(R << (127 - t1), t1 - n + q, sign ^ (up ? 1 : 0), R2, up2));
    return true;
}

// (hi, lo) of one output from its part sums (summed over the k-splits).
__device__ __forceinline__ void recombine_one(const long long (&v)[TS], bool one_split, int q, double& hi,
                                              double& lo) {
    // the 128-bit path: always taken for the sums of one k-split of the GEMM
    if (one_split && v[0] >= -(1LL << 30) && v[0] < (1LL << 30) && round_dd_one_split(v, q, hi, lo)) return;
    uint64_t z[3];
    xr::exact_sum<TS, 3>(v, z);
    double out[2];
    if (xr::fast_path_ok(z, q)) {
        xr::round_parts<3, 2>(z, q, out);
    } else {
        wide::U256 Z;
        Z.lo = ((wide::u128)z[1] << 64) | z[0];
        Z.hi = (wide::u128)(__int128)(int64_t)z[2];
        wide::round_into_doubles<2>(Z, q, out);
    }
    hi = out[0];
    lo = out[1];
}

// V consecutive outputs of a row per thread (V = 4: 16-byte loads of every
// part plane; vec_store: 16-byte stores of C when aligned).
template <int V>
__global__ void __launch_bounds__(256, 3) recombine_tc_kernel(const int32_t* __restrict__ P, int splits, int64_t Mp,
                                                           int64_t Np, const int32_t* __restrict__ e,
                                                           const int32_t* __restrict__ f, int64_t M, int64_t N,
                                                           double* __restrict__ C_hi, double* __restrict__ C_lo,
                                                           int64_t ldc, bool vec_store) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t j0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (j0 >= N) return;
    const int64_t plane = Mp * Np;
    int fj[V];
#pragma unroll
    for (int c = 0; c < V; ++c) fj[c] = j0 + c < N ? effective_exponent(f[j0 + c]) + 1 : 0;
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        const int32_t* p = P + i * Np + j0;
        if (!in_bounds((int64_t)(splits * TS - 1) * plane + i * Np + j0 + V - 1, (int64_t)splits * TS * plane,
                       kSiteTcRecombineLoadP) ||
            !in_bounds(i * ldc + min(j0 + V - 1, N - 1), (M - 1) * ldc + N, kSiteTcRecombineStoreC))
            continue;
        const int qi = effective_exponent(e[i]) + 1 - TD * (TS + 1);
        double h[V], l[V];
        if (splits == 1) {
            int32_t w[TS][V];
#pragma unroll
            for (int d = 0; d < TS; ++d) {
                if constexpr (V == 4) {
                    const int4 x = __ldg(reinterpret_cast<const int4*>(p + (int64_t)d * plane));
                    w[d][0] = x.x; w[d][1] = x.y; w[d][2] = x.z; w[d][3] = x.w;
                } else {
                    w[d][0] = __ldg(p + (int64_t)d * plane);
                }
            }
#pragma unroll
            for (int c = 0; c < V; ++c) {
                long long v[TS];
#pragma unroll
                for (int d = 0; d < TS; ++d) v[d] = w[d][c];
                recombine_one(v, true, qi + fj[c], h[c], l[c]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < V; ++c) {
                long long v[TS];
#pragma unroll
                for (int d = 0; d < TS; ++d) v[d] = 0;
                for (int zz = 0; zz < splits; ++zz) {
#pragma unroll
                    for (int d = 0; d < TS; ++d) v[d] += __ldg(p + c + ((int64_t)zz * TS + d) * plane);
                }
                recombine_one(v, false, qi + fj[c], h[c], l[c]);
            }
        }
        double* ch = C_hi + i * ldc + j0;
        double* cl = C_lo + i * ldc + j0;
        if (V == 4 && vec_store && j0 + 3 < N) {
            reinterpret_cast<double2*>(ch)[0] = make_double2(h[0], h[1]);
            reinterpret_cast<double2*>(ch)[1] = make_double2(h[2], h[3]);
            reinterpret_cast<double2*>(cl)[0] = make_double2(l[0], l[1]);
            reinterpret_cast<double2*>(cl)[1] = make_double2(l[2], l[3]);
        } else {
#pragma unroll
            for (int c = 0; c < V; ++c)
                if (j0 + c < N) {
                    ch[c] = h[c];
                    cl[c] = l[c];
                }
        }
    }
}

// ---------------------------------------------------------------------------
// Quad doubles: 27 parts of 8 bits.  X = trunc(x 2^(216 - e')) for x the sum
// of the four doubles (|X| < 2^215, in 256-bit arithmetic), and its 27
// balanced base-256 digits read off Y = X + 128 (256^25 + ... + 1) as for
// double doubles; the same block layout with 27 parts; the exact sum of the
// 27 part sums rounded once into four doubles.
// ---------------------------------------------------------------------------

struct TcQdSplitGrid {
    const double* A[4]; int64_t lda, M; int32_t* e; int64_t a_tasks;
    const double* B[4]; int64_t ldb, N; int32_t* f; int64_t b_tasks;
    int64_t K, KB;
    uint16_t* planesA; uint16_t* planesB;
};

// Y = X + C for the element (x0..x3) against e', as eight 32-bit words.
__device__ __forceinline__ void qd_biased(const double (&x)[4], int ep, uint32_t (&y)[8]) {
    uint64_t sign;
    wide::U256 X = fxp::fixed_point_qd<QFIX>(x, ep, sign);
    if (sign) X = wide::u256_neg(X);
    wide::U256 C;  // 128 in each of the 26 low bytes
    C.lo = ((wide::u128)0x8080808080808080ULL << 64) | 0x8080808080808080ULL;
    C.hi = ((wide::u128)0x8080ULL << 64) | 0x8080808080808080ULL;
    const wide::U256 Y = wide::u256_add(X, C);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        y[w] = (uint32_t)(Y.lo >> (32 * w));
        y[4 + w] = (uint32_t)(Y.hi >> (32 * w));
    }
}

// f32 bit pattern (upper half = bf16) of part s of a biased value.
__device__ __forceinline__ uint32_t qd_part(const uint32_t (&y)[8], int s) {
    if (s == 0) return __float_as_uint(__int2float_rn((int)(y[6] >> 16) | ((int)y[7] << 16)));  // Y >> 208, signed
    const int b = QS - 1 - s;
    const uint32_t bits = __byte_perm(y[b >> 2], 0x4B000000u, 0x7440u | (uint32_t)(b & 3));
    return __float_as_uint(__fsub_rn(__uint_as_float(bits), 8388736.0f));
}

// One warp per task of 256 elements, as for double doubles: 4 rows of A, or 4
// columns of B, x 64 k (lane = row or column (lane/8), 8 consecutive k
// (lane%8)).  Each lane forms Y for its 8 elements, then writes one 16-byte
// chunk of each of the 27 part rows (a warp writes whole 128-byte rows).
__global__ void __launch_bounds__(256, 3) split_bf16_qd_kernel(TcQdSplitGrid g) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * 8;
    const int64_t tasks = g.a_tasks + g.b_tasks;
    for (int64_t task = gw; task < tasks; task += nw) {
        const bool is_a = task < g.a_tasks;
        int64_t r, kb;
        int kc;
        if (is_a) {
            kb = task % g.KB;
            r = (task / g.KB) * 4 + (lane >> 3);
            kc = lane & 7;
        } else {
            // 4 columns x one k-block, consecutive tasks on neighbouring columns
            const int64_t local = task - g.a_tasks;
            const int64_t groups = g.b_tasks / g.KB;
            kb = local / groups;
            r = (local % groups) * 4 + (lane >> 3);
            kc = lane & 7;
        }
        const int64_t rows = is_a ? g.M : g.N;
        int ep = 1;
        if (r < rows) {
            int32_t* ex = is_a ? g.e : g.f;
            const int32_t er = ex[r];
            if (kb == 0 && kc == 0 && er == EXP_NONE) ex[r] = 0;
            ep = effective_exponent(er) + 1;
        }
        const int64_t k0 = kb * TBK + kc * 8;
        uint32_t y[8][8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            double x[4] = {0.0, 0.0, 0.0, 0.0};
            if (r < rows && k0 + j < g.K) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    x[q] = is_a ? __ldg(g.A[q] + r * g.lda + k0 + j) : __ldg(g.B[q] + (k0 + j) * g.ldb + r);
            }
            qd_biased(x, ep, y[j]);
        }
        uint16_t* planes = is_a ? g.planesA : g.planesB;
        const int brows = is_a ? TBM : TBN;
        const int64_t blk = r / brows;
        const int rin = (int)(r % brows);
#pragma unroll
        for (int s = 0; s < QS; ++s) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) w[j >> 1] = pack_bf16(qd_part(y[j], s), qd_part(y[j + 1], s));
            uint8_t* base = reinterpret_cast<uint8_t*>(planes + ((blk * QS + s) * g.KB + kb) * ((int64_t)brows * TBK));
            *reinterpret_cast<uint4*>(base + swizzled(rin, kc)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

__global__ void __launch_bounds__(256, 2) recombine_tc_qd_kernel(const int32_t* __restrict__ P, int splits, int64_t Mp,
                                                              int64_t Np, const int32_t* __restrict__ e,
                                                              const int32_t* __restrict__ f, int64_t M, int64_t N,
                                                              double* C0, double* C1, double* C2, double* C3,
                                                              int64_t ldc) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const int64_t plane = Mp * Np;
    const int fj = effective_exponent(f[j]) + 1;
    double* Cs[4] = {C0, C1, C2, C3};
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        // Z = sum_d v_d 256^(26 - d) as column sums of 32-bit words: each
        // k-split's part sums in groups of three at their offsets (all loads of
        // a split independent), then one carry pass (|Z| < 2^250)
        long long acc[10];
#pragma unroll
        for (int w = 0; w < 10; ++w) acc[w] = 0;
        for (int zz = 0; zz < splits; ++zz) {
            const int32_t* p = P + ((int64_t)zz * QS) * plane + i * Np + j;
#pragma unroll
            for (int g = 0; g < QS / 3; ++g) {
                const long long h = ((long long)__ldg(p + (int64_t)(3 * g) * plane) * 256 +
                                     __ldg(p + (int64_t)(3 * g + 1) * plane)) * 256 +
                                    __ldg(p + (int64_t)(3 * g + 2) * plane);
                xr::add_at(acc, h, TD * (QS - 3 - 3 * g));
            }
        }
        uint64_t z[4];
        xr::carry_to_limbs(acc, z);
        const int q = effective_exponent(e[i]) + 1 + fj - TD * (QS + 1);
        double out[4];
        if (!xr::round_parts_scan<4>(z, q, out, 4)) {
            wide::U256 Z;
            Z.lo = ((wide::u128)z[1] << 64) | z[0];
            Z.hi = ((wide::u128)z[3] << 64) | z[2];
            wide::round_into_doubles<4>(Z, q, out);
        }
#pragma unroll
        for (int pq = 0; pq < 4; ++pq) Cs[pq][i * ldc + j] = out[pq];
    }
}

}  // namespace

cudaError_t launch_split_bf16(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                              uint16_t* planesA, uint16_t* planesB, cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    TcSplitGrid g{};
    g.K = K;
    g.KB = Kp / TBK;
    if (A) {
        g.A_hi = A->hi; g.A_lo = A->lo; g.lda = A->ld; g.M = A->rows; g.e = A->exp; g.a_given = A->exp_given;
        g.a_tasks = (round_up(A->rows, PAIR_M) / 4) * g.KB;
        g.a_vec = (uintptr_t)A->hi % 16 == 0 && (uintptr_t)A->lo % 16 == 0 && A->ld % 2 == 0;
    }
    if (B) {
        g.B_hi = B->hi; g.B_lo = B->lo; g.ldb = B->ld; g.N = B->rows; g.f = B->exp; g.b_given = B->exp_given;
        g.b_tasks = (round_up(B->rows, TBN) / 4) * g.KB;
    }
    g.planesA = planesA;
    g.planesB = planesB;
    const int64_t tasks = g.a_tasks + g.b_tasks;
    if (tasks == 0) return cudaSuccess;
    // one task per warp, no grid-stride: blocks in flight write one compact range
    const unsigned blocks = (unsigned)std::min<int64_t>((tasks + 7) / 8, 0x7FFFFFFF);
    return launch_pdl(split_bf16_kernel, dim3(blocks), dim3(256), 0, st, g);
}

cudaError_t launch_slice_gemm_tc(const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                 int64_t Kp, int splits, int32_t* P, cudaStream_t st) {
    return launch_slice_gemm_parts<TS>(planesA, planesB, Mp, Np, Kp, splits, P, st);
}

cudaError_t launch_slice_gemm_tc_qd(const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                    int64_t Kp, int splits, int32_t* P, cudaStream_t st) {
    return launch_slice_gemm_parts<QS>(planesA, planesB, Mp, Np, Kp, splits, P, st);
}

cudaError_t launch_recombine_tc(const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                const int32_t* f, int64_t M, int64_t N, double* C_hi, double* C_lo, int64_t ldc,
                                cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    const unsigned gx = (unsigned)((N + 255) / 256);
    const unsigned gy = (unsigned)(M < 65535 ? M : 65535);
    const bool vec_store = (uintptr_t)C_hi % 16 == 0 && (uintptr_t)C_lo % 16 == 0 && ldc % 2 == 0;
    // one k-split with aligned part sums: 4 columns per thread (the rows of the
    // planes are multiples of 256 columns, so every 4-column group is aligned)
    if (splits == 1 && (uintptr_t)P % 16 == 0) {
        const unsigned gx4 = (unsigned)((N + 1023) / 1024);
        return launch_pdl(recombine_tc_kernel<4>, dim3(gx4, gy), dim3(256), 0, st, P, splits, Mp, Np, e, f, M, N,
                          C_hi, C_lo, ldc, vec_store);
    }
    return launch_pdl(recombine_tc_kernel<1>, dim3(gx, gy), dim3(256), 0, st, P, splits, Mp, Np, e, f, M, N, C_hi,
                      C_lo, ldc, false);
}

cudaError_t launch_split_bf16_qd(const double* const* A, int64_t lda, int64_t M, int32_t* e, const double* const* B,
                                 int64_t ldb, int64_t N, int32_t* f, int64_t K, int64_t Kp, uint16_t* planesA,
                                 uint16_t* planesB, cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    TcQdSplitGrid g{};
    g.K = K;
    g.KB = Kp / TBK;
    if (A && M > 0) {
        for (int q = 0; q < 4; ++q) g.A[q] = A[q];
        g.lda = lda; g.M = M; g.e = e;
        g.a_tasks = (round_up(M, PAIR_M) / 4) * g.KB;
    }
    if (B && N > 0) {
        for (int q = 0; q < 4; ++q) g.B[q] = B[q];
        g.ldb = ldb; g.N = N; g.f = f;
        g.b_tasks = (round_up(N, TBN) / 4) * g.KB;
    }
    g.planesA = planesA;
    g.planesB = planesB;
    const int64_t tasks = g.a_tasks + g.b_tasks;
    if (tasks == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((tasks + 7) / 8, 0x7FFFFFFF);  // one task per warp
    split_bf16_qd_kernel<<<blocks, 256, 0, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_recombine_tc_qd(const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                   const int32_t* f, int64_t M, int64_t N, double* const* C, int64_t ldc,
                                   cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    const unsigned gx = (unsigned)((N + 255) / 256);
    const unsigned gy = (unsigned)(M < 65535 ? M : 65535);
    recombine_tc_qd_kernel<<<dim3(gx, gy), 256, 0, st>>>(P, splits, Mp, Np, e, f, M, N, C[0], C[1], C[2], C[3], ldc);
    return cudaGetLastError();
}

cudaError_t read_and_reset_wait_timeouts_tc(unsigned int* count) { return reset_tc_timeouts(count); }

DDG_DEFINE_CHECK_READER(check_record_tc)

cudaError_t peek_wait_timeouts_tc(unsigned int* count, cudaStream_t st) { return peek_tc_timeouts(count, st); }

int tc_resident_pairs() { return resident_pairs<TS>(); }

}  // namespace ddg
