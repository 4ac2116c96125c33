// tc_md.cu -- octo and hexa doubles (8 and 16 doubles per number) with 8-bit
// parts on the bf16 tensor cores.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2: the
// rewriting works for general multiple doubles; Table 2 gives the dimensions
// of quartered quad, octo and hexa doubles.  The scheme of the double-double
// and quad-double bf16 variants, for NIN doubles per number:
//  1. e' = e + 1 (e from the leading doubles), X = trunc(x 2^(8 NP - e')) for
//     x the sum of the NIN doubles (|X| < 2^(8 NP - 1), in WX 64-bit limbs),
//     and its NP balanced base-256 digits read off Y = X + 128 (256^(NP-2) +
//     ... + 1): the low bytes of Y are the digits + 128, its top the first
//     digit.  NP = 54 for octo doubles (432 bits), 107 for hexa doubles (856);
//  2. P_d = sum_{s+t=d} A_s B_t^T on the tensor cores (the pair kernel of
//     tc_gemm.cuh with NP parts; a k-split covers at most 2048 / 1024 of k);
//  3. Z = sum_d P_d 256^(NP-1-d) exactly (WZ limbs), rounded once into NIN
//     doubles x_0 = RN(Z 2^q), x_1 = RN(Z 2^q - x_0), ...
#include "tc_gemm.cuh"
#include "exact_round.cuh"

namespace ddg {
namespace {

template <int NIN>
struct MdShape;
template <>
struct MdShape<8> {
    static constexpr int NP = DDGEMM_TC_OD_SLICES;  // 54 parts
    static constexpr int WX = 7;                    // limbs of X and Y (|X| < 2^431)
    static constexpr int WZ = 8;                    // limbs of Z (|Z| < 2^467)
    static constexpr int SPLIT_MINB = 1;            // blocks per SM the split kernels are built for
};
template <>
struct MdShape<16> {
    static constexpr int NP = DDGEMM_TC_HD_SLICES;  // 107 parts
    static constexpr int WX = 14;                   // |X| < 2^855
    static constexpr int WZ = 14;                   // |Z| < 2^891
    static constexpr int SPLIT_MINB = 2;            // 128 registers: two blocks per SM beat one of 169
};

constexpr uint64_t ABS = 0x7FFFFFFFFFFFFFFFULL;

struct UnpM {
    uint64_t m;  // integer significand
    int E;       // |x| = m 2^E
};

__device__ __forceinline__ UnpM unpack_m(uint64_t bits) {
    const uint64_t a = bits & ABS;
    const int biased = (int)(a >> 52);
    UnpM u;
    if (biased == 0) { u.m = a & ((1ULL << 52) - 1); u.E = -1074; }
    else { u.m = (a & ((1ULL << 52) - 1)) | (1ULL << 52); u.E = biased - 1075; }
    return u;
}

// X = floor(|x_0 + ... + x_(NIN-1)| 2^(FIXB - e)) for a normalised multiple
// double (|x_(p+1)| <= ulp(x_p) / 2) and the sign of the element.  With every
// double signed relative to the leading one, the doubles that are integers at
// this scale add exactly; at the first double with a fraction, floor(a + rest)
// = floor(a) when a has a nonzero fraction (the rest is below half its last
// bit), else floor(a) - 1 when the first nonzero later double is negative
// (the borrow of Problem 3.3, eq. (7)).
template <int NIN, int W>
__device__ __forceinline__ void fixed_point_n(const double (&x)[NIN], int e, int FIXB, uint64_t (&X)[W],
                                              uint64_t& sign_out) {
    // the integer parts of the doubles are added as 64-bit column sums of
    // 32-bit words (dynamic positions, so the sums live in local memory), and
    // one carry pass gives the limbs: the value is nonnegative
    long long acc[2 * W + 2];
#pragma unroll
    for (int w = 0; w < 2 * W + 2; ++w) acc[w] = 0;
#pragma unroll
    for (int j = 0; j < W; ++j) X[j] = 0;
    int lead = -1;
#pragma unroll
    for (int p = NIN - 1; p >= 0; --p)
        if ((f64_bits(x[p]) & ABS) != 0) lead = p;
    sign_out = 0;
    if (lead < 0) return;
    uint64_t sign = 0;
#pragma unroll
    for (int p = 0; p < NIN; ++p)
        if (p == lead) sign = f64_bits(x[p]) >> 63;
    sign_out = sign;
    bool done = false;
#pragma unroll
    for (int p = 0; p < NIN; ++p) {
        const uint64_t b = f64_bits(x[p]);
        if (done || (b & ABS) == 0) continue;
        const bool negp = (b >> 63) != sign;
        const UnpM u = unpack_m(b);
        const int sh = u.E + FIXB - e;
        if (sh >= 0) {
            const int s = min(sh, 64 * W - 53);  // clamped only out of contract
            const int w = s >> 5;
            const unsigned __int128 G = (unsigned __int128)u.m << (s & 31);  // < 2^85
            const long long p0 = (long long)(uint32_t)G, p1 = (long long)(uint32_t)(G >> 32),
                            p2 = (long long)(uint32_t)(G >> 64);
            if (negp) {
                acc[w] -= p0;
                acc[w + 1] -= p1;
                acc[w + 2] -= p2;
            } else {
                acc[w] += p0;
                acc[w + 1] += p1;
                acc[w + 2] += p2;
            }
            continue;
        }
        const int rs = -sh;
        const uint64_t ip = rs >= 64 ? 0 : (u.m >> rs);
        const bool frac = rs >= 64 ? (u.m != 0) : ((u.m & ((1ULL << rs) - 1)) != 0);
        long long F = negp ? -(long long)(ip + (frac ? 1 : 0)) : (long long)ip;
        if (!frac) {
            bool seen = false;
#pragma unroll
            for (int r = 0; r < NIN; ++r) {
                if (r <= p || seen) continue;
                const uint64_t c = f64_bits(x[r]);
                if ((c & ABS) != 0) {
                    if ((c >> 63) != sign) F -= 1;
                    seen = true;
                }
            }
        }
        acc[0] += F;  // |F| < 2^53: the column sums absorb it before the carry pass
        done = true;
    }
    xr::carry_to_limbs(acc, X);
}

struct TcMdSplitGrid {
    const double* A[16]; int64_t lda, M; int32_t* e; int64_t a_tasks;
    const double* B[16]; int64_t ldb, N; int32_t* f; int64_t b_tasks;
    int64_t K, KB;
    uint16_t* planesA; uint16_t* planesB;
    bool a_vec;  // every plane of A 16-byte aligned and lda even: 16-byte loads
};

// Part s of a biased value Y as an f32 bit pattern (upper half = bf16).
template <int NP, int W>
__device__ __forceinline__ uint32_t md_part(const uint64_t (&y)[W], int s) {
    if (s == 0) {  // the first digit: 16 bits from position 8 (NP - 1), signed
        constexpr int pos = 8 * (NP - 1);
        const int i = pos >> 6, o = pos & 63;
        uint64_t v = 0, nx = 0;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            if (j == i) v = y[j];
            if (j == i + 1) nx = y[j];
        }
        const uint64_t bits = (v >> o) | (o > 48 ? nx << (64 - o) : 0);
        return __float_as_uint(__int2float_rn((int)(int16_t)(uint16_t)bits));
    }
    const int b = NP - 1 - s;  // byte of Y
    uint64_t limb = 0;
#pragma unroll
    for (int j = 0; j < W; ++j)
        if (j == (b >> 3)) limb = y[j];
    const uint32_t E = (uint32_t)(limb >> (8 * (b & 7))) & 0xFFu;
    return __float_as_uint(__fsub_rn(__uint_as_float(0x4B000000u | E), 8388736.0f));
}

// Y = X + 128 (256^(NP-2) + ... + 1) for one element (NIN doubles) against
// e': its low NP - 1 bytes are the balanced digits + 128, its top the first.
template <int NIN>
__device__ __forceinline__ void biased_md(const double (&x)[NIN], int ep, uint64_t (&y)[MdShape<NIN>::WX]) {
    constexpr int NP = MdShape<NIN>::NP, W = MdShape<NIN>::WX;
    uint64_t sign;
    fixed_point_n<NIN, W>(x, ep, 8 * NP, y, sign);
    if (sign) xr::negate(y);
    uint64_t c = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const int n = NP - 1 - 8 * i;  // bytes of the bias in this limb
        const uint64_t Ci = n >= 8 ? 0x8080808080808080ULL : n > 0 ? (0x8080808080808080ULL >> (64 - 8 * n)) : 0;
        const uint64_t u = y[i] + Ci;
        const uint64_t c1 = u < y[i];
        const uint64_t u2 = u + c;
        c = c1 | (u2 < u);
        y[i] = u2;
    }
}

// The NP parts of two consecutive elements (k, k + 1) of one part row: the
// lane writes word jj of 16-byte chunk kc of every part row, so the 32 lanes
// of a warp (kc = lane / 4, jj = lane % 4) write whole 128-byte rows.
template <int NIN>
__device__ __forceinline__ void store_parts2(uint16_t* planes, int64_t blk, int64_t KB, int64_t kb, int brows,
                                             int rin, int kc, int jj, const uint64_t (&y0)[MdShape<NIN>::WX],
                                             const uint64_t (&y1)[MdShape<NIN>::WX]) {
    constexpr int NP = MdShape<NIN>::NP, W = MdShape<NIN>::WX;
    uint8_t* base = reinterpret_cast<uint8_t*>(planes + (blk * NP * KB + kb) * ((int64_t)brows * TBK)) +
                    swizzled(rin, kc) + 4 * jj;
    const int64_t part_stride = KB * (int64_t)brows * TBK * 2;  // bytes from part s to s + 1
#pragma unroll
    for (int s = 0; s < NP; ++s)
        *reinterpret_cast<uint32_t*>(base + s * part_stride) =
            pack_bf16(md_part<NP, W>(y0, s), md_part<NP, W>(y1, s));
}

// A: one warp per row of A and k-block (64 k); lane (kc = lane / 4, jj =
// lane % 4) splits k = 64 kb + 8 kc + 2 jj and the next, loading both with
// 16-byte loads where aligned.  Rows up to Mp and k up to Kp are written (as
// 0 beyond the matrix).
template <int NIN>
__global__ void __launch_bounds__(256, MdShape<NIN>::SPLIT_MINB) split_md_rows_kernel(TcMdSplitGrid g) {
    constexpr int W = MdShape<NIN>::WX;
    const int lane = threadIdx.x & 31, kc = lane >> 2, jj = lane & 3;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * 8;
    for (int64_t task = gw; task < g.a_tasks; task += nw) {
        const int64_t r = task / g.KB, kb = task % g.KB;
        int ep = 1;
        double x0[NIN], x1[NIN];
#pragma unroll
        for (int q = 0; q < NIN; ++q) x0[q] = x1[q] = 0.0;
        const int64_t k = kb * TBK + kc * 8 + 2 * jj;
        if (r < g.M) {
            const int32_t er = g.e[r];
            if (kb == 0 && lane == 0 && er == EXP_NONE) g.e[r] = 0;
            ep = effective_exponent(er) + 1;
            if (g.a_vec && k + 1 < g.K) {
#pragma unroll
                for (int q = 0; q < NIN; ++q) {
                    const double2 v = __ldg(reinterpret_cast<const double2*>(g.A[q] + r * g.lda + k));
                    x0[q] = v.x;
                    x1[q] = v.y;
                }
            } else {
#pragma unroll
                for (int q = 0; q < NIN; ++q) {
                    if (k < g.K) x0[q] = __ldg(g.A[q] + r * g.lda + k);
                    if (k + 1 < g.K) x1[q] = __ldg(g.A[q] + r * g.lda + k + 1);
                }
            }
        }
        uint64_t y0[W], y1[W];
        biased_md<NIN>(x0, ep, y0);
        biased_md<NIN>(x1, ep, y1);
        store_parts2<NIN>(g.planesA, r / TBM, g.KB, kb, TBM, (int)(r % TBM), kc, jj, y0, y1);
    }
}

// B: one block per 8 columns of B and k-block.  The block stages the 64 x 8
// doubles of every plane in shared memory (each row of 8 columns is 64
// contiguous bytes of B), then warp w splits column 8 cg + w along k as the
// row kernel does (a column of B is a row of its part blocks).
constexpr int MD_COLS = 8;
constexpr int MD_TILE_LD = MD_COLS + 1;  // padded row of the staged tile
template <int NIN>
constexpr int md_cols_smem() { return NIN * TBK * MD_TILE_LD * 8; }

template <int NIN>
__global__ void __launch_bounds__(256, MdShape<NIN>::SPLIT_MINB) split_md_cols_kernel(TcMdSplitGrid g) {
    constexpr int W = MdShape<NIN>::WX;
    extern __shared__ double tile[];  // [NIN][64][MD_TILE_LD]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, kc = lane >> 2, jj = lane & 3;
    const int64_t groups = g.b_tasks / g.KB;
    for (int64_t task = blockIdx.x; task < g.b_tasks; task += gridDim.x) {
        const int64_t kb = task / groups, cg = task % groups;
        const int64_t n0 = cg * MD_COLS, k0 = kb * TBK;
        for (int idx = threadIdx.x; idx < NIN * TBK * MD_COLS; idx += blockDim.x) {
            const int q = idx / (TBK * MD_COLS), rem = idx % (TBK * MD_COLS);
            const int kk = rem / MD_COLS, c = rem % MD_COLS;
            const int64_t n = n0 + c, k = k0 + kk;
            tile[(q * TBK + kk) * MD_TILE_LD + c] = (n < g.N && k < g.K) ? __ldg(g.B[q] + k * g.ldb + n) : 0.0;
        }
        __syncthreads();
        const int64_t n = n0 + warp;
        int ep = 1;
        if (n < g.N) {
            const int32_t fr = g.f[n];
            if (kb == 0 && lane == 0 && fr == EXP_NONE) g.f[n] = 0;
            ep = effective_exponent(fr) + 1;
        }
        const int kk = kc * 8 + 2 * jj;
        double x0[NIN], x1[NIN];
#pragma unroll
        for (int q = 0; q < NIN; ++q) {
            x0[q] = tile[(q * TBK + kk) * MD_TILE_LD + warp];
            x1[q] = tile[(q * TBK + kk + 1) * MD_TILE_LD + warp];
        }
        __syncthreads();  // the tile is free for the next task
        uint64_t y0[W], y1[W];
        biased_md<NIN>(x0, ep, y0);
        biased_md<NIN>(x1, ep, y1);
        store_parts2<NIN>(g.planesB, n / TBN, g.KB, kb, TBN, (int)(n % TBN), kc, jj, y0, y1);
    }
}

struct PlanePtrs {
    double* c[16];  // the output planes (device pointers), passed by value
};

// Z = sum_d v_d 256^(NP-1-d) with v_d = sum over the k-splits, formed as
// column sums of 32-bit words, split by split (the sum is linear, so each
// split's int32 part sums are grouped by three and placed on their own; all
// loads of a split are independent), then one carry pass; rounded once into
// NIN doubles.
template <int NIN>
__global__ void __launch_bounds__(256) recombine_tc_md_kernel(const int32_t* __restrict__ P, int splits, int64_t Mp,
                                                              int64_t Np, const int32_t* __restrict__ e,
                                                              const int32_t* __restrict__ f, int64_t M, int64_t N,
                                                              PlanePtrs C, int64_t ldc) {
    constexpr int NP = MdShape<NIN>::NP, W = MdShape<NIN>::WZ, NW = 2 * W;
    constexpr int G = NP / 3, R = NP % 3;
    static_assert(8 * (NP - 3) + 63 + 24 < 32 * (NW + 2), "column sums cover the top group");
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const int64_t plane = Mp * Np;
    const int fj = effective_exponent(f[j]) + 1;
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        long long acc[NW + 2];
#pragma unroll
        for (int w = 0; w < NW + 2; ++w) acc[w] = 0;
        for (int zz = 0; zz < splits; ++zz) {
            const int32_t* p = P + ((int64_t)zz * NP) * plane + i * Np + j;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const long long h = ((long long)__ldg(p + (int64_t)(3 * g) * plane) * 256 +
                                     __ldg(p + (int64_t)(3 * g + 1) * plane)) * 256 +
                                    __ldg(p + (int64_t)(3 * g + 2) * plane);
                xr::add_at(acc, h, 8 * (NP - 3 - 3 * g));
            }
            if (R == 1) xr::add_at(acc, __ldg(p + (int64_t)(NP - 1) * plane), 0);
            if (R == 2)
                xr::add_at(acc, (long long)__ldg(p + (int64_t)(NP - 2) * plane) * 256 + __ldg(p + (int64_t)(NP - 1) * plane),
                           0);
        }
        // one carry pass: Z in W limbs (two's complement; |Z| < 2^(64 W - 1))
        uint64_t z[W];
        xr::carry_to_limbs(acc, z);
        const int q = effective_exponent(e[i]) + 1 + fj - TD * (NP + 1);
        double out[NIN];
        if (!xr::round_parts_scan<W>(z, q, out, NIN)) xr::round_parts_general<W>(z, q, out, NIN);
#pragma unroll
        for (int pq = 0; pq < NIN; ++pq) C.c[pq][i * ldc + j] = out[pq];
    }
}

template <int NIN>
cudaError_t split_md(const double* const* A, int64_t lda, int64_t M, int32_t* e, const double* const* B, int64_t ldb,
                     int64_t N, int32_t* f, int64_t K, int64_t Kp, uint16_t* planesA, uint16_t* planesB,
                     cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    TcMdSplitGrid g{};
    g.K = K;
    g.KB = Kp / TBK;
    if (A && M > 0) {
        bool vec = lda % 2 == 0;
        for (int q = 0; q < NIN; ++q) {
            g.A[q] = A[q];
            vec = vec && (uintptr_t)A[q] % 16 == 0;
        }
        g.lda = lda; g.M = M; g.e = e;
        g.a_tasks = round_up(M, PAIR_M) * g.KB;
        g.a_vec = vec;
    }
    if (B && N > 0) {
        for (int q = 0; q < NIN; ++q) g.B[q] = B[q];
        g.ldb = ldb; g.N = N; g.f = f;
        g.b_tasks = (round_up(N, TBN) / MD_COLS) * g.KB;
    }
    g.planesA = planesA;
    g.planesB = planesB;
    if (g.a_tasks > 0) {
        const unsigned blocks = (unsigned)std::min<int64_t>((g.a_tasks + 7) / 8, 0x7FFFFFFF);  // one task per warp
        split_md_rows_kernel<NIN><<<blocks, 256, 0, st>>>(g);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if (g.b_tasks > 0) {
        cudaError_t err = cudaFuncSetAttribute(split_md_cols_kernel<NIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               md_cols_smem<NIN>());
        if (err != cudaSuccess) return err;
        const unsigned blocks = (unsigned)std::min<int64_t>(g.b_tasks, 0x7FFFFFFF);  // one task per block
        split_md_cols_kernel<NIN><<<blocks, 256, md_cols_smem<NIN>(), st>>>(g);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

template <int NIN>
cudaError_t recombine_md(const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e, const int32_t* f,
                         int64_t M, int64_t N, double* const* C, int64_t ldc, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    PlanePtrs pc{};
    for (int q = 0; q < NIN; ++q) pc.c[q] = C[q];
    const unsigned gx = (unsigned)((N + 255) / 256);
    const unsigned gy = (unsigned)(M < 65535 ? M : 65535);
    recombine_tc_md_kernel<NIN><<<dim3(gx, gy), 256, 0, st>>>(P, splits, Mp, Np, e, f, M, N, pc, ldc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split_bf16_md(int nin, const double* const* A, int64_t lda, int64_t M, int32_t* e,
                                 const double* const* B, int64_t ldb, int64_t N, int32_t* f, int64_t K, int64_t Kp,
                                 uint16_t* planesA, uint16_t* planesB, cudaStream_t st) {
    if (nin == 8) return split_md<8>(A, lda, M, e, B, ldb, N, f, K, Kp, planesA, planesB, st);
    if (nin == 16) return split_md<16>(A, lda, M, e, B, ldb, N, f, K, Kp, planesA, planesB, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_slice_gemm_tc_md(int nin, const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                    int64_t Kp, int splits, int32_t* P, cudaStream_t st) {
    if (nin == 8) return launch_slice_gemm_parts<MdShape<8>::NP>(planesA, planesB, Mp, Np, Kp, splits, P, st);
    if (nin == 16) return launch_slice_gemm_parts<MdShape<16>::NP>(planesA, planesB, Mp, Np, Kp, splits, P, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_recombine_tc_md(int nin, const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                   const int32_t* f, int64_t M, int64_t N, double* const* C, int64_t ldc,
                                   cudaStream_t st) {
    if (nin == 8) return recombine_md<8>(P, splits, Mp, Np, e, f, M, N, C, ldc, st);
    if (nin == 16) return recombine_md<16>(P, splits, Mp, Np, e, f, M, N, C, ldc, st);
    return cudaErrorInvalidValue;
}

cudaError_t read_and_reset_wait_timeouts_tc_md(unsigned int* count) { return reset_tc_timeouts(count); }

DDG_DEFINE_CHECK_READER(check_record_tc_md)

}  // namespace ddg
