// split.cu -- step 1 of the dd GEMM: shared exponents and 13-bit part planes.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2 (split every
// double double into 8 parts of 13 bits: 4 quarters of hi, 4 of lo) with the
// parts of a row of A / column of B placed on one exponent grid (the goal of
// Section 3, Problems 3.2 and 3.4).  Bandwidth-bound: each input element is
// read once as (hi, lo) and written as 8 doubles.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.cuh"

namespace ddg {
namespace {

constexpr uint64_t ABS_MASK = 0x7FFFFFFFFFFFFFFFULL;

__device__ __forceinline__ uint64_t abs_bits(double x) {
    return (uint64_t)__double_as_longlong(x) & ABS_MASK;
}

// ---------------------------------------------------------------------------
// Exponents: e[i] = max over the row of the smallest e with |A_hi| < 2^e.
// The maximum of |x| is taken on the IEEE bit patterns (for non-negative
// doubles the integer order of the bits is the order of the values).
// ---------------------------------------------------------------------------

__global__ void init_exponents_kernel(int32_t* e, int64_t M, int32_t* f, int64_t N, int32_t value) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e != nullptr && i < M) e[i] = value;
    if (f != nullptr && i < N) f[i] = value;
}

// One warp per row and k-chunk; 128-bit loads when VEC == 2.
template <int VEC>
__global__ void __launch_bounds__(256) row_exponents_kernel(const double* __restrict__ A_hi,
                                                            int64_t lda, int64_t M, int64_t K,
                                                            int64_t kchunk, int32_t* e) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= M) return;
    const int64_t k0 = (int64_t)blockIdx.y * kchunk;
    const int64_t k1 = min(K, k0 + kchunk);
    const double* p = A_hi + row * lda;
    uint64_t m = 0;
    if (VEC == 2) {
        // four independent 128-bit loads in flight per lane
        uint64_t m1 = 0, m2 = 0, m3 = 0;
        int64_t k = k0 + 2 * lane;
        for (; k + 193 < k1; k += 256) {
            const double2 v0 = __ldg(reinterpret_cast<const double2*>(p + k));
            const double2 v1 = __ldg(reinterpret_cast<const double2*>(p + k + 64));
            const double2 v2 = __ldg(reinterpret_cast<const double2*>(p + k + 128));
            const double2 v3 = __ldg(reinterpret_cast<const double2*>(p + k + 192));
            m = max(m, max(abs_bits(v0.x), abs_bits(v0.y)));
            m1 = max(m1, max(abs_bits(v1.x), abs_bits(v1.y)));
            m2 = max(m2, max(abs_bits(v2.x), abs_bits(v2.y)));
            m3 = max(m3, max(abs_bits(v3.x), abs_bits(v3.y)));
        }
        for (; k < k1; k += 64) {
            if (k + 1 < k1) {
                double2 v = __ldg(reinterpret_cast<const double2*>(p + k));
                m = max(m, max(abs_bits(v.x), abs_bits(v.y)));
            } else {
                m = max(m, abs_bits(__ldg(p + k)));
            }
        }
        m = max(max(m, m1), max(m2, m3));
    } else {
        for (int64_t k = k0 + lane; k < k1; k += 32) m = max(m, abs_bits(__ldg(p + k)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, (uint64_t)__shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)m, off));
    if (lane == 0 && m != 0) atomicMax(&e[row], exponent_from_abs_bits(m));
}

// One thread per column and k-chunk; a warp reads 32 consecutive columns of a
// row (256 contiguous bytes) per load.
__global__ void __launch_bounds__(128) col_exponents_kernel(const double* __restrict__ B_hi,
                                                            int64_t ldb, int64_t K, int64_t N,
                                                            int64_t kchunk, int32_t* f) {
    const int64_t col = (int64_t)blockIdx.x * 128 + threadIdx.x;
    if (col >= N) return;
    const int64_t k0 = (int64_t)blockIdx.y * kchunk;
    const int64_t k1 = min(K, k0 + kchunk);
    const double* p = B_hi + col;
    uint64_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    int64_t k = k0;
    for (; k + 7 < k1; k += 8) {  // eight loads in flight per thread
        const double x0 = __ldg(p + (k + 0) * ldb), x1 = __ldg(p + (k + 1) * ldb);
        const double x2 = __ldg(p + (k + 2) * ldb), x3 = __ldg(p + (k + 3) * ldb);
        const double x4 = __ldg(p + (k + 4) * ldb), x5 = __ldg(p + (k + 5) * ldb);
        const double x6 = __ldg(p + (k + 6) * ldb), x7 = __ldg(p + (k + 7) * ldb);
        m0 = max(m0, max(abs_bits(x0), abs_bits(x4)));
        m1 = max(m1, max(abs_bits(x1), abs_bits(x5)));
        m2 = max(m2, max(abs_bits(x2), abs_bits(x6)));
        m3 = max(m3, max(abs_bits(x3), abs_bits(x7)));
    }
    for (; k < k1; ++k) m0 = max(m0, abs_bits(__ldg(p + k * ldb)));
    uint64_t m = max(max(m0, m1), max(m2, m3));
    if (m != 0) atomicMax(&f[col], exponent_from_abs_bits(m));
}

// ---------------------------------------------------------------------------
// Digits.  X = floor(|hi + lo| * 2^(104 - e)) < 2^104 is formed exactly in
// 128-bit integer arithmetic; the parts are its 13-bit fields, most
// significant first, with the sign of the element.
//
// With |hi| = mh 2^Eh (mh < 2^53) and a normalised lo (|lo| <= ulp(hi)/2),
// put a = |hi| 2^(104-e) = mh 2^sh and b = |lo| 2^(104-e) <= 2^(sh-1):
//   same signs:      floor(a + b) = floor(a) + floor(b)
//                    (sh >= 0: a is an integer; sh < 0: b < 1/2 and
//                     frac(a) + b < 1)
//   opposite signs:  floor(a - b) = floor(a) - floor(b) - borrow, where
//                    borrow = [frac(b) > 0] when sh >= 0 (frac(a) = 0), and
//                    borrow = [frac(a) == 0] when sh < 0 (then 0 < b < 2^sh
//                    and frac(a) is 0 or >= 2^sh).
// The borrow is the move of Problem 3.3, eq. (7): the low double's opposite
// sign is taken from the high digits without changing the value.
// ---------------------------------------------------------------------------

struct Unpacked {
    uint64_t m;  // integer significand (< 2^53)
    int E;       // |x| = m * 2^E
};

__device__ __forceinline__ Unpacked unpack_abs(uint64_t bits) {
    uint64_t a = bits & ABS_MASK;
    int biased = (int)(a >> 52);
    uint64_t frac = a & ((1ULL << 52) - 1);
    Unpacked u;
    if (biased == 0) { u.m = frac; u.E = -1074; }
    else { u.m = frac | (1ULL << 52); u.E = biased - 1075; }
    return u;
}

// floor(m * 2^sh) for m < 2^53 (shifts beyond the 104-bit window are clamped
// so that out-of-contract inputs cannot shift by >= 128).
__device__ __forceinline__ unsigned __int128 scaled_floor(uint64_t m, int sh) {
    if (sh >= 0) return (unsigned __int128)m << (sh > 74 ? 74 : sh);
    if (sh <= -64) return 0;
    return (unsigned __int128)(m >> (-sh));
}

__device__ __forceinline__ bool scaled_frac_zero(uint64_t m, int sh) {
    if (sh >= 0) return true;
    if (sh <= -64) return m == 0;
    return (m & ((1ULL << (-sh)) - 1)) == 0;
}

// X = floor(|hi + lo| * 2^(104 - e)) and the sign of the element.
__device__ __forceinline__ unsigned __int128 fixed_point(double hi, double lo, int e, uint64_t& sign_out) {
    uint64_t hb = (uint64_t)__double_as_longlong(hi);
    uint64_t lb = (uint64_t)__double_as_longlong(lo);
    if ((hb & ABS_MASK) == 0) { hb = lb; lb = 0; }  // hi = 0: the element is lo alone
    const uint64_t sign = hb >> 63;
    unsigned __int128 X = 0;
    if ((hb & ABS_MASK) != 0) {
        Unpacked h = unpack_abs(hb);
        int sh = h.E + FIX - e;
        X = scaled_floor(h.m, sh);
        if ((lb & ABS_MASK) != 0) {
            Unpacked l = unpack_abs(lb);
            int sl = l.E + FIX - e;
            unsigned __int128 bint = scaled_floor(l.m, sl);
            if ((lb >> 63) == sign) {
                X += bint;
            } else {
                bool borrow = (sh >= 0) ? !scaled_frac_zero(l.m, sl) : scaled_frac_zero(h.m, sh);
                X -= bint + (borrow ? 1 : 0);
            }
        }
    }
    sign_out = sign;
    return X;
}

// 13-bit field s of X, most significant first.
__device__ __forceinline__ uint32_t digit_field(unsigned __int128 X, int s) {
    return (uint32_t)(X >> (DIGIT * (S - 1 - s))) & ((1u << DIGIT) - 1);
}

// The 8 parts as doubles (exact small integers).
__device__ __forceinline__ void split_digits(double hi, double lo, int e, double out[S]) {
    uint64_t sign;
    const unsigned __int128 X = fixed_point(hi, lo, e, sign);
#pragma unroll
    for (int s = 0; s < S; ++s) out[s] = small_int_to_double(digit_field(X, s), sign);
}

// The 8 parts as int16, packed two per 32-bit word (part 2j in the low half).
__device__ __forceinline__ uint4 split_digits_i16(double hi, double lo, int e) {
    uint64_t sign;
    const unsigned __int128 X = fixed_point(hi, lo, e, sign);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t d0 = digit_field(X, 2 * j), d1 = digit_field(X, 2 * j + 1);
        if (sign) { d0 = (uint32_t)(-(int32_t)d0); d1 = (uint32_t)(-(int32_t)d1); }
        w[j] = (d0 & 0xFFFFu) | (d1 << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Each split block covers one 32-row (A) or 32-column (B) tile and 32
// consecutive k (4 k-chunks).  Its parts form one contiguous 64 KB block of
// the plane array ([chunk][part][k4 group][row in tile][k % 4]); the block is
// assembled in shared memory and written with one bulk asynchronous copy
// (TMA engine), so every DRAM line is written whole.
constexpr int SPLIT_THREADS = 256;
constexpr int SPLIT_CHUNKS = 32 / BK;                              // k-chunks per block
constexpr size_t SPLIT_SMEM = (size_t)SPLIT_CHUNKS * CHUNK_DOUBLES * sizeof(double);  // 64 KB
constexpr int PART_STRIDE = (BK / 4) * TM * 4;                     // doubles between parts s, s+1

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Parts of 4 consecutive elements (k0 .. k0+3) of one row or column into the
// staging block, two elements per 16-byte shared-memory store.
__device__ __forceinline__ void stage_parts(const double (&hi)[4], const double (&lo)[4], int ex,
                                            double* dst) {
#pragma unroll
    for (int r = 0; r < 4; r += 2) {
        double d0[S], d1[S];
        split_digits(hi[r], lo[r], ex, d0);
        split_digits(hi[r + 1], lo[r + 1], ex, d1);
#pragma unroll
        for (int s = 0; s < S; ++s)
            *reinterpret_cast<double2*>(dst + s * PART_STRIDE + r) = make_double2(d0[s], d1[s]);
    }
}

// Write the staged block (`chunks` k-chunks) to global memory and wait until
// the copy has read shared memory, so the stage can be refilled.
__device__ __forceinline__ void flush_stage(double* stage, double* gdst, int chunks) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)chunks * CHUNK_DOUBLES * sizeof(double);
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                     "r"(smem_u32(stage)), "r"(bytes)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    __syncthreads();
}

// Rows of A.  Block = 32 rows (lanes) x 8 groups of 4 consecutive k (warps);
// blockIdx.x walks k in steps of 32, blockIdx.y strides over the row tiles.
// Each thread reads 4 hi and 4 lo values of its row (two 128-bit loads each
// when VEC == 2) and stages its 32 parts.
template <int VEC>
__global__ void __launch_bounds__(SPLIT_THREADS, 3) split_rows_kernel(const double* __restrict__ A_hi,
                                                                   const double* __restrict__ A_lo,
                                                                   int64_t lda, int64_t M, int64_t K,
                                                                   int64_t Kp, int32_t* e,
                                                                   double* __restrict__ planes) {
    extern __shared__ __align__(128) double stage[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t KC = Kp / BK;
    const int64_t kc0 = (int64_t)blockIdx.x * SPLIT_CHUNKS;
    const int chunks = (int)min((int64_t)SPLIT_CHUNKS, KC - kc0);
    const int64_t k0 = kc0 * BK + 4 * w;
    const bool active = (w >> 1) < chunks;  // this warp's k-chunk exists
    double* dst = stage + (((w >> 1) * S * (BK / 4) + (w & 1)) * TM + lane) * 4;
    const int64_t tiles = (M + TM - 1) / TM;
    for (int64_t mt = blockIdx.y; mt < tiles; mt += gridDim.y) {
        if (active) {
            const int64_t i = mt * TM + lane;
            double hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
            int ex = 0;
            if (i < M) {
                const int32_t er = e[i];
                ex = effective_exponent(er);
                if (blockIdx.x == 0 && w == 0 && er == EXP_NONE) e[i] = 0;
                const double* ph = A_hi + i * lda + k0;
                const double* pl = A_lo + i * lda + k0;
                if (VEC == 2 && k0 + 3 < K) {
                    double2 h0 = __ldg(reinterpret_cast<const double2*>(ph));
                    double2 h1 = __ldg(reinterpret_cast<const double2*>(ph + 2));
                    double2 l0 = __ldg(reinterpret_cast<const double2*>(pl));
                    double2 l1 = __ldg(reinterpret_cast<const double2*>(pl + 2));
                    hi[0] = h0.x; hi[1] = h0.y; hi[2] = h1.x; hi[3] = h1.y;
                    lo[0] = l0.x; lo[1] = l0.y; lo[2] = l1.x; lo[3] = l1.y;
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        if (k0 + r < K) { hi[r] = __ldg(ph + r); lo[r] = __ldg(pl + r); }
                }
            }
            stage_parts(hi, lo, ex, dst);
        }
        flush_stage(stage, planes + (mt * KC + kc0) * CHUNK_DOUBLES, chunks);
    }
}

// Columns of B (K x N row-major).  Block = 32 columns (lanes) x 8 groups of 4
// consecutive k (warps), grid as split_rows_kernel; every load of a warp
// reads 32 consecutive columns of one row.  Stages and writes as
// split_rows_kernel, in B's plane layout.
__global__ void __launch_bounds__(SPLIT_THREADS, 3) split_cols_kernel(const double* __restrict__ B_hi,
                                                                   const double* __restrict__ B_lo,
                                                                   int64_t ldb, int64_t K, int64_t N,
                                                                   int64_t Kp, int32_t* f,
                                                                   double* __restrict__ planes) {
    extern __shared__ __align__(128) double stage[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t KC = Kp / BK;
    const int64_t kc0 = (int64_t)blockIdx.x * SPLIT_CHUNKS;
    const int chunks = (int)min((int64_t)SPLIT_CHUNKS, KC - kc0);
    const int64_t k0 = kc0 * BK + 4 * w;
    const bool active = (w >> 1) < chunks;
    double* dst = stage + (((w >> 1) * S * (BK / 4) + (w & 1)) * TN + lane) * 4;
    const int64_t tiles = (N + TN - 1) / TN;
    for (int64_t nt = blockIdx.y; nt < tiles; nt += gridDim.y) {
        if (active) {
            const int64_t j = nt * TN + lane;
            double hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
            int ex = 0;
            if (j < N) {
                const int32_t fr = f[j];
                ex = effective_exponent(fr);
                if (blockIdx.x == 0 && w == 0 && fr == EXP_NONE) f[j] = 0;
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (k0 + r < K) {
                        hi[r] = __ldg(B_hi + (k0 + r) * ldb + j);
                        lo[r] = __ldg(B_lo + (k0 + r) * ldb + j);
                    }
            }
            stage_parts(hi, lo, ex, dst);
        }
        flush_stage(stage, planes + (nt * KC + kc0) * CHUNK_DOUBLES, chunks);
    }
}

// ---------------------------------------------------------------------------
// Part planes as int16 for the integer-pipe slice GEMM.  Layout
// [tile][k-chunk][k in chunk][row in tile][part]: the 8 parts of one element
// are 16 contiguous bytes, so one 128-bit load brings all of them.  A warp
// (32 rows or columns of a tile, one k) writes 512 contiguous bytes.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int64_t i16_offset(int64_t tile, int64_t KC, int64_t k, int ti) {
    return (((tile * KC + k / BK) * BK + k % BK) * TM + ti) * S;
}

template <int VEC>
__global__ void __launch_bounds__(256, 4) split_rows_i16_kernel(const double* __restrict__ A_hi,
                                                              const double* __restrict__ A_lo,
                                                              int64_t lda, int64_t M, int64_t K,
                                                              int64_t Kp, int32_t* e,
                                                              int16_t* __restrict__ planes) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t k0 = (int64_t)blockIdx.x * 32 + 4 * w;
    if (k0 >= Kp) return;
    const int64_t KC = Kp / BK;
    const int64_t tiles = (M + TM - 1) / TM;
    for (int64_t mt = blockIdx.y; mt < tiles; mt += gridDim.y) {
        const int64_t i = mt * TM + lane;
        double hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
        int ex = 0;
        if (i < M) {
            const int32_t er = e[i];
            ex = effective_exponent(er);
            if (blockIdx.x == 0 && w == 0 && er == EXP_NONE) e[i] = 0;
            const double* ph = A_hi + i * lda + k0;
            const double* pl = A_lo + i * lda + k0;
            if (VEC == 2 && k0 + 3 < K) {
                double2 h0 = __ldg(reinterpret_cast<const double2*>(ph));
                double2 h1 = __ldg(reinterpret_cast<const double2*>(ph + 2));
                double2 l0 = __ldg(reinterpret_cast<const double2*>(pl));
                double2 l1 = __ldg(reinterpret_cast<const double2*>(pl + 2));
                hi[0] = h0.x; hi[1] = h0.y; hi[2] = h1.x; hi[3] = h1.y;
                lo[0] = l0.x; lo[1] = l0.y; lo[2] = l1.x; lo[3] = l1.y;
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (k0 + r < K) { hi[r] = __ldg(ph + r); lo[r] = __ldg(pl + r); }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<uint4*>(planes + i16_offset(mt, KC, k0 + r, lane)) = split_digits_i16(hi[r], lo[r], ex);
    }
}

__global__ void __launch_bounds__(256, 4) split_cols_i16_kernel(const double* __restrict__ B_hi,
                                                              const double* __restrict__ B_lo,
                                                              int64_t ldb, int64_t K, int64_t N,
                                                              int64_t Kp, int32_t* f,
                                                              int16_t* __restrict__ planes) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t k0 = (int64_t)blockIdx.x * 32 + 4 * w;
    if (k0 >= Kp) return;
    const int64_t KC = Kp / BK;
    const int64_t tiles = (N + TN - 1) / TN;
    for (int64_t nt = blockIdx.y; nt < tiles; nt += gridDim.y) {
        const int64_t j = nt * TN + lane;
        double hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
        int ex = 0;
        if (j < N) {
            const int32_t fr = f[j];
            ex = effective_exponent(fr);
            if (blockIdx.x == 0 && w == 0 && fr == EXP_NONE) f[j] = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (k0 + r < K) {
                    hi[r] = __ldg(B_hi + (k0 + r) * ldb + j);
                    lo[r] = __ldg(B_lo + (k0 + r) * ldb + j);
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<uint4*>(planes + i16_offset(nt, KC, k0 + r, lane)) = split_digits_i16(hi[r], lo[r], ex);
    }
}

int num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 152;
    return sms;
}

}  // namespace

cudaError_t launch_split_rows_i16(const double* A_hi, const double* A_lo, int64_t lda, int64_t M,
                                  int64_t K, int64_t Kp, int32_t* e, int16_t* planes, cudaStream_t st) {
    const int64_t Mp = round_up(M, TM);
    if (Mp == 0 || Kp == 0) return cudaSuccess;
    dim3 grid((unsigned)((Kp + 31) / 32), (unsigned)std::min<int64_t>(Mp / TM, 65535));
    const bool vec = ((uintptr_t)A_hi % 16 == 0) && ((uintptr_t)A_lo % 16 == 0) && (lda % 2 == 0);
    if (vec) split_rows_i16_kernel<2><<<grid, 256, 0, st>>>(A_hi, A_lo, lda, M, K, Kp, e, planes);
    else split_rows_i16_kernel<1><<<grid, 256, 0, st>>>(A_hi, A_lo, lda, M, K, Kp, e, planes);
    return cudaGetLastError();
}

cudaError_t launch_split_cols_i16(const double* B_hi, const double* B_lo, int64_t ldb, int64_t K,
                                  int64_t N, int64_t Kp, int32_t* f, int16_t* planes, cudaStream_t st) {
    const int64_t Np = round_up(N, TN);
    if (Np == 0 || Kp == 0) return cudaSuccess;
    dim3 grid((unsigned)((Kp + 31) / 32), (unsigned)std::min<int64_t>(Np / TN, 65535));
    split_cols_i16_kernel<<<grid, 256, 0, st>>>(B_hi, B_lo, ldb, K, N, Kp, f, planes);
    return cudaGetLastError();
}

cudaError_t launch_init_exponents(int32_t* e, int64_t M, int32_t* f, int64_t N, int64_t K,
                                  cudaStream_t st) {
    int64_t n = M > N ? M : N;
    if (n == 0) return cudaSuccess;
    // K = 0 has no elements to take a maximum over: every exponent is final 0.
    init_exponents_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(e, M, f, N, K == 0 ? 0 : EXP_NONE);
    return cudaGetLastError();
}

cudaError_t launch_row_exponents(const double* A_hi, int64_t lda, int64_t M, int64_t K,
                                 int32_t* e, cudaStream_t st) {
    if (M == 0 || K == 0) return cudaSuccess;
    const int64_t row_blocks = (M + 7) / 8;
    const int64_t want = 4LL * num_sms();
    int64_t ksplit = (want + row_blocks - 1) / row_blocks;
    ksplit = std::max<int64_t>(1, std::min<int64_t>(ksplit, (K + 511) / 512));
    const int64_t kchunk = round_up((K + ksplit - 1) / ksplit, 64);
    ksplit = (K + kchunk - 1) / kchunk;
    dim3 grid((unsigned)row_blocks, (unsigned)ksplit);
    const bool vec = ((uintptr_t)A_hi % 16 == 0) && (lda % 2 == 0);
    if (vec) row_exponents_kernel<2><<<grid, 256, 0, st>>>(A_hi, lda, M, K, kchunk, e);
    else row_exponents_kernel<1><<<grid, 256, 0, st>>>(A_hi, lda, M, K, kchunk, e);
    return cudaGetLastError();
}

cudaError_t launch_col_exponents(const double* B_hi, int64_t ldb, int64_t K, int64_t N,
                                 int32_t* f, cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    const int64_t col_blocks = (N + 127) / 128;
    const int64_t want = 4LL * num_sms();
    int64_t ksplit = (want + col_blocks - 1) / col_blocks;
    ksplit = std::max<int64_t>(1, std::min<int64_t>(ksplit, (K + 63) / 64));
    const int64_t kchunk = (K + ksplit - 1) / ksplit;
    ksplit = (K + kchunk - 1) / kchunk;
    dim3 grid((unsigned)col_blocks, (unsigned)ksplit);
    col_exponents_kernel<<<grid, 128, 0, st>>>(B_hi, ldb, K, N, kchunk, f);
    return cudaGetLastError();
}

cudaError_t launch_split_rows(const double* A_hi, const double* A_lo, int64_t lda, int64_t M,
                              int64_t K, int64_t Kp, int32_t* e, double* planes, cudaStream_t st) {
    const int64_t Mp = round_up(M, TM);
    if (Mp == 0 || Kp == 0) return cudaSuccess;
    dim3 grid((unsigned)((Kp / BK + SPLIT_CHUNKS - 1) / SPLIT_CHUNKS), (unsigned)std::min<int64_t>(Mp / TM, 65535));
    const bool vec = ((uintptr_t)A_hi % 16 == 0) && ((uintptr_t)A_lo % 16 == 0) && (lda % 2 == 0);
    cudaError_t err;
    if (vec) {
        err = cudaFuncSetAttribute(split_rows_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPLIT_SMEM);
        if (err != cudaSuccess) return err;
        split_rows_kernel<2><<<grid, SPLIT_THREADS, SPLIT_SMEM, st>>>(A_hi, A_lo, lda, M, K, Kp, e, planes);
    } else {
        err = cudaFuncSetAttribute(split_rows_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPLIT_SMEM);
        if (err != cudaSuccess) return err;
        split_rows_kernel<1><<<grid, SPLIT_THREADS, SPLIT_SMEM, st>>>(A_hi, A_lo, lda, M, K, Kp, e, planes);
    }
    return cudaGetLastError();
}

cudaError_t launch_split_cols(const double* B_hi, const double* B_lo, int64_t ldb, int64_t K,
                              int64_t N, int64_t Kp, int32_t* f, double* planes, cudaStream_t st) {
    const int64_t Np = round_up(N, TN);
    if (Np == 0 || Kp == 0) return cudaSuccess;
    dim3 grid((unsigned)((Kp / BK + SPLIT_CHUNKS - 1) / SPLIT_CHUNKS), (unsigned)std::min<int64_t>(Np / TN, 65535));
    cudaError_t err = cudaFuncSetAttribute(split_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPLIT_SMEM);
    if (err != cudaSuccess) return err;
    split_cols_kernel<<<grid, SPLIT_THREADS, SPLIT_SMEM, st>>>(B_hi, B_lo, ldb, K, N, Kp, f, planes);
    return cudaGetLastError();
}

}  // namespace ddg
