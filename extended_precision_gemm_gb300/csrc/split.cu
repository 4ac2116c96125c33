// split.cu -- step 1 of the dd GEMM: shared exponents and 13-bit part planes.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2 (split every
// double double into 8 parts of 13 bits: 4 quarters of hi, 4 of lo) with the
// parts of a row of A / column of B placed on one exponent grid (the goal of
// Section 3, Problems 3.2 and 3.4).  Bandwidth-bound: each input element is
// read as (hi, lo) and written as 8 parts.
//
// Three launches cover both operands: exponent reset, exponents (rows of A
// and columns of B in one grid), split (A tiles and B tiles in one grid).
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "digits.cuh"
#include "fixed_point.cuh"
#include "launch.cuh"

namespace ddg {
namespace {

constexpr uint64_t ABS_MASK = 0x7FFFFFFFFFFFFFFFULL;

__device__ __forceinline__ uint64_t abs_bits(double x) {
    return f64_bits(x) & ABS_MASK;
}

// ---------------------------------------------------------------------------
// Exponents: e[i] = max over the row of the smallest e with |A_hi| < 2^e
// (f[j] likewise over the column of B).  The maximum of |x| is taken on the
// IEEE bit patterns (for non-negative doubles the integer order of the bits
// is the order of the values) and combined over k-chunks with atomicMax.
// ---------------------------------------------------------------------------

__global__ void init_exponents_kernel(int32_t* e, int64_t M, int32_t* f, int64_t N, int32_t value) {
    pdl_wait();
    pdl_launch_dependents();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e != nullptr && i < M) e[i] = value;
    if (f != nullptr && i < N) f[i] = value;
}

// Work split of the exponent grid: one item per block, each thread issuing
// all its loads (8 x 16 bytes) before it reduces, so a block has 32 KB in
// flight, and the blocks in flight read one compact range (a grid-stride loop
// with fewer loads in flight reads at half the DRAM rate on GB300).
//   A-item: one row x EXP_A_SEG consecutive k (256 threads x 2 k x 8 loads);
//           block maximum, one atomicMax.
//   B-item: EXP_B_COLS columns x EXP_B_ROWS k (8 warps x 8 rows; a lane two
//           columns with 16-byte loads, or one); the 8 warps' maxima are
//           combined in shared memory, one atomicMax per column.
// Items are ordered so that neighbouring blocks read neighbouring memory:
// A by (row, k-segment), B by (k-segment, column group).
constexpr int EXP_THREADS = 256;
constexpr int EXP_LOADS = 8;
constexpr int64_t EXP_A_SEG = (int64_t)EXP_THREADS * 2 * EXP_LOADS;  // 4096 k
constexpr int EXP_B_ROWS = (EXP_THREADS / 32) * EXP_LOADS;           // 64 k

struct ExpGrid {
    const double* A_hi; int64_t lda, M, a_segs, a_items;
    const double* B_hi; int64_t ldb, N, b_groups, b_items;
    int64_t K;
    int32_t* e; int32_t* f;
    bool b_vec;  // B_hi 16-byte aligned and ldb even: two columns per lane, 16-byte loads
};

template <int VEC>
__device__ __forceinline__ void exponents_a_item(const ExpGrid& g, int64_t item, uint64_t* red) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int64_t row = item / g.a_segs;
    const int64_t k0 = (item % g.a_segs) * EXP_A_SEG;
    const int64_t k1 = min(g.K, k0 + EXP_A_SEG);
    // the row is read in [row * lda + k0, row * lda + k1): within the span of A
    const bool live = in_bounds(row * g.lda + k1 - 1, (g.M - 1) * g.lda + g.K, kSiteExpLoadA);
    const double* p = g.A_hi + row * g.lda;
    uint64_t m = 0;
    if (live) {
        if (VEC == 2) {
            double2 v[EXP_LOADS];
#pragma unroll
            for (int j = 0; j < EXP_LOADS; ++j) {
                const int64_t k = k0 + 2 * t + 2 * EXP_THREADS * j;
                v[j] = make_double2(0.0, 0.0);
                if (k + 1 < k1) v[j] = __ldg(reinterpret_cast<const double2*>(p + k));
                else if (k < k1) v[j].x = __ldg(p + k);
            }
#pragma unroll
            for (int j = 0; j < EXP_LOADS; ++j) m = max(m, max(abs_bits(v[j].x), abs_bits(v[j].y)));
        } else {
            double v[2 * EXP_LOADS];
#pragma unroll
            for (int j = 0; j < 2 * EXP_LOADS; ++j) {
                const int64_t k = k0 + t + EXP_THREADS * j;
                v[j] = k < k1 ? __ldg(p + k) : 0.0;
            }
#pragma unroll
            for (int j = 0; j < 2 * EXP_LOADS; ++j) m = max(m, abs_bits(v[j]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        m = max(m, (uint64_t)__shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)m, off));
    if (lane == 0) red[w] = m;
    __syncthreads();
    if (t == 0) {
        uint64_t mm = red[0];
#pragma unroll
        for (int j = 1; j < EXP_THREADS / 32; ++j) mm = max(mm, red[j]);
        if (mm != 0) atomicMax(&g.e[row], exponent_from_abs_bits(mm));
    }
}

__device__ __forceinline__ void exponents_b_item(const ExpGrid& g, int64_t item, uint64_t* red) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int per = g.b_vec ? 2 : 1;  // columns per lane
    const int64_t col = (item % g.b_groups) * 32 * per + (int64_t)lane * per;
    const int64_t k0 = (item / g.b_groups) * EXP_B_ROWS + (int64_t)w * EXP_LOADS;
    const int64_t k1 = min(g.K, k0 + EXP_LOADS);
    uint64_t m0 = 0, m1 = 0;
    if (col < g.N && k0 < g.K) {
        const bool pair = g.b_vec && col + 1 < g.N;
        if (in_bounds((k1 - 1) * g.ldb + col + (pair ? 1 : 0), (g.K - 1) * g.ldb + g.N, kSiteExpLoadB)) {
            const double* p = g.B_hi + col;
            if (pair) {
                double2 v[EXP_LOADS];
#pragma unroll
                for (int j = 0; j < EXP_LOADS; ++j)
                    v[j] = k0 + j < k1 ? __ldg(reinterpret_cast<const double2*>(p + (k0 + j) * g.ldb))
                                       : make_double2(0.0, 0.0);
#pragma unroll
                for (int j = 0; j < EXP_LOADS; ++j) {
                    m0 = max(m0, abs_bits(v[j].x));
                    m1 = max(m1, abs_bits(v[j].y));
                }
            } else {
                double v[EXP_LOADS];
#pragma unroll
                for (int j = 0; j < EXP_LOADS; ++j) v[j] = k0 + j < k1 ? __ldg(p + (k0 + j) * g.ldb) : 0.0;
#pragma unroll
                for (int j = 0; j < EXP_LOADS; ++j) m0 = max(m0, abs_bits(v[j]));
            }
        }
    }
    // red: [warp][64 columns]
    red[w * 64 + lane * per] = m0;
    if (per == 2) red[w * 64 + lane * 2 + 1] = m1;
    __syncthreads();
    if (t < 32 * per) {
        uint64_t mm = red[t];
#pragma unroll
        for (int j = 1; j < EXP_THREADS / 32; ++j) mm = max(mm, red[j * 64 + t]);
        const int64_t c = (item % g.b_groups) * 32 * per + t;
        if (mm != 0 && c < g.N) atomicMax(&g.f[c], exponent_from_abs_bits(mm));
    }
}

template <int VEC>
__global__ void __launch_bounds__(EXP_THREADS) exponents_kernel(ExpGrid g) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ uint64_t red[(EXP_THREADS / 32) * 64];
    const int64_t items = g.a_items + g.b_items;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        if (item < g.a_items) exponents_a_item<VEC>(g, item, red);
        else exponents_b_item(g, item - g.a_items, red);
        __syncthreads();  // red is reused by the next item
    }
}

// The 8 parts as int16, packed two per 32-bit word (part 2j in the low half).
__device__ __forceinline__ uint4 split_digits_i16(double hi, double lo, int e) {
    uint64_t sign;
    const unsigned __int128 X = fxp::fixed_point(hi, lo, e, sign);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t d0 = digit_field(X, 2 * j), d1 = digit_field(X, 2 * j + 1);
        if (sign) { d0 = (uint32_t)(-(int32_t)d0); d1 = (uint32_t)(-(int32_t)d1); }
        w[j] = (d0 & 0xFFFFu) | (d1 << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// Split.  A work item is one 32-row tile of A (32-column tile of B) and 32
// consecutive k (4 k-chunks): 32 lanes = rows (columns) x 8 warps = groups
// of 4 consecutive k.  Items [0, a_items) are A's, the rest B's.
// FP64 parts: the item's parts form one contiguous 64 KB block of the plane
// array ([chunk][part][k4 group][row in tile][k % 4]), written straight from
// registers in whole 32-byte DRAM sectors.
// int16 parts: layout [tile][k-chunk][k in chunk][row in tile][part]; each
// lane writes the 16 bytes of one element, a warp 512 contiguous bytes.
// ---------------------------------------------------------------------------

constexpr int SPLIT_THREADS = 256;
constexpr int SPLIT_CHUNKS = 32 / BK;                                                // k-chunks per item
constexpr int PART_STRIDE = (BK / 4) * TM * 4;                                       // doubles between parts

struct SplitGrid {
    const double* A_hi; const double* A_lo; int64_t lda, M, a_tiles;
    const double* B_hi; const double* B_lo; int64_t ldb, N, b_tiles;
    int64_t K, Kp, KT;  // KT = k-items per tile
    int32_t* e; int32_t* f;
    bool a_given, b_given;  // exponents supplied by the caller: never written
    void* planesA; void* planesB;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Load the 4 consecutive elements (k0 .. k0+3) of row / column `r` handled by
// this thread (zeros outside the matrix) and the exponent of that row or
// column; also writes back the final exponent of an all-zero row/column.
template <int VEC>
__device__ __forceinline__ int load_item(const SplitGrid& g, bool is_a, int64_t tile, int64_t k0, int lane,
                                         int w, int64_t kt, double (&hi)[4], double (&lo)[4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) hi[r] = lo[r] = 0.0;
    const int64_t rr = tile * TM + lane;
    if (is_a) {
        if (rr >= g.M) return 0;
        const int32_t er = g.e[rr];
        if (!g.a_given && kt == 0 && w == 0 && er == EXP_NONE) g.e[rr] = 0;
        const double* ph = g.A_hi + rr * g.lda + k0;
        const double* pl = g.A_lo + rr * g.lda + k0;
        if (!in_bounds(rr * g.lda + min(k0 + 3, g.K - 1), (g.M - 1) * g.lda + g.K, kSiteSplitLoadA))
            return effective_exponent(er);
        if (VEC == 2 && k0 + 3 < g.K) {
            double2 h0 = __ldg(reinterpret_cast<const double2*>(ph));
            double2 h1 = __ldg(reinterpret_cast<const double2*>(ph + 2));
            double2 l0 = __ldg(reinterpret_cast<const double2*>(pl));
            double2 l1 = __ldg(reinterpret_cast<const double2*>(pl + 2));
            hi[0] = h0.x; hi[1] = h0.y; hi[2] = h1.x; hi[3] = h1.y;
            lo[0] = l0.x; lo[1] = l0.y; lo[2] = l1.x; lo[3] = l1.y;
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (k0 + r < g.K) { hi[r] = __ldg(ph + r); lo[r] = __ldg(pl + r); }
        }
        return effective_exponent(er);
    }
    if (rr >= g.N) return 0;
    const int32_t fr = g.f[rr];
    if (!g.b_given && kt == 0 && w == 0 && fr == EXP_NONE) g.f[rr] = 0;
    if (!in_bounds(min(k0 + 3, g.K - 1) * g.ldb + rr, (g.K - 1) * g.ldb + g.N, kSiteSplitLoadB))
        return effective_exponent(fr);
#pragma unroll
    for (int r = 0; r < 4; ++r)
        if (k0 + r < g.K) {
            hi[r] = __ldg(g.B_hi + (k0 + r) * g.ldb + rr);
            lo[r] = __ldg(g.B_lo + (k0 + r) * g.ldb + rr);
        }
    return effective_exponent(fr);
}

// Decomposition of a work item index.
struct Item {
    bool is_a;
    int64_t tile, kt;
    int chunks;  // k-chunks present (the last k-item of a tile may be short)
};

__device__ __forceinline__ Item item_of(const SplitGrid& g, int64_t item, int64_t KC) {
    Item it;
    it.is_a = item < g.a_tiles * g.KT;
    const int64_t local = it.is_a ? item : item - g.a_tiles * g.KT;
    it.tile = local / g.KT;
    it.kt = local % g.KT;
    it.chunks = (int)min((int64_t)SPLIT_CHUNKS, KC - it.kt * SPLIT_CHUNKS);
    return it;
}

// One item per block (a grid-stride walk only past 2^31 - 1 items, with the
// next item's loads issued before the current one is split).  A lane keeps the fixed-point values
// of its 4 elements (one row, 4 consecutive k) and forms the parts one plane
// at a time: part s of the 4 elements is 32 contiguous bytes of the plane
// block, written by one 256-bit store, so a warp writes 1 KB per part and
// every DRAM sector is written whole, straight from registers.
__device__ __forceinline__ void st_global_v4(double* p, double a, double b, double c, double d) {
    asm volatile("st.global.v4.f64 [%0], {%1, %2, %3, %4};" ::"l"(p), "d"(a), "d"(b), "d"(c), "d"(d) : "memory");
}

template <int VEC>
__global__ void __launch_bounds__(SPLIT_THREADS, 4) split_f64_kernel(SplitGrid g) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t items = (g.a_tiles + g.b_tiles) * g.KT;
    const int64_t KC = g.Kp / BK;
    double nhi[4] = {0, 0, 0, 0}, nlo[4] = {0, 0, 0, 0};
    int nex = 0;
    int64_t item = blockIdx.x;
    Item nit;
    if (item < items) {
        nit = item_of(g, item, KC);
        if ((w >> 1) < nit.chunks)
            nex = load_item<VEC>(g, nit.is_a, nit.tile, nit.kt * 32 + 4 * w, lane, w, nit.kt, nhi, nlo);
    }
    for (; item < items; item += gridDim.x) {
        const Item it = nit;
        unsigned __int128 X[4];
        uint64_t sign[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) X[r] = fxp::fixed_point(nhi[r], nlo[r], nex, sign[r]);
        const int64_t next = item + gridDim.x;
        if (next < items) {
            nit = item_of(g, next, KC);
            if ((w >> 1) < nit.chunks)
                nex = load_item<VEC>(g, nit.is_a, nit.tile, nit.kt * 32 + 4 * w, lane, w, nit.kt, nhi, nlo);
        }
        if ((w >> 1) >= it.chunks) continue;  // this warp's k-chunk does not exist
        // part s of this warp's (k-chunk, k4 group): 32 rows x 4 k, 1 KB contiguous
        const int64_t off = (it.tile * KC + it.kt * SPLIT_CHUNKS + (w >> 1)) * CHUNK_DOUBLES + (w & 1) * TM * 4;
        const int64_t extent = (it.is_a ? g.a_tiles : g.b_tiles) * KC * CHUNK_DOUBLES;
        if (!in_bounds(off + (S - 1) * PART_STRIDE + TM * 4 - 1, extent, kSiteSplitStore)) continue;
        double* out = static_cast<double*>(it.is_a ? g.planesA : g.planesB) + off + lane * 4;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            double d[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) d[r] = small_int_to_double(digit_field(X[r], s), sign[r]);
            st_global_v4(out + s * PART_STRIDE, d[0], d[1], d[2], d[3]);
        }
    }
}

__device__ __forceinline__ int64_t i16_offset(int64_t tile, int64_t KC, int64_t k, int ti) {
    return (((tile * KC + k / BK) * BK + k % BK) * TM + ti) * S;
}

template <int VEC>
__global__ void __launch_bounds__(SPLIT_THREADS, 4) split_i16_kernel(SplitGrid g) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t items = (g.a_tiles + g.b_tiles) * g.KT;
    const int64_t KC = g.Kp / BK;
    double nhi[4] = {0, 0, 0, 0}, nlo[4] = {0, 0, 0, 0};
    int nex = 0;
    int64_t item = blockIdx.x;
    Item nit;
    if (item < items) {
        nit = item_of(g, item, KC);
        if ((w >> 1) < nit.chunks)
            nex = load_item<VEC>(g, nit.is_a, nit.tile, nit.kt * 32 + 4 * w, lane, w, nit.kt, nhi, nlo);
    }
    for (; item < items; item += gridDim.x) {
        const Item it = nit;
        double hi[4], lo[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) { hi[r] = nhi[r]; lo[r] = nlo[r]; }
        const int ex = nex;
        const int64_t next = item + gridDim.x;
        if (next < items) {
            nit = item_of(g, next, KC);
            if ((w >> 1) < nit.chunks)
                nex = load_item<VEC>(g, nit.is_a, nit.tile, nit.kt * 32 + 4 * w, lane, w, nit.kt, nhi, nlo);
        }
        if ((w >> 1) >= it.chunks) continue;
        const int64_t k0 = it.kt * 32 + 4 * w;
        int16_t* planes = static_cast<int16_t*>(it.is_a ? g.planesA : g.planesB);
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<uint4*>(planes + i16_offset(it.tile, KC, k0 + r, lane)) = split_digits_i16(hi[r], lo[r], ex);
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

DDG_DEFINE_CHECK_READER(check_record_split)

cudaError_t launch_reset_exponents(int32_t* e, int64_t M, int32_t* f, int64_t N, int32_t value,
                                   cudaStream_t st) {
    int64_t n = std::max(e ? M : 0, f ? N : 0);
    if (n == 0) return cudaSuccess;
    return launch_pdl(init_exponents_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, e, M, f, N, value);
}

cudaError_t launch_shared_exponents(const SplitOperand* A, const SplitOperand* B, int64_t K, int32_t zero_k_value,
                                    cudaStream_t st) {
    int32_t* e = A ? A->exp : nullptr;
    int32_t* f = B ? B->exp : nullptr;
    const int64_t M = A ? A->rows : 0, N = B ? B->rows : 0;
    if (K == 0) return launch_reset_exponents(e, M, f, N, zero_k_value, st);
    cudaError_t err = launch_reset_exponents(e, M, f, N, EXP_NONE, st);
    if (err != cudaSuccess) return err;
    return launch_exponents(A, B, K, st);
}

cudaError_t launch_exponents(const SplitOperand* A, const SplitOperand* B, int64_t K, cudaStream_t st) {
    if (K == 0) return cudaSuccess;
    ExpGrid g{};
    g.K = K;
    if (A && A->rows > 0) {
        g.A_hi = A->hi; g.lda = A->ld; g.M = A->rows; g.e = A->exp;
        g.a_segs = (K + EXP_A_SEG - 1) / EXP_A_SEG;
        g.a_items = A->rows * g.a_segs;
    }
    if (B && B->rows > 0) {
        g.b_vec = (uintptr_t)B->hi % 16 == 0 && B->ld % 2 == 0;
        g.B_hi = B->hi; g.ldb = B->ld; g.N = B->rows; g.f = B->exp;
        g.b_groups = (B->rows + (g.b_vec ? 63 : 31)) / (g.b_vec ? 64 : 32);
        g.b_items = g.b_groups * ((K + EXP_B_ROWS - 1) / EXP_B_ROWS);
    }
    const int64_t items = g.a_items + g.b_items;
    if (items == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>(items, 0x7FFFFFFF);
    const bool vec = !A || (((uintptr_t)A->hi % 16 == 0) && (A->ld % 2 == 0));
    return vec ? launch_pdl(exponents_kernel<2>, dim3(blocks), dim3(EXP_THREADS), 0, st, g)
               : launch_pdl(exponents_kernel<1>, dim3(blocks), dim3(EXP_THREADS), 0, st, g);
}

static SplitGrid make_split_grid(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                                 void* planesA, void* planesB) {
    SplitGrid g{};
    g.K = K;
    g.Kp = Kp;
    g.KT = (Kp / BK + SPLIT_CHUNKS - 1) / SPLIT_CHUNKS;
    if (A) {
        g.A_hi = A->hi; g.A_lo = A->lo; g.lda = A->ld; g.M = A->rows; g.a_tiles = (A->rows + TM - 1) / TM;
        g.e = A->exp; g.a_given = A->exp_given;
    }
    if (B) {
        g.B_hi = B->hi; g.B_lo = B->lo; g.ldb = B->ld; g.N = B->rows; g.b_tiles = (B->rows + TN - 1) / TN;
        g.f = B->exp; g.b_given = B->exp_given;
    }
    g.planesA = planesA;
    g.planesB = planesB;
    return g;
}

static bool a_vec(const SplitOperand* A) {
    return !A || (((uintptr_t)A->hi % 16 == 0) && ((uintptr_t)A->lo % 16 == 0) && (A->ld % 2 == 0));
}

// Split grids: one block per item.  The block scheduler hands out the items in
// order as blocks finish, so the blocks in flight write one compact range of
// the planes; a persistent grid drifts apart and spreads its writes over
// many DRAM pages (on GB300 a grid-stride loop of 256-bit stores reaches
// about 6.5 TB/s, the same stores from a one-item-per-block grid 7.7 TB/s).
static unsigned split_grid(int64_t items) {
    return (unsigned)std::min<int64_t>(items, 0x7FFFFFFF);
}

cudaError_t launch_split_f64(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                             double* planesA, double* planesB, cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    SplitGrid g = make_split_grid(A, B, K, Kp, planesA, planesB);
    const int64_t items = (g.a_tiles + g.b_tiles) * g.KT;
    if (items == 0) return cudaSuccess;
    const cudaError_t err = a_vec(A) ? launch_pdl(split_f64_kernel<2>, dim3(split_grid(items)), dim3(SPLIT_THREADS),
                                                  0, st, g)
                                     : launch_pdl(split_f64_kernel<1>, dim3(split_grid(items)), dim3(SPLIT_THREADS),
                                                  0, st, g);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_split_i16(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                             int16_t* planesA, int16_t* planesB, cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    SplitGrid g = make_split_grid(A, B, K, Kp, planesA, planesB);
    const int64_t items = (g.a_tiles + g.b_tiles) * g.KT;
    if (items == 0) return cudaSuccess;
    const unsigned blocks = split_grid(items);
    if (a_vec(A)) split_i16_kernel<2><<<blocks, SPLIT_THREADS, 0, st>>>(g);
    else split_i16_kernel<1><<<blocks, SPLIT_THREADS, 0, st>>>(g);
    return cudaGetLastError();
}

}  // namespace ddg
