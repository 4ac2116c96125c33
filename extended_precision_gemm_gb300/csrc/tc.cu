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
//     each product is at most 2^14, so 512 of them sum to at most 2^23 and the
//     f32 accumulator is exact; every 512 products per output ("a chunk") the
//     accumulator is read from tensor memory and added into an exact int32
//     total (|P_d| <= 13 K 2^14 < 2^31 for K <= 8192 per k-split);
//  3. Z = sum_d P_d 2^(8 (12 - d)) exactly (256-bit), rounded once to the
//     nearest double double of Z 2^(e'_i + f'_j - 112).
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "fixed_point.cuh"
#include "fixed_point_md.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"
#include "wide_int.cuh"
#include "exact_round.cuh"

namespace ddg {
namespace {

constexpr int TS = DDGEMM_TC_SLICES;        // 13 parts
constexpr int TD = DDGEMM_TC_DIGIT_BITS;    // 8 bits per part
constexpr int TBM = DDGEMM_TC_BLOCK_M;      // 128 rows of A per block
constexpr int TBN = DDGEMM_TC_TILE_N;       // 256 columns of B per block
constexpr int TBK = DDGEMM_TC_CHUNK_K;      // 64 k per block (128-byte rows)
constexpr int QS = DDGEMM_TC_QD_SLICES;     // 27 parts of a quad double
constexpr int QFIX = QS * TD;               // 216 fraction bits
static_assert(TS * TD == fxp::FIX_BITS, "13 parts of 8 bits cover the 104-bit fixed-point value");

// Largest k per slice-GEMM CTA (a k-split) for NP parts: NP 2^14 per k-step
// keeps the int32 totals of a split below 2^31.
__host__ __device__ constexpr int ksplit_max(int np) { return np <= TS ? DDGEMM_TC_MAX_K_SPLIT : DDGEMM_TC_QD_MAX_K_SPLIT; }
static_assert(TBK * 2 == 128, "one block row is one 128-byte swizzle row");

constexpr int PAIR_M = DDGEMM_TC_TILE_M;    // 256 output rows per CTA pair
constexpr int A_BLOCK_BYTES = TBM * TBK * 2;  // 16 KB
constexpr int B_HALF_BYTES = (TBN / 2) * TBK * 2;  // 16 KB: half of a 256-row block of B
constexpr int STAGE_BLOCKS = 2;   // k-blocks per ring stage: 8 MMAs per wait and commit
constexpr int STAGES = 3;
constexpr int STAGE_BYTES = STAGE_BLOCKS * (A_BLOCK_BYTES + B_HALF_BYTES);  // 64 KB
static_assert(PAIR_M == 2 * TBM, "a CTA pair covers two row blocks of A");
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024;  // + alignment slack
constexpr int CHUNK_BLOCKS = 8;   // blocks of 64 k summed in f32 before a flush (512 products)
constexpr int UMMA_K = 16;        // k of one tcgen05.mma (kind::f16)
constexpr int EPI_WARPS = 8;
constexpr int GEMM_THREADS = 64 + EPI_WARPS * 32;  // producer warp, MMA warp, epilogue
constexpr uint32_t TMEM_COLS = 512;  // two f32 accumulators of 128 x 256
constexpr uint32_t IDESC = tc5::idesc_bf16_f32(PAIR_M, TBN);  // pair MMA: M = 256
constexpr unsigned long long WAIT_NS = 2000000000ULL;  // bounded waits: 2 s
constexpr int TILE_GROUP = 8;     // row blocks per group in the tile order (L2 reuse)

static_assert(CHUNK_BLOCKS * TBK * 128 * 128 <= (1 << 23), "a chunk's f32 sums stay within 2^23");
static_assert((long long)TS * ksplit_max(TS) * 128 * 128 < (1LL << 31), "int32 totals per k-split");
static_assert((long long)QS * ksplit_max(QS) * 128 * 128 < (1LL << 31), "int32 totals per k-split");

__device__ unsigned int g_wait_timeouts_tc = 0;

// ---------------------------------------------------------------------------
// Step 1: bf16 parts.
// ---------------------------------------------------------------------------

// Byte offset of element (row r, 16-byte chunk kc of k) in a block: rows of
// 128 bytes, chunk kc of row r stored at position kc ^ (r % 8).
__device__ __forceinline__ uint32_t swizzled(int r, int kc) { return (uint32_t)(r * 128 + ((kc ^ (r & 7)) << 4)); }

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

// Two parts' bf16 patterns in one word (first element in the low half).
__device__ __forceinline__ uint32_t pack_bf16(uint32_t f_first, uint32_t f_second) {
    return __byte_perm(f_first, f_second, 0x7632u);
}

struct TcSplitGrid {
    const double* A_hi; const double* A_lo; int64_t lda, M; int32_t* e; int64_t a_tasks;
    const double* B_hi; const double* B_lo; int64_t ldb, N; int32_t* f; int64_t b_tasks;
    int64_t K, KB;  // KB = k-blocks of 64
    uint16_t* planesA; uint16_t* planesB;
    bool a_vec;     // A_hi, A_lo 16-byte aligned and lda even: 128-bit loads
};

// One warp per task, 256 elements each.  A task: 4 rows of A x one k-block
// (lane = row (lane/8), 8 consecutive k (lane%8)): 512 contiguous bytes of hi
// per row read, 512 contiguous bytes per part written.  B task: 32 columns of
// B x 8 consecutive k (lane = column): each load instruction reads 256
// contiguous bytes of a row of B; each lane writes one 16-byte chunk of its
// part rows (the 8 tasks of a k-block complete the 128-byte rows in L2).
// Rows / k beyond the matrix are written as 0.
__global__ void __launch_bounds__(256, 3) split_bf16_kernel(TcSplitGrid g) {
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
            if (r < g.M) {
                const int32_t er = g.e[r];
                if (kb == 0 && kc == 0 && er == EXP_NONE) g.e[r] = 0;
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
#pragma unroll
            for (int s = 0; s < TS; ++s) {
                uint8_t* blk = reinterpret_cast<uint8_t*>(g.planesA + ((mt * TS + s) * g.KB + kb) * (TBM * TBK));
                *reinterpret_cast<uint4*>(blk + swizzled(rin, kc)) = make_uint4(w[s][0], w[s][1], w[s][2], w[s][3]);
            }
        } else {
            // B task: 32 columns x 8 k (one 16-byte chunk of every part row)
            const int64_t local = task - g.a_tasks;
            const int64_t cg = local / (g.KB * 8), kq = local % (g.KB * 8);
            const int64_t kb = kq >> 3;
            const int kc = (int)(kq & 7);
            const int64_t n = cg * 32 + lane;
            int ep = 1;
            if (n < g.N) {
                const int32_t fr = g.f[n];
                if (kq == 0 && fr == EXP_NONE) g.f[n] = 0;
                ep = effective_exponent(fr) + 1;
            }
            const int64_t k0 = kb * TBK + kc * 8;
            double hi[8], lo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool in = n < g.N && k0 + j < g.K;
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
#pragma unroll
            for (int s = 0; s < TS; ++s) {
                uint8_t* blk = reinterpret_cast<uint8_t*>(g.planesB + ((nt * TS + s) * g.KB + kb) * (TBN * TBK));
                *reinterpret_cast<uint4*>(blk + swizzled(nin, kc)) = make_uint4(w[s][0], w[s][1], w[s][2], w[s][3]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Step 2: P_d on the tensor cores.  One cluster of two CTAs (a CTA pair on two
// SMs) per (256 x 256 output block, k-split); the pair's MMAs are M = 256,
// N = 256, K = 16 (tcgen05 cta_group::2): each CTA holds its 128 rows of A and
// its 128 rows of B (columns of C) for a k-block, and its 128 rows of the
// accumulators.  10 warps per CTA:
//   warp 0 (one thread): bulk copies of this CTA's part halves into a 3-stage
//           ring (64 KB per stage: two 64-k blocks of one pair (s, t));
//   warp 1: allocates 512 TMEM columns in both CTAs (two f32 accumulators of
//           128 x 256 per CTA); in the even CTA one thread issues the MMAs (4
//           per 64-k block) once both CTAs' stage is full; in the odd CTA one
//           thread forwards the completion of each of its stages to the even
//           CTA;
//   warps 2-9: read each finished chunk from TMEM (warp w reads lanes
//           32 (w % 4) .. +31, i.e. rows, and one half of the columns), add it
//           into int32 totals in registers, and store the totals of P_d.
// The order of work is d = 0..12, then s = 0..d (t = d - s), then k-blocks;
// a chunk is 8 consecutive k-blocks of one d (512 products per output; the
// last chunk of a d may be shorter).  Chunks alternate between the two accumulators, so the MMAs of
// one chunk overlap the read-out of the previous one.  Completion of MMAs
// reaches both CTAs through multicast commits; the release of an
// accumulator needs all 16 epilogue warps of the pair.
// ---------------------------------------------------------------------------

struct TcGemmArgs {
    const uint16_t* planesA;
    const uint16_t* planesB;
    int32_t* P;       // [split][d][Mp][Np]
    int64_t Mp, Np;
    int64_t KB;       // k-blocks in the planes
    int64_t kb_per_split;
    int MT, NT;       // output blocks of 256 x 256 along M and N
};

__device__ __forceinline__ void note_timeout(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicAdd(&g_wait_timeouts_tc, 1u);
}

template <int NP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    slice_gemm_tc_kernel(TcGemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * STAGES + 4 + 1];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
    const bool leader = rank == 0;

    // output block of this pair (grouped order: TILE_GROUP row blocks share
    // their column blocks while they are in L2)
    const int64_t tile = blockIdx.x >> 1;
    const int64_t per_group = (int64_t)TILE_GROUP * g.NT;
    const int64_t group = tile / per_group;
    const int64_t first_m = group * TILE_GROUP;
    const int64_t gsize = min((int64_t)TILE_GROUP, (int64_t)g.MT - first_m);
    const int64_t mt = first_m + (tile % per_group) % gsize;
    const int64_t nt = (tile % per_group) / gsize;
    const int64_t z = blockIdx.y;
    const int64_t kb0 = z * g.kb_per_split;
    const int64_t nkb = max((int64_t)0, min(g.KB, kb0 + g.kb_per_split) - kb0);
    const int64_t a_block = mt * 2 + rank;  // this CTA's 128 rows of A

    const uint32_t full0 = smem_addr(&bars[0]), empty0 = smem_addr(&bars[STAGES]);
    const uint32_t pfull0 = smem_addr(&bars[2 * STAGES]);
    const uint32_t accf0 = smem_addr(&bars[3 * STAGES]), acce0 = smem_addr(&bars[3 * STAGES + 2]);
    const uint32_t done_bar = smem_addr(&bars[3 * STAGES + 4]);

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
            mbar_init(pfull0 + 8 * i, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 2 * EPI_WARPS);
        }
        mbar_init(done_bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc5::tmem_alloc_pair(smem_addr(&tmem_slot), TMEM_COLS);
        tc5::tmem_relinquish_pair();
    }
    tc5::fence_before_sync();
    cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated
    tc5::fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---- producer (both CTAs): a stage holds up to two k-blocks of one pair ----
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            for (int d = 0; d < NP && !abort_flag; ++d) {
                for (int s = 0; s <= d && !abort_flag; ++s) {
                    const int t = d - s;
                    const uint16_t* a_src = g.planesA + ((a_block * NP + s) * g.KB + kb0) * (TBM * TBK);
                    const uint16_t* b_src =
                        g.planesB + ((nt * NP + t) * g.KB + kb0) * (TBN * TBK) + rank * (TBN / 2) * TBK;
                    for (int64_t kb = 0; kb < nkb; kb += STAGE_BLOCKS) {
                        const int nb = (int)min((int64_t)STAGE_BLOCKS, nkb - kb);
                        if (!mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1, WAIT_NS)) {
                            note_timeout(&abort_flag);
                            break;
                        }
                        uint8_t* dst = smem + stage * STAGE_BYTES;
                        mbar_expect_tx(full0 + 8 * stage, (uint32_t)nb * (A_BLOCK_BYTES + B_HALF_BYTES));
                        // consecutive k-blocks of A are contiguous; B's halves are not
                        bulk_load(dst, a_src + kb * (TBM * TBK), (uint32_t)nb * A_BLOCK_BYTES, full0 + 8 * stage);
                        for (int j = 0; j < nb; ++j)
                            bulk_load(dst + STAGE_BLOCKS * A_BLOCK_BYTES + j * B_HALF_BYTES,
                                      b_src + (kb + j) * (TBN * TBK), B_HALF_BYTES, full0 + 8 * stage);
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // copies still in flight must land before the CTA exits
            const int64_t first = issued > STAGES ? issued - STAGES : 0;
            for (int64_t j = first; j < issued; ++j)
                if (!mbar_wait_bounded(full0 + 8 * (uint32_t)(j % STAGES), (uint32_t)((j / STAGES) & 1), WAIT_NS))
                    note_timeout(&abort_flag);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---- MMA issuer (even CTA) ----
            // One thread issues every MMA of the pair, so the loop is kept
            // short: the descriptor of a block is the ring's first descriptor
            // plus the block's offset (the address field counts 16-byte units;
            // a k sub-step adds 32 bytes), counters are 32-bit, and the abort
            // flag is read only when a wait fails.
            const uint32_t ring = smem_addr(smem);
            const uint64_t adesc0 = tc5::desc_kmajor_sw128(ring);
            const uint64_t bdesc0 = tc5::desc_kmajor_sw128(ring + STAGE_BLOCKS * A_BLOCK_BYTES);
            const int nkb32 = (int)nkb;
            uint32_t stage = 0, phase = 0, chunk = 0, buf = 0;
            bool ok = true;
            for (int d = 0; d < NP && ok; ++d) {
                int left = (d + 1) * nkb32;  // k-blocks of this d still to issue
                int in_chunk = 0;            // k-blocks issued into the current chunk
                for (int s = 0; s <= d && ok; ++s) {
                    for (int kb = 0; kb < nkb32; kb += STAGE_BLOCKS) {
                        const int nb = min(STAGE_BLOCKS, nkb32 - kb);
                        if (!mbar_wait_bounded(full0 + 8 * stage, phase, WAIT_NS) ||
                            !mbar_wait_bounded(pfull0 + 8 * stage, phase, WAIT_NS)) {
                            if (!abort_flag) note_timeout(&abort_flag);
                            ok = false;
                            break;
                        }
                        tc5::fence_after_sync();
#pragma unroll
                        for (int j = 0; j < STAGE_BLOCKS; ++j) {
                            if (j >= nb) break;
                            if (in_chunk == 0) {
                                buf = chunk & 1;
                                if (!mbar_wait_bounded(acce0 + 8 * buf, ((chunk >> 1) & 1) ^ 1, WAIT_NS)) {
                                    if (!abort_flag) note_timeout(&abort_flag);
                                    ok = false;
                                    break;
                                }
                                tc5::fence_after_sync();
                            }
                            const uint32_t d_tmem = tmem + buf * TBN;
                            const uint64_t off = (uint64_t)((stage * STAGE_BYTES) >> 4);
                            const uint64_t ad = adesc0 + off + (uint64_t)(j * (A_BLOCK_BYTES >> 4));
                            const uint64_t bd = bdesc0 + off + (uint64_t)(j * (B_HALF_BYTES >> 4));
                            tc5::mma_bf16_pair(d_tmem, ad, bd, IDESC, in_chunk != 0 ? 1u : 0u);
#pragma unroll
                            for (int kk = 1; kk < TBK / UMMA_K; ++kk)
                                tc5::mma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, IDESC, 1u);
                            --left;
                            if (++in_chunk == CHUNK_BLOCKS || left == 0) {
                                tc5::commit_pair(accf0 + 8 * buf, 0x3);  // the chunk is complete in both CTAs
                                ++chunk;
                                in_chunk = 0;
                            }
                        }
                        if (!ok) break;
                        tc5::commit_pair(empty0 + 8 * stage, 0x3);  // the stage is free in both CTAs
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // every MMA issued has finished (in both CTAs) before either
            // releases its tensor memory or shared memory
            tc5::commit_pair(done_bar, 0x3);
            if (!mbar_wait_bounded(done_bar, 0, WAIT_NS)) note_timeout(&abort_flag);
        } else if (lane == 0) {
            // ---- forwarder (odd CTA): its stage s is full -> tell the even CTA ----
            uint32_t stage = 0, phase = 0;
            const int64_t total = (int64_t)(NP * (NP + 1) / 2) * ((nkb + STAGE_BLOCKS - 1) / STAGE_BLOCKS);
            for (int64_t j = 0; j < total; ++j) {
                if (abort_flag || !mbar_wait_bounded(full0 + 8 * stage, phase, WAIT_NS)) {
                    if (!abort_flag) note_timeout(&abort_flag);
                    break;
                }
                mbar_arrive_remote(pfull0 + 8 * stage, 0);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            // the even CTA's MMAs read this CTA's shared memory and write its
            // tensor memory: wait until they have all finished
            if (!mbar_wait_bounded(done_bar, 0, WAIT_NS)) note_timeout(&abort_flag);
        }
    } else {
        // ---- epilogue: warps 2..9 (both CTAs) ----
        const int q = warp & 3;                  // TMEM lanes 32q .. 32q + 31
        const int half = (warp - 2) >> 2;        // columns 128 half .. + 127
        const int row = q * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128);
        int64_t chunk = 0;
        bool ok = true;
        for (int d = 0; d < NP; ++d) {
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            const int64_t nch = ok ? ((int64_t)(d + 1) * nkb + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS : 0;
            for (int64_t c = 0; c < nch; ++c, ++chunk) {
                const uint32_t buf = (uint32_t)(chunk & 1), use = (uint32_t)(chunk >> 1);
                if (abort_flag || !mbar_wait_bounded(accf0 + 8 * buf, use & 1, WAIT_NS)) {
                    if (!abort_flag) note_timeout(&abort_flag);
                    ok = false;
                    break;
                }
                tc5::fence_after_sync();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t v[32];
                    tc5::ld32(lane_base + buf * TBN + j * 32, v);
                    // every chunk sum is an integer-valued f32 with |x| <= 2^23:
                    // the conversion is exact (one instruction each)
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[j * 32 + i] += __float2int_rz(__uint_as_float(v[i]));
                }
                tc5::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (leader) mbar_arrive(acce0 + 8 * buf);
                    else mbar_arrive_remote(acce0 + 8 * buf, 0);
                }
            }
            int32_t* dst =
                g.P + (((z * NP + d) * g.Mp + mt * PAIR_M + rank * TBM + row) * g.Np + nt * TBN + half * 128);
#pragma unroll
            for (int i = 0; i < 128; i += 4)
                *reinterpret_cast<int4*>(dst + i) = make_int4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        }
    }

    // neither CTA leaves while its peer may still touch its shared memory
    tc5::fence_before_sync();
    cluster_sync();
    tc5::fence_after_sync();
    if (warp == 1) {
        __syncwarp();  // the whole warp, converged, releases tensor memory
        tc5::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Step 3: exact sum of the parts and one rounding into a double double.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) recombine_tc_kernel(const int32_t* __restrict__ P, int splits, int64_t Mp,
                                                           int64_t Np, const int32_t* __restrict__ e,
                                                           const int32_t* __restrict__ f, int64_t M, int64_t N,
                                                           double* __restrict__ C_hi, double* __restrict__ C_lo,
                                                           int64_t ldc) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const int64_t plane = Mp * Np;
    const int fj = effective_exponent(f[j]) + 1;
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        long long v[TS];
        const int32_t* p = P + i * Np + j;
#pragma unroll
        for (int d = 0; d < TS; ++d) v[d] = __ldg(p + (int64_t)d * plane);
        for (int zz = 1; zz < splits; ++zz) {
#pragma unroll
            for (int d = 0; d < TS; ++d) v[d] += __ldg(p + ((int64_t)zz * TS + d) * plane);
        }
        const int q = effective_exponent(e[i]) + 1 + fj - TD * (TS + 1);
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
        C_hi[i * ldc + j] = out[0];
        C_lo[i * ldc + j] = out[1];
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

// One warp per task of 256 elements, as for double doubles: an A task is 4 rows
// x 64 k (lane = row (lane/8), 8 consecutive k (lane%8)), a B task 32 columns
// x 8 k (lane = column).  Each lane forms Y for its 8 elements, then writes one
// 16-byte chunk of each of the 27 part rows.
__global__ void __launch_bounds__(256) split_bf16_qd_kernel(TcQdSplitGrid g) {
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
            const int64_t local = task - g.a_tasks;
            const int64_t kq = local % (g.KB * 8);
            kb = kq >> 3;
            kc = (int)(kq & 7);
            r = (local / (g.KB * 8)) * 32 + lane;
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
        const int32_t* p = P + i * Np + j;
        // all loads of a split are issued before any is used
        long long v[QS];
#pragma unroll
        for (int d = 0; d < QS; ++d) v[d] = __ldg(p + (int64_t)d * plane);
        for (int zz = 1; zz < splits; ++zz) {
#pragma unroll
            for (int d = 0; d < QS; ++d) v[d] += __ldg(p + ((int64_t)zz * QS + d) * plane);
        }
        const int q = effective_exponent(e[i]) + 1 + fj - TD * (QS + 1);
        uint64_t z[4];
        xr::exact_sum<QS, 4>(v, z);
        double out[4];
        if (xr::fast_path_ok(z, q)) {
            xr::round_parts<4, 4>(z, q, out);
        } else {
            wide::U256 Z;
            Z.lo = ((wide::u128)z[1] << 64) | z[0];
            Z.hi = ((wide::u128)z[3] << 64) | z[2];
            wide::round_into_doubles<4>(Z, q, out);
        }
#pragma unroll
        for (int pq = 0; pq < 4; ++pq) Cs[pq][i * ldc + j] = out[pq];
    }
}

int num_sms_tc() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 152;
    return sms;
}

}  // namespace

cudaError_t launch_split_bf16(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                              uint16_t* planesA, uint16_t* planesB, cudaStream_t st) {
    if (Kp == 0) return cudaSuccess;
    TcSplitGrid g{};
    g.K = K;
    g.KB = Kp / TBK;
    if (A) {
        g.A_hi = A->hi; g.A_lo = A->lo; g.lda = A->ld; g.M = A->rows; g.e = A->exp;
        g.a_tasks = (round_up(A->rows, PAIR_M) / 4) * g.KB;
        g.a_vec = (uintptr_t)A->hi % 16 == 0 && (uintptr_t)A->lo % 16 == 0 && A->ld % 2 == 0;
    }
    if (B) {
        g.B_hi = B->hi; g.B_lo = B->lo; g.ldb = B->ld; g.N = B->rows; g.f = B->exp;
        g.b_tasks = (round_up(B->rows, TBN) / 32) * g.KB * 8;
    }
    g.planesA = planesA;
    g.planesB = planesB;
    const int64_t tasks = g.a_tasks + g.b_tasks;
    if (tasks == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((tasks + 7) / 8, (int64_t)num_sms_tc() * 8));
    split_bf16_kernel<<<blocks, 256, 0, st>>>(g);
    return cudaGetLastError();
}

template <int NP>
static cudaError_t launch_slice_gemm_parts(const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                           int64_t Kp, int splits, int32_t* P, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    if (splits < 1 || Mp % PAIR_M != 0 || Np % TBN != 0 || Kp % TBK != 0) return cudaErrorInvalidValue;
    if (((Kp / TBK + splits - 1) / splits) * TBK > ksplit_max(NP)) return cudaErrorInvalidValue;
    cudaError_t err =
        cudaFuncSetAttribute(slice_gemm_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (err != cudaSuccess) return err;
    TcGemmArgs g;
    g.planesA = planesA;
    g.planesB = planesB;
    g.P = P;
    g.Mp = Mp;
    g.Np = Np;
    g.KB = Kp / TBK;
    g.kb_per_split = (g.KB + splits - 1) / splits;
    g.MT = (int)(Mp / PAIR_M);
    g.NT = (int)(Np / TBN);
    dim3 grid((unsigned)(2 * (int64_t)g.MT * g.NT), (unsigned)splits);  // clusters of 2 along x
    slice_gemm_tc_kernel<NP><<<grid, GEMM_THREADS, GEMM_SMEM, st>>>(g);
    return cudaGetLastError();
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
    recombine_tc_kernel<<<dim3(gx, gy), 256, 0, st>>>(P, splits, Mp, Np, e, f, M, N, C_hi, C_lo, ldc);
    return cudaGetLastError();
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
        g.b_tasks = (round_up(N, TBN) / 32) * g.KB * 8;
    }
    g.planesA = planesA;
    g.planesB = planesB;
    const int64_t tasks = g.a_tasks + g.b_tasks;
    if (tasks == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((tasks + 7) / 8, (int64_t)num_sms_tc() * 8));
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

cudaError_t read_and_reset_wait_timeouts_tc(unsigned int* count) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(count, g_wait_timeouts_tc, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_timeouts_tc, &zero, sizeof(unsigned int));
}

}  // namespace ddg
