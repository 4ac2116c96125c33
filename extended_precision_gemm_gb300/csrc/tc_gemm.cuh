// tc_gemm.cuh -- the slice-pair GEMM of the bf16 variants on CTA pairs
// (tcgen05 cta_group::2), shared by the double-double / quad-double file and
// the octo / hexa-double file: constants of the part-block layout, the
// kernel templated on the number of parts, and its launcher.  Everything is
// in an unnamed namespace, so each including file gets its own copy (and its
// own count of bounded waits that gave up).
#pragma once

#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace ddg {
namespace {

constexpr int TD = DDGEMM_TC_DIGIT_BITS;    // 8 bits per part
constexpr int TBM = DDGEMM_TC_BLOCK_M;      // 128 rows of A per block
constexpr int TBN = DDGEMM_TC_TILE_N;       // 256 columns of B per block
constexpr int TBK = DDGEMM_TC_CHUNK_K;      // 64 k per block (128-byte rows)

// Largest k per slice-GEMM CTA (a k-split) for NP parts: the largest power of
// two with NP K 2^14 < 2^31, so that the int32 totals of a split stay exact
// (8192 for 13 parts, 4096 for 27, 2048 for 54, 1024 for 107).
__host__ __device__ constexpr int ksplit_max(int np) {
    int k = 1 << 20;
    while ((long long)np * k * 128 * 128 >= (1LL << 31)) k >>= 1;
    return k;
}
static_assert(ksplit_max(13) == DDGEMM_TC_MAX_K_SPLIT && ksplit_max(27) == DDGEMM_TC_QD_MAX_K_SPLIT,
              "k-split bounds");
static_assert(TBK * 2 == 128, "one block row is one 128-byte swizzle row");

constexpr int PAIR_M = DDGEMM_TC_TILE_M;    // 256 output rows per CTA pair
constexpr int A_BLOCK_BYTES = TBM * TBK * 2;  // 16 KB
constexpr int B_HALF_BYTES = (TBN / 2) * TBK * 2;  // 16 KB: half of a 256-row block of B
constexpr int STAGE_BLOCKS = 2;   // k-blocks per ring stage: 8 MMAs per wait and commit
constexpr int STAGES = 3;
constexpr int STAGE_BYTES = STAGE_BLOCKS * (A_BLOCK_BYTES + B_HALF_BYTES);  // 64 KB
static_assert(PAIR_M == 2 * TBM, "a CTA pair covers two row blocks of A");
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024;  // + alignment slack
constexpr int CHUNK_BLOCKS = 16;  // blocks of 64 k summed in f32 before a flush (1024 products)
constexpr int UMMA_K = 16;        // k of one tcgen05.mma (kind::f16)
constexpr int EPI_WARPS = 8;
constexpr int GEMM_THREADS = 64 + EPI_WARPS * 32;  // producer warp, MMA warp, epilogue
constexpr uint32_t TMEM_COLS = 512;  // two f32 accumulators of 128 x 256
constexpr uint32_t IDESC = tc5::idesc_bf16_f32(PAIR_M, TBN);  // pair MMA: M = 256
constexpr unsigned long long WAIT_NS = 2000000000ULL;  // bounded waits: 2 s
constexpr int TILE_GROUP = 8;     // row blocks per group in the tile order (L2 reuse)

static_assert(CHUNK_BLOCKS * TBK * 128 * 128 <= (1 << 24), "a chunk's f32 sums stay within 2^24");

__device__ unsigned int g_wait_timeouts_tc = 0;

// Byte offset of element (row r, 16-byte chunk kc of k) in a block: rows of
// 128 bytes, chunk kc of row r stored at position kc ^ (r % 8).
__device__ __forceinline__ uint32_t swizzled(int r, int kc) { return (uint32_t)(r * 128 + ((kc ^ (r & 7)) << 4)); }

// Two parts' bf16 patterns in one word (first element in the low half).
__device__ __forceinline__ uint32_t pack_bf16(uint32_t f_first, uint32_t f_second) {
    return __byte_perm(f_first, f_second, 0x7632u);
}

// ---------------------------------------------------------------------------
// Step 2: P_d on the tensor cores.  Persistent clusters of two CTAs (a CTA
// pair on two SMs, as many pairs as can be resident) share out the units of
// work (a diagonal d of a 256 x 256 output block and k-split: d + 1 pairs);
// the pair's MMAs are M = 256, N = 256, K = 16 (tcgen05 cta_group::2): each
// CTA holds its 128 rows of A and its 128 rows of B (columns of C) for a
// k-block, and its 128 rows of the accumulators.  10 warps per CTA:
//   warp 0 (one thread): tensor copies of this CTA's part halves into a
//           3-stage ring (64 KB per stage: two 64-k blocks of one pair
//           (s, t)); the copies of both CTAs complete on the even CTA's
//           barrier of the stage (cta_group::2 copies);
//   warp 1: allocates 512 TMEM columns in both CTAs (two f32 accumulators of
//           128 x 256 per CTA); in the even CTA one thread issues the MMAs (4
//           per 64-k block) once the stage is full in both CTAs;
//   warps 2-9: read each finished chunk from TMEM (warp w reads lanes
//           32 (w % 4) .. +31, i.e. rows, and one half of the columns), add it
//           into int32 totals in registers, and store the totals of P_d.
// Within a unit the order of work is s = 0..d (t = d - s), then k-blocks; a
// chunk is 16 consecutive k-blocks of one unit (1024 products per output; the
// last chunk of a unit may be shorter).  Chunks alternate between the two
// accumulators, also across units, so the MMAs of one chunk overlap the
// read-out of the previous one and the store of a finished unit.  Completion
// of MMAs reaches both CTAs through multicast commits; the release of an
// accumulator needs all 16 epilogue warps of the pair.
// ---------------------------------------------------------------------------

struct TcGemmArgs {
    int32_t* P;       // [split][d][Mp][Np]
    int64_t Mp, Np;
    int64_t KB;       // k-blocks in the planes
    int64_t kb_per_split;
    int MT, NT;       // output blocks of 256 x 256 along M and N
    int splits;       // k-splits
    int pairs;        // CTA pairs in the grid
    int64_t units;    // output blocks x k-splits x NP diagonals
};

// A unit of work: diagonal d of one output block and k-split, i.e. the d + 1
// pairs (s, d - s) over the split's k-blocks.  Units are numbered from the
// heaviest diagonal (d = NP - 1) down to d = 0; within a diagonal by k-split,
// then by output block in grouped order (TILE_GROUP row blocks share their
// column blocks while they are in L2).
struct Unit {
    int64_t mt, nt, z, kb0, nkb;
    int d;
};

__device__ __forceinline__ Unit unit_of(const TcGemmArgs& g, int64_t u, int np) {
    Unit w;
    const int64_t tiles = (int64_t)g.MT * g.NT;
    const int64_t per_d = tiles * g.splits;
    w.d = np - 1 - (int)(u / per_d);
    const int64_t rem = u % per_d;
    w.z = rem / tiles;
    const int64_t tile = rem % tiles;
    const int64_t per_group = (int64_t)TILE_GROUP * g.NT;
    const int64_t group = tile / per_group;
    const int64_t first_m = group * TILE_GROUP;
    const int64_t gsize = min((int64_t)TILE_GROUP, (int64_t)g.MT - first_m);
    w.mt = first_m + (tile % per_group) % gsize;
    w.nt = (tile % per_group) / gsize;
    w.kb0 = w.z * g.kb_per_split;
    w.nkb = max((int64_t)0, min(g.KB, w.kb0 + g.kb_per_split) - w.kb0);
    return w;
}

// The r-th unit of CTA pair p: units are dealt out in rounds of one unit per
// pair, the order of the pairs reversed every other round.  Unit weights fall
// along the numbering (a shorter last k-split aside), so the pairs' totals
// stay within about one light unit of each other, and in every round the
// pairs work on neighbouring output blocks at the same diagonal (their copies
// share L2).
__device__ __forceinline__ int64_t unit_index(const TcGemmArgs& g, int64_t p, int64_t r) {
    return r * g.pairs + ((r & 1) ? g.pairs - 1 - p : p);
}

__device__ __forceinline__ void note_timeout(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicAdd(&g_wait_timeouts_tc, 1u);
}

template <int NP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    slice_gemm_tc_kernel(const __grid_constant__ TcGemmArgs g, const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * STAGES + 4 + 1];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
    const bool leader = rank == 0;

    // both CTAs of a pair walk the same units
    const int64_t pair = blockIdx.x >> 1;

    const uint32_t full0 = smem_addr(&bars[0]), empty0 = smem_addr(&bars[STAGES]);
    const uint32_t accf0 = smem_addr(&bars[2 * STAGES]), acce0 = smem_addr(&bars[2 * STAGES + 2]);
    const uint32_t done_bar = smem_addr(&bars[2 * STAGES + 4]);

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
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
            // The copies of both CTAs complete on the even CTA's full barrier
            // (tensor copies with cta_group::2), which expects the bytes of both.
            const uint32_t full_lead0 = cluster_addr(full0, 0);
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            for (int64_t r = 0, u; (u = unit_index(g, pair, r)) < g.units && !abort_flag; ++r) {
                const Unit w = unit_of(g, u, NP);
                const int d = w.d;
                const int64_t a_block = w.mt * 2 + rank;  // this CTA's 128 rows of A
                const int64_t nkb = w.nkb;
                for (int s = 0; s <= d && !abort_flag; ++s) {
                    const int t = d - s;
                    // first 128-byte row of the k-blocks in the tensors of part rows
                    const int a_row = (int)(((a_block * NP + s) * g.KB + w.kb0) * TBM);
                    const int b_row = (int)(((w.nt * NP + t) * g.KB + w.kb0) * TBN + rank * (TBN / 2));
                    for (int64_t kb = 0; kb < nkb; kb += STAGE_BLOCKS) {
                        const int nb = (int)min((int64_t)STAGE_BLOCKS, nkb - kb);
                        if (!mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1, WAIT_NS)) {
                            note_timeout(&abort_flag);
                            break;
                        }
                        uint8_t* dst = smem + stage * STAGE_BYTES;
                        if (leader)
                            mbar_expect_tx(full0 + 8 * stage, 2u * (uint32_t)nb * (A_BLOCK_BYTES + B_HALF_BYTES));
                        const uint32_t bar = full_lead0 + 8 * stage;
                        for (int j = 0; j < nb; ++j) {
                            tma_load_2d_pair(dst + j * A_BLOCK_BYTES, &tmA, 0, a_row + (int)(kb + j) * TBM, bar);
                            tma_load_2d_pair(dst + STAGE_BLOCKS * A_BLOCK_BYTES + j * B_HALF_BYTES, &tmB, 0,
                                             b_row + (int)(kb + j) * TBN, bar);
                        }
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // copies still in flight must land before the CTA exits: the even
            // CTA waits for its last stages to fill (its barriers count the
            // bytes of both CTAs); the odd CTA, whose copies complete on the
            // even CTA's barriers, waits for its last stages to be consumed
            // (fill j is consumed when phase j / STAGES of its stage's empty
            // barrier completes)
            const int64_t first = issued > STAGES ? issued - STAGES : 0;
            for (int64_t j = first; j < issued; ++j) {
                const uint32_t bar = (leader ? full0 : empty0) + 8 * (uint32_t)(j % STAGES);
                if (!mbar_wait_bounded(bar, (uint32_t)((j / STAGES) & 1), WAIT_NS)) {
                    if (!abort_flag) note_timeout(&abort_flag);
                    break;
                }
            }
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
            uint32_t stage = 0, phase = 0, chunk = 0, buf = 0;
            bool ok = true, issued_any = false;
            for (int64_t r = 0, u; (u = unit_index(g, pair, r)) < g.units && ok; ++r) {
                const Unit w = unit_of(g, u, NP);
                const int d = w.d;
                const int nkb32 = (int)w.nkb;
                int left = (d + 1) * nkb32;  // k-blocks of this d still to issue
                int in_chunk = 0;            // k-blocks issued into the current chunk
                for (int s = 0; s <= d && ok; ++s) {
                    for (int kb = 0; kb < nkb32; kb += STAGE_BLOCKS) {
                        const int nb = min(STAGE_BLOCKS, nkb32 - kb);
                        if (!mbar_wait_bounded(full0 + 8 * stage, phase, WAIT_NS)) {  // both CTAs' copies
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
                            issued_any = true;
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
            if (issued_any) {
                tc5::commit_pair(done_bar, 0x3);
                if (!mbar_wait_bounded(done_bar, 0, WAIT_NS)) note_timeout(&abort_flag);
            }
        } else if (lane == 0) {
            // ---- odd CTA: nothing to issue ----
            int64_t total = 0;  // stages the producers fill for this pair's units
            for (int64_t r = 0, u; (u = unit_index(g, pair, r)) < g.units; ++r) {
                const Unit w = unit_of(g, u, NP);
                total += (int64_t)(w.d + 1) * ((w.nkb + STAGE_BLOCKS - 1) / STAGE_BLOCKS);
            }
            // the even CTA's MMAs read this CTA's shared memory and write its
            // tensor memory: wait until they have all finished (a pair whose
            // share is empty issues none)
            if (total > 0 && !mbar_wait_bounded(done_bar, 0, WAIT_NS)) note_timeout(&abort_flag);
        }
    } else {
        // ---- epilogue: warps 2..9 (both CTAs) ----
        const int q = warp & 3;                  // TMEM lanes 32q .. 32q + 31
        const int half = (warp - 2) >> 2;        // columns 128 half .. + 127
        const int row = q * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128);
        int64_t chunk = 0;
        bool ok = true;
        for (int64_t r = 0, u; (u = unit_index(g, pair, r)) < g.units; ++r) {
            const Unit w = unit_of(g, u, NP);
            const int d = w.d;
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            const int64_t nch = ok ? ((int64_t)(d + 1) * w.nkb + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS : 0;
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
                    // every chunk sum is an integer-valued f32 with |x| <= 2^24:
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
            const int64_t off = ((w.z * NP + d) * g.Mp + w.mt * PAIR_M + rank * TBM + row) * g.Np + w.nt * TBN +
                                half * 128;
            int32_t* dst = g.P + off;
            if (in_bounds(off + 127, (int64_t)g.splits * NP * g.Mp * g.Np, kSiteTcGemmStoreP)) {
#pragma unroll
                for (int i = 0; i < 128; i += 4)
                    *reinterpret_cast<int4*>(dst + i) = make_int4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
            }
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

int num_sms_tc() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 152;
    return sms;
}

// CTA pairs of the GEMM that can be resident at once: a cluster of two needs
// both SMs in one GPC, so this can be below half the SM count.
template <int NP>
int resident_pairs() {
    static std::atomic<int> cached[64];  // per device; 0 = not asked yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        dev = 0;
    }
    const int known = cached[dev].load(std::memory_order_relaxed);
    if (known > 0) return known;
    int n = 0;
    if (cudaFuncSetAttribute(slice_gemm_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(2 * std::max(1, num_sms_tc() / 2)), 1, 1);
        cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = GEMM_SMEM;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, slice_gemm_tc_kernel<NP>, &cfg) != cudaSuccess) n = 0;
    }
    if (n <= 0) {
        // no answer (no device, or a failure that may pass): half the SMs,
        // not remembered, so that a later call asks again
        (void)cudaGetLastError();
        return std::max(1, num_sms_tc() / 2);
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static std::atomic<EncodeTiledFn> cached{nullptr};
    EncodeTiledFn fn = cached.load(std::memory_order_acquire);
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
            cached.store(fn, std::memory_order_release);
        } else {
            (void)cudaGetLastError();
        }
    }
    return fn;
}

// The part blocks of one operand as a 2-D tensor of `rows` rows of 64 bf16
// (128 bytes), copied in boxes of 128 rows.  The blocks are already swizzled
// in memory, so the copies move bytes unchanged (no swizzle in the map).
cudaError_t make_part_map(CUtensorMap* m, const uint16_t* planes, int64_t rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return cudaErrorNotSupported;
    if (rows <= 0 || rows >= (1LL << 31) || (uintptr_t)planes % 16 != 0) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)TBK, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)TBK * 2};
    const cuuint32_t box[2] = {(cuuint32_t)TBK, (cuuint32_t)TBM};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(planes), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NP>
cudaError_t launch_slice_gemm_parts(const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                           int64_t Kp, int splits, int32_t* P, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    if (splits < 1 || Mp % PAIR_M != 0 || Np % TBN != 0 || Kp % TBK != 0) return cudaErrorInvalidValue;
    if (((Kp / TBK + splits - 1) / splits) * TBK > ksplit_max(NP)) return cudaErrorInvalidValue;
    cudaError_t err =
        cudaFuncSetAttribute(slice_gemm_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (err != cudaSuccess) return err;
    TcGemmArgs g;
    g.P = P;
    g.Mp = Mp;
    g.Np = Np;
    g.KB = Kp / TBK;
    g.kb_per_split = (g.KB + splits - 1) / splits;
    g.MT = (int)(Mp / PAIR_M);
    g.NT = (int)(Np / TBN);
    g.splits = splits;
    g.units = (int64_t)g.MT * g.NT * splits * NP;
    // as many persistent CTA pairs as can be resident (never more than units)
    g.pairs = (int)std::max<int64_t>(1, std::min<int64_t>(resident_pairs<NP>(), g.units));
    CUtensorMap tmA, tmB;  // with K = 0 no copy is issued: the maps stay unused
    memset(&tmA, 0, sizeof(tmA));
    memset(&tmB, 0, sizeof(tmB));
    if (g.KB > 0) {
        err = make_part_map(&tmA, planesA, (Mp / TBM) * NP * g.KB * TBM);
        if (err == cudaSuccess) err = make_part_map(&tmB, planesB, (Np / TBN) * NP * g.KB * TBN);
        if (err != cudaSuccess) return err;
    }
    dim3 grid((unsigned)(2 * g.pairs), 1);  // clusters of 2 along x
    slice_gemm_tc_kernel<NP><<<grid, GEMM_THREADS, GEMM_SMEM, st>>>(g, tmA, tmB);
    return cudaGetLastError();
}

// This translation unit's count of bounded waits that gave up, read once the
// work on `st` before it has finished (synchronises `st`).
cudaError_t peek_tc_timeouts(unsigned int* count, cudaStream_t st) {
    cudaError_t err = cudaMemcpyFromSymbolAsync(count, g_wait_timeouts_tc, sizeof(unsigned int), 0,
                                                cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    return err;
}

// Read and clear this translation unit's count of bounded waits that gave up.
cudaError_t reset_tc_timeouts(unsigned int* count) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(count, g_wait_timeouts_tc, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_timeouts_tc, &zero, sizeof(unsigned int));
}


}  // namespace
}  // namespace ddg
