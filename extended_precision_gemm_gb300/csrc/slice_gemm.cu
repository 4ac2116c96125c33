// slice_gemm.cu -- step 2 of the dd GEMM: the slice-pair products on the FP64
// tensor pipe.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", eqs. (1)-(4): the
// product of two double doubles split into 8 parts each is a convolution of
// the part sequences; part d of the product collects the pairs s + t = d.
// With the pairs of index sum >= 8 dropped this is 36 FP64 matrix products,
//     P_d = sum_{s+t=d} A_s B_t,   d = 0..7,
// and, because the parts are integers below 2^13 on a shared grid, every
// partial sum is an integer below 2^53 (K <= 2^24): the FP64 tensor cores
// compute them exactly and in any order (the argument of eq. (5)).
//
// GB300 mapping:
//  * one 128-thread block per 32x32 tile of P (all 8 index sums) and k-split,
//    tiles walked in groups of 16 tile rows so resident blocks share operands;
//  * operands arrive by bulk asynchronous copies (TMA engine, no tensor map
//    needed: the part planes are stored tile-contiguous) into a 3-stage
//    shared-memory ring, one mbarrier per stage; 16 KB of A and 16 KB of B
//    parts per stage;
//  * each of the four warps owns a 16x16 quadrant of the tile and issues all
//    36 pairs for it (4 m8n8 blocks x 8 index sums = 32 accumulators); all
//    warps run one instruction stream, which keeps the unrolled loop small
//    enough for the instruction cache;
//  * mma.sync.m8n8k4.f64 fragments are read straight from the stage: the
//    layout [part][k4][row][k%4] makes each fragment 32 consecutive doubles.
// Every wait on an mbarrier is bounded in time; a block that gives up counts
// itself in a device counter (see dd_wait_timeouts) and stops.
#include <atomic>
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "slice_mma.cuh"

namespace ddg {
namespace {

constexpr int THREADS = 128;
constexpr int STAGES = 3;
constexpr int STAGE_DOUBLES = 2 * CHUNK_DOUBLES;            // A block + B block
constexpr uint32_t COPY_BYTES = CHUNK_DOUBLES * sizeof(double);  // 16 KB per operand
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_DOUBLES * sizeof(double) + 64;
constexpr unsigned long long WAIT_BUDGET_NS = 2000000000ULL;  // 2 s per wait

static_assert(COPY_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");

__device__ unsigned int g_wait_timeouts = 0;

// Post the expected byte count on the stage barrier and start the two bulk
// copies (A block, B block) that complete it.  offA / offB are the blocks'
// offsets in their planes (checked against extA / extB in the checked build;
// a block out of bounds is not copied and the barrier completes without it).
__device__ __forceinline__ void issue_stage(uint32_t bar, double* dst, const double* planesA, int64_t offA,
                                            int64_t extA, const double* planesB, int64_t offB, int64_t extB) {
    if (!in_bounds(offA + CHUNK_DOUBLES - 1, extA, kSiteGemmCopyA) ||
        !in_bounds(offB + CHUNK_DOUBLES - 1, extB, kSiteGemmCopyB)) {
        mbar_arrive(bar);
        return;
    }
    mbar_expect_tx(bar, 2u * COPY_BYTES);
    bulk_load(dst, planesA + offA, COPY_BYTES, bar);
    bulk_load(dst + CHUNK_DOUBLES, planesB + offB, COPY_BYTES, bar);
}

template <bool RECOMBINE>
__global__ void __launch_bounds__(THREADS, 2)
    slice_gemm_kernel(const double* __restrict__ planesA, const double* __restrict__ planesB,
                      int64_t KC, int splits, TileOut out) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(128) double smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_DOUBLES);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t mt, nt;
    tile_of(blockIdx.x, out.Mp / TM, out.Np / TN, mt, nt);
    const int z = blockIdx.y;
    const int64_t kc0 = (int64_t)z * KC / splits, kc1 = (int64_t)(z + 1) * KC / splits;
    const int nk = (int)(kc1 - kc0);
    const int64_t offA = (mt * KC + kc0) * CHUNK_DOUBLES, offB = (nt * KC + kc0) * CHUNK_DOUBLES;
    const int64_t extA = (out.Mp / TM) * KC * CHUNK_DOUBLES, extB = (out.Np / TN) * KC * CHUNK_DOUBLES;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < STAGES && i < nk; ++i)
            issue_stage(smem_addr(&bars[i]), smem + i * STAGE_DOUBLES, planesA, offA + (int64_t)i * CHUNK_DOUBLES,
                        extA, planesB, offB + (int64_t)i * CHUNK_DOUBLES, extB);

    const int mq = warp >> 1, nq = warp & 1;
    double acc[S][2][2][2];
#pragma unroll
    for (int d = 0; d < S; ++d)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[d][i][j][0] = acc[d][i][j][1] = 0.0;

    for (int it = 0; it < nk; ++it) {
        const int st = it % STAGES;
        const uint32_t parity = (uint32_t)(it / STAGES) & 1u;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[st]), parity, WAIT_BUDGET_NS);
        // Every thread has finished chunk it-1 once past this barrier, so its
        // stage can be refilled; all threads agree on whether the wait failed.
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                atomicAdd(&g_wait_timeouts, 1u);
                // Let the copies still in flight land before the block exits.
                const int issued = min(nk, max(it - 1, 0) + STAGES);
                for (int j = it; j < issued; ++j)
                    mbar_wait_bounded(smem_addr(&bars[j % STAGES]), (uint32_t)(j / STAGES) & 1u,
                                      WAIT_BUDGET_NS);
            }
            return;
        }
        if (tid == 0 && it >= 1 && it - 1 + STAGES < nk) {
            const int nxt = it - 1 + STAGES, ns = (it - 1) % STAGES;
            issue_stage(smem_addr(&bars[ns]), smem + ns * STAGE_DOUBLES, planesA,
                        offA + (int64_t)nxt * CHUNK_DOUBLES, extA, planesB, offB + (int64_t)nxt * CHUNK_DOUBLES, extB);
        }
        const double* As = smem + st * STAGE_DOUBLES;
        chunk_products(As, As + CHUNK_DOUBLES, lane, mq, nq, acc);
    }

    store_tile<RECOMBINE>(acc, out, lane, mq, nq, mt, nt, z);
}

// Register-only throughput loop of the same mma.sync.m8n8k4.f64 instruction:
// four independent accumulator chains per warp.  Measures the FP64 tensor
// pipe's rate on this device (the roof of the slice GEMM).
__global__ void __launch_bounds__(128) dmma_roof_kernel(double* out, int iters) {
    const int lane = threadIdx.x & 31;
    double a = 1.0 + lane * 0x1p-10, b = 1.0 - lane * 0x1p-10;
    double c[4][2] = {{0, 0}, {0, 0}, {0, 0}, {0, 0}};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 4; ++i) dmma(c[i][0], c[i][1], a, b);
    }
    out[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = c[0][0] + c[1][1] + c[2][0] + c[3][1];
}

}  // namespace

cudaError_t measure_dmma_roof(double* tflops, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const int blocks = sms * 4, threads = 128, iters = 4096;
    double* out = nullptr;
    err = cudaMallocAsync(&out, (size_t)blocks * threads * sizeof(double), st);
    if (err != cudaSuccess) return err;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    dmma_roof_kernel<<<blocks, threads, 0, st>>>(out, iters);  // warm-up
    cudaEventRecord(e0, st);
    for (int r = 0; r < 5; ++r) dmma_roof_kernel<<<blocks, threads, 0, st>>>(out, iters);
    cudaEventRecord(e1, st);
    err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFreeAsync(out, st);
    if (err != cudaSuccess) return err;
    const double flops = 5.0 * blocks * (threads / 32) * (double)iters * 4 * (2.0 * 8 * 8 * 4);
    *tflops = flops / (ms * 1e-3) / 1e12;
    return cudaGetLastError();
}

int slice_gemm_ctas_per_sm() {
    static std::atomic<int> cached{0};  // per-SM count of this kernel (the same on every device)
    if (const int c = cached.load(std::memory_order_relaxed); c > 0) return c;
    int n = 0;
    if (cudaFuncSetAttribute(slice_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, slice_gemm_kernel<false>, THREADS, SMEM_BYTES) !=
            cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return 1;
    }
    cached.store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_slice_gemm(const double* planesA, const double* planesB, int64_t Mp,
                              int64_t Np, int64_t Kp, int splits, double* P, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(slice_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    TileOut out{};
    out.P = P;
    out.Mp = Mp;
    out.Np = Np;
    out.p_extent = (int64_t)splits * S * Mp * Np;
    dim3 grid((unsigned)((Mp / TM) * (Np / TN)), (unsigned)splits);
    return launch_pdl(slice_gemm_kernel<false>, grid, dim3(THREADS), SMEM_BYTES, st, planesA, planesB, Kp / BK, splits,
                      out);
}

cudaError_t launch_slice_gemm_recombine(const double* planesA, const double* planesB, int64_t Mp, int64_t Np,
                                        int64_t Kp, const int32_t* e, const int32_t* f, int64_t M, int64_t N,
                                        double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(slice_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const TileOut out = recombine_out(Mp, Np, e, f, M, N, C_hi, C_lo, ldc);
    dim3 grid((unsigned)((Mp / TM) * (Np / TN)), 1u);
    return launch_pdl(slice_gemm_kernel<true>, grid, dim3(THREADS), SMEM_BYTES, st, planesA, planesB, Kp / BK, 1, out);
}

cudaError_t peek_wait_timeouts(unsigned int* count, cudaStream_t st) {
    cudaError_t err = cudaMemcpyFromSymbolAsync(count, g_wait_timeouts, sizeof(unsigned int), 0,
                                                cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    return err;
}

DDG_DEFINE_CHECK_READER(check_record_slice_gemm)

cudaError_t read_and_reset_wait_timeouts(unsigned int* count) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace ddg
