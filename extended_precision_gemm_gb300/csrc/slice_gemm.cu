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
//  * one 128-thread block per 32x32 tile of P (all 8 index sums) and k-split;
//  * operands arrive by bulk asynchronous copies (TMA engine, no tensor map
//    needed: the part planes are stored tile-contiguous) into a 3-stage
//    shared-memory ring, one mbarrier per stage; 16 KB of A and 16 KB of B
//    parts per stage;
//  * the four warps share the 36 pairs evenly: warp w owns index sums w and
//    7 - w, i.e. (w + 1) + (8 - w) = 9 pairs, over the whole 32x32 tile
//    (16 m8n8 accumulator tiles per index sum);
//  * mma.sync.m8n8k4.f64 fragments are read straight from the stage: the
//    layout [part][k4][row][k%4] makes each fragment 32 consecutive doubles.
// Every wait on an mbarrier is bounded in time; a block that gives up counts
// itself in a device counter (see dd_wait_timeouts) and stops.
#include <algorithm>

#include "common.cuh"
#include "launch.cuh"

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

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of the barrier to complete, for at most `budget` ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long budget) {
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > budget) return false;
    }
}

// Post the expected byte count on the stage barrier and start the two bulk
// copies (A block, B block) that complete it.
__device__ __forceinline__ void issue_stage(uint32_t bar, double* dst, const double* srcA,
                                            const double* srcB) {
    asm volatile(
        "{\n"
        " .reg .b64 st;\n"
        " mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n"
        "}\n" ::"r"(bar),
        "r"(2u * COPY_BYTES)
        : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(srcA), "r"(COPY_BYTES), "r"(bar)
        : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst + CHUNK_DOUBLES)),
        "l"(srcB), "r"(COPY_BYTES), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void dmma(double& c0, double& c1, double a, double b) {
    asm("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0,%1}, {%2}, {%3}, {%0,%1};"
        : "+d"(c0), "+d"(c1)
        : "d"(a), "d"(b));
}

// One k-chunk (8 values of k) of the pairs owned by warp W: index sums W and
// 7 - W.  acc[g][mb][nb][2]: g = 0 for index sum W, 1 for 7 - W.
template <int W>
__device__ __forceinline__ void chunk_products(const double* __restrict__ As,
                                               const double* __restrict__ Bs, int lane,
                                               double (&acc)[2][4][4][2]) {
#pragma unroll
    for (int q = 0; q < BK / 4; ++q) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            constexpr int D0 = W, D1 = S - 1 - W;
            if (s > D1) continue;  // no pair of this warp uses A_s
            double a[4];
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) a[mb] = As[((s * (BK / 4) + q) * TM + mb * 8) * 4 + lane];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int t = (g == 0 ? D0 : D1) - s;
                if (t < 0) continue;
                double b[4];
#pragma unroll
                for (int nb = 0; nb < 4; ++nb) b[nb] = Bs[((t * (BK / 4) + q) * TN + nb * 8) * 4 + lane];
#pragma unroll
                for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb) dmma(acc[g][mb][nb][0], acc[g][mb][nb][1], a[mb], b[nb]);
            }
        }
    }
}

__global__ void __launch_bounds__(THREADS, 2)
    slice_gemm_kernel(const double* __restrict__ planesA, const double* __restrict__ planesB,
                      int64_t KC, int splits, double* __restrict__ P, int64_t Mp, int64_t Np) {
    extern __shared__ __align__(128) double smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_DOUBLES);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nt = blockIdx.x, mt = blockIdx.y;
    const int z = blockIdx.z;
    const int64_t kc0 = (int64_t)z * KC / splits, kc1 = (int64_t)(z + 1) * KC / splits;
    const int nk = (int)(kc1 - kc0);
    const double* srcA = planesA + (mt * KC + kc0) * CHUNK_DOUBLES;
    const double* srcB = planesB + (nt * KC + kc0) * CHUNK_DOUBLES;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < STAGES && i < nk; ++i)
            issue_stage(smem_addr(&bars[i]), smem + i * STAGE_DOUBLES, srcA + (int64_t)i * CHUNK_DOUBLES,
                        srcB + (int64_t)i * CHUNK_DOUBLES);

    double acc[2][4][4][2];
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int mb = 0; mb < 4; ++mb)
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) acc[g][mb][nb][0] = acc[g][mb][nb][1] = 0.0;

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
            issue_stage(smem_addr(&bars[ns]), smem + ns * STAGE_DOUBLES,
                        srcA + (int64_t)nxt * CHUNK_DOUBLES, srcB + (int64_t)nxt * CHUNK_DOUBLES);
        }
        const double* As = smem + st * STAGE_DOUBLES;
        const double* Bs = As + CHUNK_DOUBLES;
        switch (warp) {
            case 0: chunk_products<0>(As, Bs, lane, acc); break;
            case 1: chunk_products<1>(As, Bs, lane, acc); break;
            case 2: chunk_products<2>(As, Bs, lane, acc); break;
            default: chunk_products<3>(As, Bs, lane, acc); break;
        }
    }

    // Epilogue: thread (lane) holds rows mb*8 + lane/4, columns nb*8 + 2(lane%4) + {0,1}.
    const int64_t plane = Mp * Np;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int d = (g == 0) ? warp : S - 1 - warp;
        double* out = P + ((int64_t)z * S + d) * plane;
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
            const int64_t row = mt * TM + mb * 8 + (lane >> 2);
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                const int64_t col = nt * TN + nb * 8 + 2 * (lane & 3);
                *reinterpret_cast<double2*>(out + row * Np + col) =
                    make_double2(acc[g][mb][nb][0], acc[g][mb][nb][1]);
            }
        }
    }
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
    static int cached = 0;
    if (cached > 0) return cached;
    int n = 0;
    if (cudaFuncSetAttribute(slice_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, slice_gemm_kernel, THREADS, SMEM_BYTES) !=
            cudaSuccess ||
        n <= 0)
        return 1;
    cached = n;
    return n;
}

cudaError_t launch_slice_gemm(const double* planesA, const double* planesB, int64_t Mp,
                              int64_t Np, int64_t Kp, int splits, double* P, cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(slice_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)(Np / TN), (unsigned)(Mp / TM), (unsigned)splits);
    slice_gemm_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(planesA, planesB, Kp / BK, splits, P, Mp, Np);
    return cudaGetLastError();
}

cudaError_t read_and_reset_wait_timeouts(unsigned int* count) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace ddg
