// slice_gemm_fused.cu -- the FP64 slice-pair GEMM with the split fused into
// its prologue: the 13-bit parts are formed on the fly from hi/lo tiles of A
// and B, so no part planes are written or read.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2: the parts
// of a double double are formed (step 1), the products of the parts run as
// FP64 matrix products on the tensor cores (steps 2-3, eqs. (1)-(5)), and the
// parts of the product are added back (steps 4-5).  The page forms the parts
// before the products; "Ozaki 2.5: Engineering the Deconstruction Path of
// fp64-Emulated Dense Matrix Multiplication on FP8 Tensor Cores" (summary)
// pipelines the conversion behind the matrix products.  On GB300 the FP64
// pipe (which runs mma.sync f64) is the narrowest unit, while the integer
// pipes and the memory system have room to spare: forming 8 parts of 512
// elements per k-chunk costs about 500 issue cycles per block against about
// 170,000 cycles of FP64 MMAs on the same chunk.  The parts of an element of
// A are formed once per column tile of B that uses it (N / 32 times), those
// of B once per row tile of A -- 16 bytes of hi/lo read where the planes
// cost 64 bytes of parts.
//
// Mapping (one 128-thread block per 32 x 32 tile of P and k-split, the tile
// order of the plane-reading kernel):
//  * two shared-memory stages of 8 part blocks each for A and B (the
//    [part][k4][row][k % 4] layout of the part planes, so the MMA loop is the
//    plane-reading kernel's);
//  * while the warps multiply one stage, every thread holds the hi/lo of the
//    next k-chunk in registers (2 elements of A and 2 of B), loaded a whole
//    chunk of MMAs earlier, and then writes their parts into the other stage;
//  * each thread keeps the exponents of its row of A and its column of B.
// No thread waits on anything but the block's own barrier.
#include <atomic>
#include <algorithm>

#include "common.cuh"
#include "digits.cuh"
#include "launch.cuh"
#include "slice_mma.cuh"

namespace ddg {
namespace {

constexpr int THREADS = 128;
constexpr int STAGE_DOUBLES = 2 * CHUNK_DOUBLES;  // A parts + B parts of one k-chunk: 32 KB
constexpr size_t SMEM_BYTES = 2 * STAGE_DOUBLES * sizeof(double);

static_assert(THREADS * 2 == TM * BK && THREADS * 2 == TN * BK, "two elements of A and two of B per thread");

// The hi/lo of one k-chunk a thread converts: A elements (row ar, k ak and
// ak + 1) and B elements (k bk and bk + 1, column bc), zero outside the matrix.
struct Pending {
    double ah[2], al[2], bh[2], bl[2];
};

__device__ __forceinline__ void load_chunk(const FusedSrc& g, int64_t row, int64_t col, int64_t k0, int ak, int bk,
                                           Pending& p) {
#pragma unroll
    for (int r = 0; r < 2; ++r) p.ah[r] = p.al[r] = p.bh[r] = p.bl[r] = 0.0;
    if (row < g.M && in_bounds(row * g.lda + min(k0 + ak + 1, g.K - 1), (g.M - 1) * g.lda + g.K, kSiteFusedLoadA)) {
        const int64_t k = k0 + ak;
        const double* ph = g.A_hi + row * g.lda + k;
        const double* pl = g.A_lo + row * g.lda + k;
        if (g.a_vec && k + 1 < g.K) {
            const double2 h = __ldg(reinterpret_cast<const double2*>(ph));
            const double2 l = __ldg(reinterpret_cast<const double2*>(pl));
            p.ah[0] = h.x; p.ah[1] = h.y; p.al[0] = l.x; p.al[1] = l.y;
        } else {
#pragma unroll
            for (int r = 0; r < 2; ++r)
                if (k + r < g.K) { p.ah[r] = __ldg(ph + r); p.al[r] = __ldg(pl + r); }
        }
    }
    if (col < g.N && in_bounds(min(k0 + bk + 1, g.K - 1) * g.ldb + col, (g.K - 1) * g.ldb + g.N, kSiteFusedLoadB)) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int64_t k = k0 + bk + r;
            if (k < g.K) {
                p.bh[r] = __ldg(g.B_hi + k * g.ldb + col);
                p.bl[r] = __ldg(g.B_lo + k * g.ldb + col);
            }
        }
    }
}

// The parts of the pending elements into a stage: part s of element (row i,
// k) of the tile at [s][k / 4][i][k % 4]; both elements of a thread share
// k / 4 and sit side by side (k % 4 in {0, 1} or {2, 3}).
__device__ __forceinline__ void store_parts(double* stage, const Pending& p, int ea, int fb, int ar, int ak, int bc,
                                            int bk) {
    double* As = stage;
    double* Bs = stage + CHUNK_DOUBLES;
    {
        double d0[S], d1[S];
        split_digits(p.ah[0], p.al[0], ea, d0);
        split_digits(p.ah[1], p.al[1], ea, d1);
#pragma unroll
        for (int s = 0; s < S; ++s)
            *reinterpret_cast<double2*>(As + ((s * (BK / 4) + ak / 4) * TM + ar) * 4 + ak % 4) = make_double2(d0[s], d1[s]);
    }
    {
        double d0[S], d1[S];
        split_digits(p.bh[0], p.bl[0], fb, d0);
        split_digits(p.bh[1], p.bl[1], fb, d1);
#pragma unroll
        for (int s = 0; s < S; ++s)
            *reinterpret_cast<double2*>(Bs + ((s * (BK / 4) + bk / 4) * TN + bc) * 4 + bk % 4) = make_double2(d0[s], d1[s]);
    }
}

template <bool RECOMBINE>
__global__ void __launch_bounds__(THREADS, 2) slice_gemm_fused_kernel(FusedSrc g, int64_t KC, int splits,
                                                                      TileOut out) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(128) double smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t mt, nt;
    tile_of(blockIdx.x, out.Mp / TM, out.Np / TN, mt, nt);
    const int z = blockIdx.y;
    const int64_t kc0 = (int64_t)z * KC / splits, kc1 = (int64_t)(z + 1) * KC / splits;
    const int nk = (int)(kc1 - kc0);

    // element assignment: A row ar, k ak..ak+1 (4 threads per row, 64
    // contiguous bytes of hi and of lo); B column bc, k bk..bk+1, a warp
    // covering 16 columns at two k (128 contiguous bytes of a row of B per
    // load) so that its part stores fill 512 contiguous bytes of the stage
    const int ar = tid >> 2, ak = (tid & 3) * 2;
    const int bc = 16 * (warp & 1) + (lane & 15), bk = 4 * (warp >> 1) + 2 * (lane >> 4);
    const int64_t row = mt * TM + ar, col = nt * TN + bc;
    const int ea = row < g.M && in_bounds(row, g.M, kSiteFusedExp) ? effective_exponent(g.e[row]) : 0;
    const int fb = col < g.N && in_bounds(col, g.N, kSiteFusedExp) ? effective_exponent(g.f[col]) : 0;

    const int mq = warp >> 1, nq = warp & 1;
    double acc[S][2][2][2];
#pragma unroll
    for (int d = 0; d < S; ++d)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[d][i][j][0] = acc[d][i][j][1] = 0.0;

    Pending p;
    if (nk > 0) {
        load_chunk(g, row, col, kc0 * BK, ak, bk, p);
        store_parts(smem, p, ea, fb, ar, ak, bc, bk);
        if (nk > 1) load_chunk(g, row, col, (kc0 + 1) * BK, ak, bk, p);
    }
    __syncthreads();
    for (int it = 0; it < nk; ++it) {
        const double* stage = smem + (it & 1) * STAGE_DOUBLES;
        chunk_products(stage, stage + CHUNK_DOUBLES, lane, mq, nq, acc);
        if (it + 1 < nk) {
            // the other stage was last read in iteration it - 1, which every
            // thread finished before the barrier that ended it
            store_parts(smem + ((it + 1) & 1) * STAGE_DOUBLES, p, ea, fb, ar, ak, bc, bk);
            if (it + 2 < nk) load_chunk(g, row, col, (kc0 + it + 2) * BK, ak, bk, p);
        }
        __syncthreads();
    }
    store_tile<RECOMBINE>(acc, out, lane, mq, nq, mt, nt, z);
}

template <bool RECOMBINE>
cudaError_t launch_fused(const FusedSrc& g, int64_t Mp, int64_t Np, int64_t Kp, int splits, const TileOut& out,
                         cudaStream_t st) {
    if (Mp == 0 || Np == 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(slice_gemm_fused_kernel<RECOMBINE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)((Mp / TM) * (Np / TN)), (unsigned)splits);
    return launch_pdl(slice_gemm_fused_kernel<RECOMBINE>, grid, dim3(THREADS), SMEM_BYTES, st, g, Kp / BK, splits, out);
}

}  // namespace

FusedSrc make_fused_src(const double* A_hi, const double* A_lo, int64_t lda, const double* B_hi, const double* B_lo,
                        int64_t ldb, const int32_t* e, const int32_t* f, int64_t M, int64_t N, int64_t K) {
    FusedSrc g{};
    g.A_hi = A_hi; g.A_lo = A_lo; g.lda = lda;
    g.B_hi = B_hi; g.B_lo = B_lo; g.ldb = ldb;
    g.e = e; g.f = f;
    g.M = M; g.N = N; g.K = K;
    g.a_vec = (uintptr_t)A_hi % 16 == 0 && (uintptr_t)A_lo % 16 == 0 && lda % 2 == 0;
    return g;
}

cudaError_t launch_slice_gemm_fused(const FusedSrc& g, int64_t Mp, int64_t Np, int64_t Kp, int splits, double* P,
                                    cudaStream_t st) {
    TileOut out{};
    out.P = P;
    out.Mp = Mp;
    out.Np = Np;
    out.p_extent = (int64_t)splits * S * Mp * Np;
    return launch_fused<false>(g, Mp, Np, Kp, splits, out, st);
}

cudaError_t launch_slice_gemm_fused_recombine(const FusedSrc& g, int64_t Mp, int64_t Np, int64_t Kp,
                                              double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st) {
    const TileOut out = recombine_out(Mp, Np, g.e, g.f, g.M, g.N, C_hi, C_lo, ldc);
    return launch_fused<true>(g, Mp, Np, Kp, 1, out, st);
}

DDG_DEFINE_CHECK_READER(check_record_fused)

int slice_gemm_fused_ctas_per_sm() {
    static std::atomic<int> cached{0};  // per-SM count of this kernel (the same on every device)
    if (const int c = cached.load(std::memory_order_relaxed); c > 0) return c;
    int n = 0;
    if (cudaFuncSetAttribute(slice_gemm_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, slice_gemm_fused_kernel<false>, THREADS, SMEM_BYTES) !=
            cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return 1;
    }
    cached.store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace ddg
