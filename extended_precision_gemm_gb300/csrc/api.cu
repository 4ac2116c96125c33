// api.cu -- the C ABI of the dd GEMM library (declarations in ddgemm.h).
//
// Argument checking, the workspace layout, and the launch sequence of the
// three steps: split (exponents + part planes), slice-pair GEMM, recombine.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "launch.cuh"

using namespace ddg;

namespace {

constexpr int64_t kAlign = 256;
constexpr int kMaxSplits = 64;
constexpr int64_t kMaxTiles = 0x7FFFFFFF;  // output tiles (grid.x of the FP64 and integer slice GEMMs)

struct Layout {
    int64_t Mp, Np, Kp, KC;
    int splits;
    // byte offsets inside the workspace
    int64_t off_e, off_f, off_A, off_B, off_P, total;
};

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 152;
    return sms;
}

// Which slice GEMM a layout is for: FP64 parts for mma.sync f64, or int16
// parts for the integer pipe.
enum class Engine { kFp64Tensor, kInt64Pipe, kQuadInt64 };

// k-split of the slice GEMM: the smallest split count whose waves of blocks
// fill the GPU best (tiles * splits over whole waves of resident blocks),
// keeping at least 4 k-chunks per split.
int choose_splits(int64_t Mp, int64_t Np, int64_t KC, Engine eng) {
    const int64_t tiles = (Mp / TM) * (Np / TN);
    if (tiles == 0 || KC <= 1) return 1;
    const int per_sm = eng == Engine::kFp64Tensor ? slice_gemm_ctas_per_sm()
                       : eng == Engine::kInt64Pipe ? slice_gemm_i64_ctas_per_sm()
                                                   : slice_gemm_qd_ctas_per_sm();
    const int64_t slots = (int64_t)device_sms() * per_sm;
    // blocks per 32 x 32 tile: the integer kernels take half / quarter tiles
    const int64_t blocks_per_tile = eng == Engine::kFp64Tensor ? 1 : eng == Engine::kInt64Pipe ? 2 : 4;
    int best = 1;
    double best_score = -1.0;
    const int64_t max_s = std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, KC / 4));
    for (int64_t s = 1; s <= max_s; ++s) {
        const int64_t blocks = tiles * blocks_per_tile * s;
        const int64_t waves = (blocks + slots - 1) / slots;
        const double eff = (double)blocks / (double)(waves * slots);
        const double score = eff - 0.002 * (double)s;
        if (score > best_score + 1e-12) { best_score = score; best = (int)s; }
    }
    return best;
}

Layout make_layout(int64_t M, int64_t N, int64_t K, Engine eng = Engine::kFp64Tensor) {
    Layout L;
    L.Mp = round_up(M, TM);
    L.Np = round_up(N, TN);
    L.Kp = round_up(K, BK);
    L.KC = L.Kp / BK;
    L.splits = choose_splits(L.Mp, L.Np, L.KC, eng);
    const int64_t part_bytes = eng == Engine::kFp64Tensor ? 8 : 2;
    const int64_t parts = eng == Engine::kQuadInt64 ? 16 : S;
    int64_t off = 0;
    auto take = [&](int64_t bytes) { int64_t o = off; off = round_up(off + bytes, kAlign); return o; };
    L.off_e = take(L.Mp * 4);
    L.off_f = take(L.Np * 4);
    L.off_A = take(parts * L.Mp * L.Kp * part_bytes);
    L.off_B = take(parts * L.Np * L.Kp * part_bytes);
    L.off_P = take((int64_t)L.splits * parts * L.Mp * L.Np * 8);
    L.total = off;
    return L;
}

bool ranges_overlap(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    if (a == nullptr || b == nullptr || abytes <= 0 || bbytes <= 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// Bytes spanned by a rows x cols row-major matrix with leading dimension ld.
int64_t span_bytes(int64_t rows, int64_t cols, int64_t ld) {
    if (rows == 0 || cols == 0) return 0;
    return ((rows - 1) * ld + cols) * 8;
}

ddgemm_status check_shapes(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((round_up(M, TM) / TM) * (round_up(N, TN) / TN) > kMaxTiles) return DDGEMM_ERR_UNSUPPORTED;
    return DDGEMM_OK;
}

ddgemm_status check_gemm_args(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                              int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb,
                              const double* C_hi, const double* C_lo, int64_t ldc) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;  // empty product: no pointer is read
    if (C_hi == nullptr || C_lo == nullptr) return DDGEMM_ERR_INVALID_ARG;
    if (M > 0 && K > 0 && (A_hi == nullptr || A_lo == nullptr)) return DDGEMM_ERR_INVALID_ARG;
    if (N > 0 && K > 0 && (B_hi == nullptr || B_lo == nullptr)) return DDGEMM_ERR_INVALID_ARG;
    const int64_t a = span_bytes(M, K, lda), b = span_bytes(K, N, ldb), c = span_bytes(M, N, ldc);
    const void* ins[4] = {A_hi, A_lo, B_hi, B_lo};
    const int64_t insz[4] = {a, a, b, b};
    const void* outs[2] = {C_hi, C_lo};
    for (int o = 0; o < 2; ++o) {
        for (int i = 0; i < 4; ++i)
            if (ranges_overlap(outs[o], c, ins[i], insz[i])) return DDGEMM_ERR_INVALID_ARG;
    }
    if (ranges_overlap(C_hi, c, C_lo, c)) return DDGEMM_ERR_INVALID_ARG;
    return DDGEMM_OK;
}

ddgemm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DDGEMM_OK : DDGEMM_ERR_CUDA; }

#define DDG_TRY(call)                                   \
    do {                                                \
        cudaError_t err_ = (call);                      \
        if (err_ != cudaSuccess) return DDGEMM_ERR_CUDA; \
    } while (0)

// An NVTX range around the launches of one step of a product ("dd/split",
// "dd/slice_gemm", ...), so that a profiler can attribute and filter the
// kernels by step (e.g. ncu --nvtx --nvtx-include "dd/slice_gemm/").  The
// ranges cost nothing unless a tool is attached.
struct StepRange {
    explicit StepRange(const char* name) { nvtxRangePushA(name); }
    ~StepRange() { nvtxRangePop(); }
    StepRange(const StepRange&) = delete;
    StepRange& operator=(const StepRange&) = delete;
};

#define DDG_STEP(name, call)        \
    do {                            \
        StepRange range_(name);     \
        DDG_TRY(call);              \
    } while (0)

// Step 1 for any subset of the operands (null hi = operand absent): exponent
// reset, exponents, split into FP64 or int16 part planes -- three launches.
cudaError_t run_split(int64_t M, int64_t N, int64_t K, int64_t Kp, const double* A_hi, const double* A_lo,
                      int64_t lda, int32_t* e, void* pA, const double* B_hi, const double* B_lo, int64_t ldb,
                      int32_t* f, void* pB, bool i16, cudaStream_t st) {
    SplitOperand a{A_hi, A_lo, lda, M, e}, b{B_hi, B_lo, ldb, N, f};
    const SplitOperand* pa = (e != nullptr && M > 0) ? &a : nullptr;
    const SplitOperand* pb = (f != nullptr && N > 0) ? &b : nullptr;
    cudaError_t err = launch_shared_exponents(pa, pb, K, 0, st);
    if (err == cudaSuccess)
        err = i16 ? launch_split_i16(pa, pb, K, Kp, static_cast<int16_t*>(pA), static_cast<int16_t*>(pB), st)
                  : launch_split_f64(pa, pb, K, Kp, static_cast<double*>(pA), static_cast<double*>(pB), st);
    return err;
}

// The launch sequence on a workspace laid out by make_layout.
ddgemm_status run_gemm(const Layout& L, int64_t M, int64_t N, int64_t K, const double* A_hi,
                       const double* A_lo, int64_t lda, const double* B_hi, const double* B_lo,
                       int64_t ldb, double* C_hi, double* C_lo, int64_t ldc, char* ws,
                       cudaStream_t st) {
    if (M == 0 || N == 0) return DDGEMM_OK;
    int32_t* e = reinterpret_cast<int32_t*>(ws + L.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + L.off_f);
    double* pA = reinterpret_cast<double*>(ws + L.off_A);
    double* pB = reinterpret_cast<double*>(ws + L.off_B);
    double* P = reinterpret_cast<double*>(ws + L.off_P);
    DDG_STEP("dd/split", run_split(M, N, K, L.Kp, A_hi, A_lo, lda, e, pA, B_hi, B_lo, ldb, f, pB, false, st));
    DDG_STEP("dd/slice_gemm", launch_slice_gemm(pA, pB, L.Mp, L.Np, L.Kp, L.splits, P, st));
    DDG_STEP("dd/recombine", launch_recombine(P, L.splits, L.Mp, L.Np, e, f, M, N, C_hi, C_lo, ldc, st));
    return DDGEMM_OK;
}

// The launch sequence of the integer-pipe variant (int16 parts, int64 sums).
ddgemm_status run_gemm_i64(const Layout& L, int64_t M, int64_t N, int64_t K, const double* A_hi,
                           const double* A_lo, int64_t lda, const double* B_hi, const double* B_lo,
                           int64_t ldb, double* C_hi, double* C_lo, int64_t ldc, char* ws,
                           cudaStream_t st) {
    if (M == 0 || N == 0) return DDGEMM_OK;
    int32_t* e = reinterpret_cast<int32_t*>(ws + L.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + L.off_f);
    int16_t* pA = reinterpret_cast<int16_t*>(ws + L.off_A);
    int16_t* pB = reinterpret_cast<int16_t*>(ws + L.off_B);
    double* P = reinterpret_cast<double*>(ws + L.off_P);
    DDG_STEP("dd_i64/split", run_split(M, N, K, L.Kp, A_hi, A_lo, lda, e, pA, B_hi, B_lo, ldb, f, pB, true, st));
    DDG_STEP("dd_i64/slice_gemm", launch_slice_gemm_i64(pA, pB, L.Mp, L.Np, L.Kp, L.splits, P, st));
    DDG_STEP("dd_i64/recombine", launch_recombine(P, L.splits, L.Mp, L.Np, e, f, M, N, C_hi, C_lo, ldc, st));
    return DDGEMM_OK;
}

// A product with HOST operands and result: one stream-ordered device block
// holds A_hi, A_lo (M x K dense), B_hi, B_lo (K x N), C_hi, C_lo (M x N) and
// `ws_bytes` of workspace; the operands are copied in, `run` launches the
// product on the dense device copies, C is copied back, the block is freed,
// and the stream is synchronised before returning.
// The library's stream-ordered memory pool on the current device, from which
// every entry point that is not given a workspace (and the host-buffer
// entry points, for their device copies) allocates: created on first use
// with no release threshold, so the memory of one call stays in the pool for
// the next instead of being unmapped at every synchronisation and mapped
// again (mapping the 1.7 GB workspace of a 4096^3 bf16 product costs more
// than 10% of the product).  dd_pool_trim gives it back.
constexpr int kMaxPoolDevices = 64;
std::mutex g_pool_mutex;
cudaMemPool_t g_pool[kMaxPoolDevices] = {};

cudaError_t library_pool(cudaMemPool_t* pool, bool create) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxPoolDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (g_pool[dev] == nullptr && create) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        err = cudaMemPoolCreate(&p, &props);
        if (err != cudaSuccess) return err;
        uint64_t keep = ~0ULL;
        err = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        if (err != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return err;
        }
        g_pool[dev] = p;
    }
    *pool = g_pool[dev];
    return cudaSuccess;
}

// Stream-ordered allocation from the library's pool (cudaFreeAsync returns it).
cudaError_t pool_alloc(void** ptr, size_t bytes, cudaStream_t st) {
    cudaMemPool_t pool = nullptr;
    cudaError_t err = library_pool(&pool, true);
    if (err != cudaSuccess) return err;
    return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

// `peek` reads the slice GEMM's count of bounded waits that gave up: a count
// that grew during the call makes it return DDGEMM_ERR_CUDA.
template <class Run, class Peek>
ddgemm_status host_product(int64_t M, int64_t N, int64_t K, const double* h_A_hi, const double* h_A_lo,
                           int64_t lda, const double* h_B_hi, const double* h_B_lo, int64_t ldb, double* h_C_hi,
                           double* h_C_lo, int64_t ldc, int64_t ws_bytes, cudaStream_t st, Run run, Peek peek) {
    unsigned int timeouts_before = 0;
    if (peek(&timeouts_before, st) != cudaSuccess) return DDGEMM_ERR_CUDA;
    const int64_t a = round_up(M * K * 8, kAlign), b = round_up(K * N * 8, kAlign), c = round_up(M * N * 8, kAlign);
    const int64_t total = 2 * a + 2 * b + 2 * c + ws_bytes;
    char* dev = nullptr;
    if (pool_alloc(reinterpret_cast<void**>(&dev), (size_t)total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    double* dA_hi = reinterpret_cast<double*>(dev);
    double* dA_lo = reinterpret_cast<double*>(dev + a);
    double* dB_hi = reinterpret_cast<double*>(dev + 2 * a);
    double* dB_lo = reinterpret_cast<double*>(dev + 2 * a + b);
    double* dC_hi = reinterpret_cast<double*>(dev + 2 * a + 2 * b);
    double* dC_lo = reinterpret_cast<double*>(dev + 2 * a + 2 * b + c);
    char* ws = dev + 2 * a + 2 * b + 2 * c;
    cudaError_t err = cudaSuccess;
    auto copy_in = [&](double* dst, const double* src, int64_t rows, int64_t cols, int64_t ld) {
        if (err != cudaSuccess || rows == 0 || cols == 0) return;
        err = cudaMemcpy2DAsync(dst, (size_t)cols * 8, src, (size_t)ld * 8, (size_t)cols * 8, (size_t)rows,
                                cudaMemcpyHostToDevice, st);
    };
    copy_in(dA_hi, h_A_hi, M, K, lda);
    copy_in(dA_lo, h_A_lo, M, K, lda);
    copy_in(dB_hi, h_B_hi, K, N, ldb);
    copy_in(dB_lo, h_B_lo, K, N, ldb);
    ddgemm_status s = err == cudaSuccess ? run(dA_hi, dA_lo, dB_hi, dB_lo, dC_hi, dC_lo, ws, st) : DDGEMM_ERR_CUDA;
    if (s == DDGEMM_OK) {
        err = cudaMemcpy2DAsync(h_C_hi, (size_t)ldc * 8, dC_hi, (size_t)N * 8, (size_t)N * 8, (size_t)M,
                                cudaMemcpyDeviceToHost, st);
        if (err == cudaSuccess)
            err = cudaMemcpy2DAsync(h_C_lo, (size_t)ldc * 8, dC_lo, (size_t)N * 8, (size_t)N * 8, (size_t)M,
                                    cudaMemcpyDeviceToHost, st);
        if (err != cudaSuccess) s = DDGEMM_ERR_CUDA;
    }
    cudaError_t fe = cudaFreeAsync(dev, st);
    cudaError_t se = cudaStreamSynchronize(st);
    if (s == DDGEMM_OK && (fe != cudaSuccess || se != cudaSuccess)) s = DDGEMM_ERR_CUDA;
    unsigned int timeouts_after = 0;
    if (s == DDGEMM_OK && (peek(&timeouts_after, st) != cudaSuccess || timeouts_after != timeouts_before))
        s = DDGEMM_ERR_CUDA;
    return s;
}

}  // namespace

extern "C" {

const char* dd_status_string(int status) {
    switch (status) {
        case DDGEMM_OK: return "DDGEMM_OK";
        case DDGEMM_ERR_INVALID_ARG: return "DDGEMM_ERR_INVALID_ARG";
        case DDGEMM_ERR_UNSUPPORTED: return "DDGEMM_ERR_UNSUPPORTED";
        case DDGEMM_ERR_ALLOC: return "DDGEMM_ERR_ALLOC";
        case DDGEMM_ERR_CUDA: return "DDGEMM_ERR_CUDA";
        case DDGEMM_ERR_TOO_LARGE: return "DDGEMM_ERR_TOO_LARGE";
        default: return "DDGEMM_UNKNOWN_STATUS";
    }
}

ddgemm_status dd_gemm_layout(int64_t M, int64_t N, int64_t K, int64_t* Mp, int64_t* Np, int64_t* Kp,
                             int* splits) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    Layout L = make_layout(M, N, K);
    if (Mp) *Mp = L.Mp;
    if (Np) *Np = L.Np;
    if (Kp) *Kp = L.Kp;
    if (splits) *splits = L.splits;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (bytes == nullptr || M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    *bytes = (size_t)make_layout(M, N, K).total;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_ws(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                         int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb,
                         double* C_hi, double* C_lo, int64_t ldc, void* workspace,
                         size_t workspace_bytes, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    Layout L = make_layout(M, N, K);
    if (workspace == nullptr || (uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)L.total)
        return DDGEMM_ERR_INVALID_ARG;
    const int64_t c = span_bytes(M, N, ldc);
    if (ranges_overlap(workspace, L.total, C_hi, c) || ranges_overlap(workspace, L.total, C_lo, c))
        return DDGEMM_ERR_INVALID_ARG;
    return run_gemm(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc,
                    static_cast<char*>(workspace), static_cast<cudaStream_t>(stream));
}

ddgemm_status dd_gemm(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                      int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, double* C_hi,
                      double* C_lo, int64_t ldc, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Layout L = make_layout(M, N, K);
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)L.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_gemm(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status dd_gemm_host(int64_t M, int64_t N, int64_t K, const double* h_A_hi,
                           const double* h_A_lo, int64_t lda, const double* h_B_hi,
                           const double* h_B_lo, int64_t ldb, double* h_C_hi, double* h_C_lo,
                           int64_t ldc, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, h_A_hi, h_A_lo, lda, h_B_hi, h_B_lo, ldb, h_C_hi,
                                      h_C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    Layout L = make_layout(M, N, K);
    return host_product(M, N, K, h_A_hi, h_A_lo, lda, h_B_hi, h_B_lo, ldb, h_C_hi, h_C_lo, ldc, L.total,
                        static_cast<cudaStream_t>(stream),
                        [&](const double* a_hi, const double* a_lo, const double* b_hi, const double* b_lo,
                            double* c_hi, double* c_lo, char* ws, cudaStream_t st) {
                            return run_gemm(L, M, N, K, a_hi, a_lo, std::max<int64_t>(K, 1), b_hi, b_lo, N,
                                            c_hi, c_lo, N, ws, st);
                        },
                        peek_wait_timeouts);
}

ddgemm_status dd_split_rows(int64_t M, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                            double* planes, int32_t* e, void* stream) {
    if (M < 0 || K < 0 || lda < std::max<int64_t>(1, K)) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0) return DDGEMM_OK;
    if (e == nullptr || (K > 0 && (A_hi == nullptr || A_lo == nullptr || planes == nullptr)))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planes % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t Kp = round_up(K, BK);
    DDG_TRY(run_split(M, 0, K, Kp, A_hi, A_lo, lda, e, planes, nullptr, nullptr, 1, nullptr, nullptr, false, st));
    return DDGEMM_OK;
}

ddgemm_status dd_split_cols(int64_t K, int64_t N, const double* B_hi, const double* B_lo, int64_t ldb,
                            double* planes, int32_t* f, void* stream) {
    if (N < 0 || K < 0 || ldb < std::max<int64_t>(1, N)) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (N == 0) return DDGEMM_OK;
    if (f == nullptr || (K > 0 && (B_hi == nullptr || B_lo == nullptr || planes == nullptr)))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planes % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t Kp = round_up(K, BK);
    DDG_TRY(run_split(0, N, K, Kp, nullptr, nullptr, 1, nullptr, nullptr, B_hi, B_lo, ldb, f, planes, false, st));
    return DDGEMM_OK;
}

// Step 1 for both operands in three launches.
static ddgemm_status split_both(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                                int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, void* planesA,
                                int32_t* e, void* planesB, int32_t* f, bool i16, void* stream) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, std::max<int64_t>(1, N));
    if (s != DDGEMM_OK) return s;
    if (M > 0 && (e == nullptr || (K > 0 && (A_hi == nullptr || A_lo == nullptr || planesA == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if (N > 0 && (f == nullptr || (K > 0 && (B_hi == nullptr || B_lo == nullptr || planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Kp = round_up(K, BK);
    return from_cuda(run_split(M, N, K, Kp, A_hi, A_lo, lda, M > 0 ? e : nullptr, planesA, B_hi, B_lo, ldb,
                               N > 0 ? f : nullptr, planesB, i16, static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_split(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                       const double* B_hi, const double* B_lo, int64_t ldb, double* planesA, int32_t* e,
                       double* planesB, int32_t* f, void* stream) {
    return split_both(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, planesA, e, planesB, f, false, stream);
}

ddgemm_status dd_split_i16(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                           const double* B_hi, const double* B_lo, int64_t ldb, int16_t* planesA, int32_t* e,
                           int16_t* planesB, int32_t* f, void* stream) {
    return split_both(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, planesA, e, planesB, f, true, stream);
}

ddgemm_status dd_exponents(int64_t M, int64_t N, int64_t K, const double* A_hi, int64_t lda, const double* B_hi,
                           int64_t ldb, int32_t* e, int32_t* f, void* stream) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, std::max<int64_t>(1, N));
    if (s != DDGEMM_OK) return s;
    if ((M > 0 && (e == nullptr || (K > 0 && A_hi == nullptr))) || (N > 0 && (f == nullptr || (K > 0 && B_hi == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SplitOperand a{A_hi, nullptr, lda, M, e, false}, b{B_hi, nullptr, ldb, N, f, false};
    const SplitOperand* pa = M > 0 ? &a : nullptr;
    const SplitOperand* pb = N > 0 ? &b : nullptr;
    DDG_TRY(launch_shared_exponents(pa, pb, K, EXP_NONE, st));
    return DDGEMM_OK;
}

ddgemm_status dd_split_with_exponents(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                                      int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb,
                                      const int32_t* e, const int32_t* f, double* planesA, double* planesB,
                                      void* stream) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, std::max<int64_t>(1, N));
    if (s != DDGEMM_OK) return s;
    if (M > 0 && (e == nullptr || (K > 0 && (A_hi == nullptr || A_lo == nullptr || planesA == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if (N > 0 && (f == nullptr || (K > 0 && (B_hi == nullptr || B_lo == nullptr || planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    // exp_given: the kernels only read the exponents
    SplitOperand a{A_hi, A_lo, lda, M, const_cast<int32_t*>(e), true};
    SplitOperand b{B_hi, B_lo, ldb, N, const_cast<int32_t*>(f), true};
    return from_cuda(launch_split_f64(M > 0 ? &a : nullptr, N > 0 ? &b : nullptr, K, round_up(K, BK), planesA,
                                      planesB, static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_slice_gemm(int64_t M, int64_t N, int64_t K, const double* planesA,
                            const double* planesB, int splits, double* P, void* stream) {
    ddgemm_status s = check_shapes(M, N, K, std::max<int64_t>(1, K), std::max<int64_t>(1, N),
                                   std::max<int64_t>(1, N));
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, TM), Np = round_up(N, TN), Kp = round_up(K, BK), KC = Kp / BK;
    if (splits < 1 || splits > kMaxSplits || (KC > 0 && splits > KC) || (KC == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (P == nullptr || (K > 0 && (planesA == nullptr || planesB == nullptr))) return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0 || (uintptr_t)P % 16 != 0)
        return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(launch_slice_gemm(planesA, planesB, Mp, Np, Kp, splits, P,
                                       static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_recombine(int64_t M, int64_t N, const double* P, int splits, const int32_t* e,
                           const int32_t* f, double* C_hi, double* C_lo, int64_t ldc, void* stream) {
    if (M < 0 || N < 0 || ldc < std::max<int64_t>(1, N)) return DDGEMM_ERR_INVALID_ARG;
    if (splits < 1 || splits > kMaxSplits) return DDGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (P == nullptr || e == nullptr || f == nullptr || C_hi == nullptr || C_lo == nullptr)
        return DDGEMM_ERR_INVALID_ARG;
    const int64_t Mp = round_up(M, TM), Np = round_up(N, TN);
    return from_cuda(launch_recombine(P, splits, Mp, Np, e, f, M, N, C_hi, C_lo, ldc,
                                      static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_fp64_tensor_roof(double* tflops, void* stream) {
    if (tflops == nullptr) return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(measure_dmma_roof(tflops, static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_wait_timeouts(unsigned int* count) {
    if (count == nullptr) return DDGEMM_ERR_INVALID_ARG;
    unsigned int a = 0, b = 0, c = 0, d = 0;
    ddgemm_status s = from_cuda(read_and_reset_wait_timeouts(&a));
    if (s == DDGEMM_OK) s = from_cuda(read_and_reset_wait_timeouts_i64(&b));
    if (s == DDGEMM_OK) s = from_cuda(read_and_reset_wait_timeouts_qd(&c));
    unsigned int m = 0;
    if (s == DDGEMM_OK) s = from_cuda(read_and_reset_wait_timeouts_tc(&d));
    if (s == DDGEMM_OK) s = from_cuda(read_and_reset_wait_timeouts_tc_md(&m));
    *count = a + b + c + d + m;
    return s;
}

int dd_checked_build(void) {
#ifdef DDGEMM_CHECKED
    return 1;
#else
    return 0;
#endif
}

ddgemm_status dd_check_report(unsigned int* count, unsigned int* site, int64_t* index) {
    if (count == nullptr || site == nullptr || index == nullptr) return DDGEMM_ERR_INVALID_ARG;
    cudaError_t (*readers[])(CheckRecord*) = {check_record_split, check_record_slice_gemm, check_record_fused,
                                              check_record_recombine, check_record_tc, check_record_tc_md};
    *count = 0;
    *site = 0;
    *index = 0;
    for (auto read : readers) {
        CheckRecord r{};
        if (read(&r) != cudaSuccess) {
            cudaGetLastError();
            return DDGEMM_ERR_CUDA;
        }
        if (r.count > 0 && *count == 0) {
            *site = r.site;
            *index = r.index;
        }
        *count += r.count;
    }
    return DDGEMM_OK;
}

ddgemm_status dd_pool_trim(void) {
    cudaMemPool_t pool = nullptr;
    if (library_pool(&pool, false) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_CUDA;
    }
    if (pool == nullptr) return DDGEMM_OK;  // nothing allocated on this device yet
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemPoolTrimTo(pool, 0) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_CUDA;
    }
    return DDGEMM_OK;
}

// ---- the comparator ----

ddgemm_status dd_gemm_simt(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                           int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, double* C_hi,
                           double* C_lo, int64_t ldc, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if ((M + 31) / 32 > 65535) return DDGEMM_ERR_UNSUPPORTED;
    return from_cuda(launch_simt_dd_gemm(A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc, M, N, K,
                                         static_cast<cudaStream_t>(stream)));
}

// ---- integer-pipe variant ----

ddgemm_status dd_gemm_i64_layout(int64_t M, int64_t N, int64_t K, int* splits) {
    if (M < 0 || N < 0 || K < 0 || splits == nullptr) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    *splits = make_layout(M, N, K, Engine::kInt64Pipe).splits;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_i64_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (bytes == nullptr || M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    *bytes = (size_t)make_layout(M, N, K, Engine::kInt64Pipe).total;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_i64(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                          int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, double* C_hi,
                          double* C_lo, int64_t ldc, void* workspace, size_t workspace_bytes, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Layout L = make_layout(M, N, K, Engine::kInt64Pipe);
    const int64_t c = span_bytes(M, N, ldc);
    if (workspace != nullptr) {
        if ((uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)L.total) return DDGEMM_ERR_INVALID_ARG;
        if (ranges_overlap(workspace, L.total, C_hi, c) || ranges_overlap(workspace, L.total, C_lo, c))
            return DDGEMM_ERR_INVALID_ARG;
        return run_gemm_i64(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc,
                            static_cast<char*>(workspace), st);
    }
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)L.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_gemm_i64(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status dd_split_rows_i16(int64_t M, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                                int16_t* planes, int32_t* e, void* stream) {
    if (M < 0 || K < 0 || lda < std::max<int64_t>(1, K)) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0) return DDGEMM_OK;
    if (e == nullptr || (K > 0 && (A_hi == nullptr || A_lo == nullptr || planes == nullptr)))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planes % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t Kp = round_up(K, BK);
    DDG_TRY(run_split(M, 0, K, Kp, A_hi, A_lo, lda, e, planes, nullptr, nullptr, 1, nullptr, nullptr, true, st));
    return DDGEMM_OK;
}

ddgemm_status dd_split_cols_i16(int64_t K, int64_t N, const double* B_hi, const double* B_lo, int64_t ldb,
                                int16_t* planes, int32_t* f, void* stream) {
    if (N < 0 || K < 0 || ldb < std::max<int64_t>(1, N)) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (N == 0) return DDGEMM_OK;
    if (f == nullptr || (K > 0 && (B_hi == nullptr || B_lo == nullptr || planes == nullptr)))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planes % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t Kp = round_up(K, BK);
    DDG_TRY(run_split(0, N, K, Kp, nullptr, nullptr, 1, nullptr, nullptr, B_hi, B_lo, ldb, f, planes, true, st));
    return DDGEMM_OK;
}

ddgemm_status dd_slice_gemm_i64(int64_t M, int64_t N, int64_t K, const int16_t* planesA,
                                const int16_t* planesB, int splits, double* P, void* stream) {
    ddgemm_status s = check_shapes(M, N, K, std::max<int64_t>(1, K), std::max<int64_t>(1, N),
                                   std::max<int64_t>(1, N));
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, TM), Np = round_up(N, TN), Kp = round_up(K, BK), KC = Kp / BK;
    if (splits < 1 || splits > kMaxSplits || (KC > 0 && splits > KC) || (KC == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (P == nullptr || (K > 0 && (planesA == nullptr || planesB == nullptr))) return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0 || (uintptr_t)P % 16 != 0)
        return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(launch_slice_gemm_i64(planesA, planesB, Mp, Np, Kp, splits, P,
                                           static_cast<cudaStream_t>(stream)));
}

// ---- quad doubles on the integer pipe ----

static ddgemm_status check_qd_args(int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                                   const double* const* B, int64_t ldb, double* const* C, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((round_up(M, TM) / TM) * (round_up(N, TN) / TN) * 4 > kMaxTiles) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (A == nullptr || B == nullptr || C == nullptr) return DDGEMM_ERR_INVALID_ARG;
    const int64_t a = span_bytes(M, K, lda), b = span_bytes(K, N, ldb), c = span_bytes(M, N, ldc);
    for (int p = 0; p < 4; ++p) {
        if (C[p] == nullptr || (K > 0 && (A[p] == nullptr || B[p] == nullptr))) return DDGEMM_ERR_INVALID_ARG;
        for (int q = 0; q < 4; ++q) {
            if (ranges_overlap(C[p], c, A[q], a) || ranges_overlap(C[p], c, B[q], b)) return DDGEMM_ERR_INVALID_ARG;
            if (q != p && ranges_overlap(C[p], c, C[q], c)) return DDGEMM_ERR_INVALID_ARG;
        }
    }
    return DDGEMM_OK;
}

static ddgemm_status run_qd(const Layout& L, int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                            const double* const* B, int64_t ldb, double* const* C, int64_t ldc, char* ws,
                            cudaStream_t st) {
    int32_t* e = reinterpret_cast<int32_t*>(ws + L.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + L.off_f);
    int16_t* pA = reinterpret_cast<int16_t*>(ws + L.off_A);
    int16_t* pB = reinterpret_cast<int16_t*>(ws + L.off_B);
    double* P = reinterpret_cast<double*>(ws + L.off_P);
    SplitOperand a{A[0], A[1], lda, M, e}, b{B[0], B[1], ldb, N, f};
    DDG_STEP("qd/exponents", launch_shared_exponents(&a, &b, K, 0, st));
    DDG_STEP("qd/split", launch_split_qd(A, lda, M, e, B, ldb, N, f, K, L.Kp, pA, pB, st));
    DDG_STEP("qd/slice_gemm", launch_slice_gemm_qd(pA, pB, L.Mp, L.Np, L.Kp, L.splits, P, st));
    DDG_STEP("qd/recombine", launch_recombine_qd(P, L.splits, L.Mp, L.Np, e, f, M, N, C, ldc, st));
    return DDGEMM_OK;
}

ddgemm_status qd_gemm_layout(int64_t M, int64_t N, int64_t K, int* splits) {
    if (M < 0 || N < 0 || K < 0 || splits == nullptr) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    *splits = make_layout(M, N, K, Engine::kQuadInt64).splits;
    return DDGEMM_OK;
}

ddgemm_status qd_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (bytes == nullptr || M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    *bytes = (size_t)make_layout(M, N, K, Engine::kQuadInt64).total;
    return DDGEMM_OK;
}

ddgemm_status qd_gemm(int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                      const double* const* B, int64_t ldb, double* const* C, int64_t ldc, void* workspace,
                      size_t workspace_bytes, void* stream) {
    ddgemm_status s = check_qd_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (s != DDGEMM_OK || M == 0 || N == 0) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Layout L = make_layout(M, N, K, Engine::kQuadInt64);
    if (workspace != nullptr) {
        if ((uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)L.total) return DDGEMM_ERR_INVALID_ARG;
        return run_qd(L, M, N, K, A, lda, B, ldb, C, ldc, static_cast<char*>(workspace), st);
    }
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)L.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_qd(L, M, N, K, A, lda, B, ldb, C, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status qd_split(int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                       const double* const* B, int64_t ldb, int16_t* planesA, int32_t* e, int16_t* planesB,
                       int32_t* f, void* stream) {
    if (M < 0 || N < 0 || K < 0 || lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((M > 0 && (e == nullptr || A == nullptr || (K > 0 && planesA == nullptr))) ||
        (N > 0 && (f == nullptr || B == nullptr || (K > 0 && planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t Kp = round_up(K, BK);
    SplitOperand a{M > 0 ? A[0] : nullptr, nullptr, lda, M, e}, b{N > 0 ? B[0] : nullptr, nullptr, ldb, N, f};
    DDG_TRY(launch_shared_exponents(M > 0 ? &a : nullptr, N > 0 ? &b : nullptr, K, 0, st));
    DDG_TRY(launch_split_qd(M > 0 ? A : nullptr, lda, M, e, N > 0 ? B : nullptr, ldb, N, f, K, Kp, planesA,
                            planesB, st));
    return DDGEMM_OK;
}

ddgemm_status qd_slice_gemm(int64_t M, int64_t N, int64_t K, const int16_t* planesA, const int16_t* planesB,
                            int splits, double* P, void* stream) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, TM), Np = round_up(N, TN), Kp = round_up(K, BK), KC = Kp / BK;
    if (splits < 1 || splits > kMaxSplits || (KC > 0 && splits > KC) || (KC == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (P == nullptr || (K > 0 && (planesA == nullptr || planesB == nullptr))) return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0 || (uintptr_t)P % 16 != 0)
        return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(launch_slice_gemm_qd(planesA, planesB, Mp, Np, Kp, splits, P, static_cast<cudaStream_t>(stream)));
}

ddgemm_status qd_recombine(int64_t M, int64_t N, const double* P, int splits, const int32_t* e, const int32_t* f,
                           double* const* C, int64_t ldc, void* stream) {
    if (M < 0 || N < 0 || ldc < std::max<int64_t>(1, N) || splits < 1 || splits > kMaxSplits)
        return DDGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (P == nullptr || e == nullptr || f == nullptr || C == nullptr) return DDGEMM_ERR_INVALID_ARG;
    for (int p = 0; p < 4; ++p)
        if (C[p] == nullptr) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Mp = round_up(M, TM), Np = round_up(N, TN);
    return from_cuda(launch_recombine_qd(P, splits, Mp, Np, e, f, M, N, C, ldc, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dd_gemm_ex: the FP64 path with options (k-split, fused split, fused
// recombination).
// ---------------------------------------------------------------------------

namespace {

struct ExPlan {
    int64_t Mp, Np, Kp;
    int splits;
    bool fuse_split, fuse_recombine;
    int64_t off_e, off_f, off_A, off_B, off_P, total;
};

ddgemm_status make_ex_plan(int64_t M, int64_t N, int64_t K, const ddgemm_opts* opts, ExPlan& X) {
    ddgemm_opts o{};
    if (opts != nullptr) o = *opts;
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((o.slices != 0 && o.slices != S) || (o.pairs != 0 && o.pairs != S * (S + 1) / 2))
        return DDGEMM_ERR_UNSUPPORTED;
    if (o.split_k < 0 || (o.fuse_recombine != 0 && o.fuse_recombine != 1) || (o.fuse_split != 0 && o.fuse_split != 1))
        return DDGEMM_ERR_INVALID_ARG;
    X.Mp = round_up(M, TM);
    X.Np = round_up(N, TN);
    X.Kp = round_up(K, BK);
    const int64_t KC = X.Kp / BK;
    if (o.split_k > 0) {
        if (o.split_k > kMaxSplits || (KC > 0 && o.split_k > KC) || (KC == 0 && o.split_k != 1))
            return DDGEMM_ERR_INVALID_ARG;
        if (o.fuse_recombine && o.split_k > 1) return DDGEMM_ERR_UNSUPPORTED;
        X.splits = o.split_k;
    } else {
        X.splits = choose_splits(X.Mp, X.Np, KC, Engine::kFp64Tensor);
    }
    X.fuse_split = o.fuse_split == 1;
    X.fuse_recombine = o.fuse_recombine == 1 && X.splits == 1;
    int64_t off = 0;
    auto take = [&](int64_t bytes) { int64_t at = off; off = round_up(off + bytes, kAlign); return at; };
    X.off_e = take(X.Mp * 4);
    X.off_f = take(X.Np * 4);
    X.off_A = X.fuse_split ? -1 : take(S * X.Mp * X.Kp * 8);
    X.off_B = X.fuse_split ? -1 : take(S * X.Np * X.Kp * 8);
    X.off_P = X.fuse_recombine ? -1 : take((int64_t)X.splits * S * X.Mp * X.Np * 8);
    X.total = off;
    return DDGEMM_OK;
}

ddgemm_status run_gemm_ex(const ExPlan& X, int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                          int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, double* C_hi,
                          double* C_lo, int64_t ldc, char* ws, cudaStream_t st) {
    if (M == 0 || N == 0) return DDGEMM_OK;
    int32_t* e = reinterpret_cast<int32_t*>(ws + X.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + X.off_f);
    double* P = X.fuse_recombine ? nullptr : reinterpret_cast<double*>(ws + X.off_P);
    if (X.fuse_split) {
        SplitOperand a{A_hi, A_lo, lda, M, e, false}, b{B_hi, B_lo, ldb, N, f, false};
        DDG_STEP("dd_ex/exponents", launch_shared_exponents(&a, &b, K, 0, st));
        const FusedSrc g = make_fused_src(A_hi, A_lo, lda, B_hi, B_lo, ldb, e, f, M, N, K);
        if (X.fuse_recombine) {
            DDG_STEP("dd_ex/slice_gemm", launch_slice_gemm_fused_recombine(g, X.Mp, X.Np, X.Kp, C_hi, C_lo, ldc, st));
            return DDGEMM_OK;
        }
        DDG_STEP("dd_ex/slice_gemm", launch_slice_gemm_fused(g, X.Mp, X.Np, X.Kp, X.splits, P, st));
    } else {
        double* pA = reinterpret_cast<double*>(ws + X.off_A);
        double* pB = reinterpret_cast<double*>(ws + X.off_B);
        DDG_STEP("dd_ex/split", run_split(M, N, K, X.Kp, A_hi, A_lo, lda, e, pA, B_hi, B_lo, ldb, f, pB, false, st));
        if (X.fuse_recombine) {
            DDG_STEP("dd_ex/slice_gemm", launch_slice_gemm_recombine(pA, pB, X.Mp, X.Np, X.Kp, e, f, M, N, C_hi, C_lo, ldc, st));
            return DDGEMM_OK;
        }
        DDG_STEP("dd_ex/slice_gemm", launch_slice_gemm(pA, pB, X.Mp, X.Np, X.Kp, X.splits, P, st));
    }
    DDG_STEP("dd_ex/recombine", launch_recombine(P, X.splits, X.Mp, X.Np, e, f, M, N, C_hi, C_lo, ldc, st));
    return DDGEMM_OK;
}

}  // namespace

extern "C" {

ddgemm_status dd_gemm_ex_plan(int64_t M, int64_t N, int64_t K, const ddgemm_opts* opts, size_t* workspace_bytes,
                              int* splits, int* fused_recombine) {
    ExPlan X;
    ddgemm_status s = make_ex_plan(M, N, K, opts, X);
    if (s != DDGEMM_OK) return s;
    if (workspace_bytes) *workspace_bytes = (size_t)X.total;
    if (splits) *splits = X.splits;
    if (fused_recombine) *fused_recombine = X.fuse_recombine ? 1 : 0;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_ex(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                         const double* B_hi, const double* B_lo, int64_t ldb, double* C_hi, double* C_lo,
                         int64_t ldc, const ddgemm_opts* opts, void* workspace, size_t workspace_bytes,
                         void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    ExPlan X;
    s = make_ex_plan(M, N, K, opts, X);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t c = span_bytes(M, N, ldc);
    if (workspace != nullptr) {
        if ((uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)X.total) return DDGEMM_ERR_INVALID_ARG;
        if (ranges_overlap(workspace, X.total, C_hi, c) || ranges_overlap(workspace, X.total, C_lo, c))
            return DDGEMM_ERR_INVALID_ARG;
        return run_gemm_ex(X, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc,
                           static_cast<char*>(workspace), st);
    }
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)X.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_gemm_ex(X, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status dd_slice_gemm_fused(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                                  int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, const int32_t* e,
                                  const int32_t* f, int splits, double* P, void* stream) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, std::max<int64_t>(1, N));
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, TM), Np = round_up(N, TN), Kp = round_up(K, BK), KC = Kp / BK;
    if (splits < 1 || splits > kMaxSplits || (KC > 0 && splits > KC) || (KC == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (P == nullptr || e == nullptr || f == nullptr) return DDGEMM_ERR_INVALID_ARG;
    if (K > 0 && (A_hi == nullptr || A_lo == nullptr || B_hi == nullptr || B_lo == nullptr))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)P % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    const FusedSrc g = make_fused_src(A_hi, A_lo, lda, B_hi, B_lo, ldb, e, f, M, N, K);
    return from_cuda(launch_slice_gemm_fused(g, Mp, Np, Kp, splits, P, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Double doubles with 8-bit parts on the bf16 tensor cores.
// ---------------------------------------------------------------------------

namespace {

constexpr int64_t kTcM = DDGEMM_TC_TILE_M, kTcN = DDGEMM_TC_TILE_N, kTcK = DDGEMM_TC_CHUNK_K;
constexpr int kTcParts = DDGEMM_TC_SLICES;
constexpr int kTcMaxSplits = 65535;  // k-splits accepted by the tensor-core step entry points

struct TcLayout {
    int64_t Mp, Np, Kp;
    int splits;
    int64_t off_e, off_f, off_A, off_B, off_P, total;
};

// k-split of the bf16 slice GEMM: at least enough splits that each covers at
// most DDGEMM_TC_MAX_K_SPLIT of k (exact int32 part sums); beyond that, the
// count whose waves of blocks (one per SM) fill the GPU best, each split
// keeping at least 512 of k, with a small cost per split (each writes its own
// part sums).  One output block occupies a pair of SMs.
// Largest k of one k-split for `parts` parts: the largest power of two with
// parts K 2^14 < 2^31 (int32 part sums stay exact).
int64_t tc_max_k_split(int parts) {
    int64_t k = 1 << 20;
    while ((int64_t)parts * k * 128 * 128 >= (1LL << 31)) k >>= 1;
    return k;
}

// Pair passes over one k-block of the busiest CTA pair of the tensor-core GEMM
// with s k-splits, dealing its units out as the kernel does: units numbered
// from the heaviest diagonal down (then k-split, then output block), one unit
// per pair and round, the order of the pairs reversed every other round.
int64_t busiest_pair(int64_t tiles, int64_t s, int np, int64_t KB, int64_t pairs) {
    const int64_t units = tiles * s * np, kb_per = (KB + s - 1) / s;
    pairs = std::max<int64_t>(1, std::min(pairs, units));
    int64_t worst = 0;
    for (int64_t p = 0; p < pairs; ++p) {
        int64_t w = 0;
        for (int64_t r = 0;; ++r) {
            const int64_t u = r * pairs + ((r & 1) ? pairs - 1 - p : p);
            if (u >= units) break;
            const int64_t d = np - 1 - u / (tiles * s), z = (u / tiles) % s;
            w += (d + 1) * std::max<int64_t>(0, std::min(KB, (z + 1) * kb_per) - z * kb_per);
        }
        worst = std::max(worst, w);
    }
    return worst;
}

// k-splits of the tensor-core GEMM: at least enough for exact int32 sums;
// more only where the finer units balance the persistent pairs by more than
// the extra part sums cost.  Model (microseconds): a pair passes one k-block
// of a 256 x 256 block (2 x 256 x 256 x 64 flops) in about 0.37 us, and each
// k-split's int32 part sums are written and read back once at about 6 TB/s.
int choose_tc_splits_uncached(int64_t Mp, int64_t Np, int64_t Kp, int parts, int64_t pairs) {
    const int64_t KB = Kp / kTcK;
    const int64_t tiles = (Mp / kTcM) * (Np / kTcN);
    if (tiles == 0 || KB == 0) return 1;
    const int64_t per_split = tc_max_k_split(parts) / kTcK;
    const int64_t smin = std::max<int64_t>(1, (KB + per_split - 1) / per_split);
    const int64_t smax = std::min<int64_t>(KB, std::max<int64_t>(4 * smin, 64));
    const double t_pass = 0.37;
    const double t_split = 2.0 * parts * (double)Mp * (double)Np * 4.0 / 6.0e6;
    int64_t best = smin, evaluated = 0;
    double best_t = -1.0;
    for (int64_t s = smin; s <= smax; ++s) {
        const int64_t kb_per = (KB + s - 1) / s;
        if ((KB + kb_per - 1) / kb_per != s) continue;  // some split would be empty
        // many units balance well anyway: bound the host work of the search
        if (s > smin && (tiles * s * parts > (1 << 18) || evaluated > (1 << 21))) break;
        evaluated += tiles * s * parts;
        const double t = (double)busiest_pair(tiles, s, parts, KB, pairs) * t_pass + s * t_split;
        if (best_t < 0.0 || t < best_t * 0.98) { best_t = t; best = s; }
    }
    return (int)best;
}

// The choice above, remembered for the last few shapes (layouts are asked for
// on every call).
int choose_tc_splits(int64_t Mp, int64_t Np, int64_t Kp, int parts) {
    struct Entry { int64_t Mp, Np, Kp, pairs; int parts, splits; };
    static std::mutex mu;
    static Entry cache[16];
    static int next = 0, used = 0;
    const int64_t pairs = tc_resident_pairs();  // of the current device
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].Mp == Mp && cache[i].Np == Np && cache[i].Kp == Kp && cache[i].parts == parts &&
                cache[i].pairs == pairs)
                return cache[i].splits;
    }
    const int s = choose_tc_splits_uncached(Mp, Np, Kp, parts, pairs);
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{Mp, Np, Kp, pairs, parts, s};
    next = (next + 1) % 16;
    used = std::min(used + 1, 16);
    return s;
}

// parts = 13 (double doubles), 27 (quad), 54 (octo) or 107 (hexa doubles).
TcLayout make_tc_layout(int64_t M, int64_t N, int64_t K, int parts = kTcParts) {
    TcLayout L;
    L.Mp = round_up(M, kTcM);
    L.Np = round_up(N, kTcN);
    L.Kp = round_up(K, kTcK);
    L.splits = choose_tc_splits(L.Mp, L.Np, L.Kp, parts);
    int64_t off = 0;
    auto take = [&](int64_t bytes) { int64_t o = off; off = round_up(off + bytes, kAlign); return o; };
    L.off_e = take(L.Mp * 4);
    L.off_f = take(L.Np * 4);
    L.off_A = take((int64_t)parts * L.Mp * L.Kp * 2);
    L.off_B = take((int64_t)parts * L.Np * L.Kp * 2);
    L.off_P = take((int64_t)L.splits * parts * L.Mp * L.Np * 4);
    L.total = off;
    return L;
}

// The tensor copies of the slice GEMM address the part blocks of an operand as
// rows of 128 bytes with 32-bit coordinates: Mp (or Np) x parts x Kp/64 rows
// must stay below 2^31 (2^31 rows are 256 GiB of parts, more than the device
// holds, so this never binds in practice).
bool tc_part_rows_ok(int64_t M, int64_t N, int64_t K, int parts) {
    const int64_t kb = round_up(K, kTcK) / kTcK;
    const int64_t lim = (1LL << 31) / std::max<int64_t>(1, (int64_t)parts * std::max<int64_t>(1, kb));
    return round_up(M, kTcM) < lim && round_up(N, kTcN) < lim;
}

ddgemm_status check_tc_shapes(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > DDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((round_up(M, kTcM) / kTcM) * (round_up(N, kTcN) / kTcN) > kMaxTiles) return DDGEMM_ERR_UNSUPPORTED;
    if (!tc_part_rows_ok(M, N, K, kTcParts)) return DDGEMM_ERR_UNSUPPORTED;
    return DDGEMM_OK;
}

cudaError_t run_split_tc(int64_t M, int64_t N, int64_t K, int64_t Kp, const double* A_hi, const double* A_lo,
                         int64_t lda, int32_t* e, uint16_t* pA, const double* B_hi, const double* B_lo, int64_t ldb,
                         int32_t* f, uint16_t* pB, cudaStream_t st) {
    SplitOperand a{A_hi, A_lo, lda, M, e}, b{B_hi, B_lo, ldb, N, f};
    const SplitOperand* pa = (e != nullptr && M > 0) ? &a : nullptr;
    const SplitOperand* pb = (f != nullptr && N > 0) ? &b : nullptr;
    cudaError_t err = launch_shared_exponents(pa, pb, K, 0, st);
    if (err == cudaSuccess) err = launch_split_bf16(pa, pb, K, Kp, pa ? pA : nullptr, pb ? pB : nullptr, st);
    return err;
}

ddgemm_status run_gemm_tc(const TcLayout& L, int64_t M, int64_t N, int64_t K, const double* A_hi,
                          const double* A_lo, int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb,
                          double* C_hi, double* C_lo, int64_t ldc, char* ws, cudaStream_t st) {
    if (M == 0 || N == 0) return DDGEMM_OK;
    int32_t* e = reinterpret_cast<int32_t*>(ws + L.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + L.off_f);
    uint16_t* pA = reinterpret_cast<uint16_t*>(ws + L.off_A);
    uint16_t* pB = reinterpret_cast<uint16_t*>(ws + L.off_B);
    int32_t* P = reinterpret_cast<int32_t*>(ws + L.off_P);
    DDG_STEP("dd_tc/split", run_split_tc(M, N, K, L.Kp, A_hi, A_lo, lda, e, pA, B_hi, B_lo, ldb, f, pB, st));
    DDG_STEP("dd_tc/slice_gemm", launch_slice_gemm_tc(pA, pB, L.Mp, L.Np, L.Kp, L.splits, P, st));
    DDG_STEP("dd_tc/recombine", launch_recombine_tc(P, L.splits, L.Mp, L.Np, e, f, M, N, C_hi, C_lo, ldc, st));
    return DDGEMM_OK;
}

// The library's copy stream on the current device (non-blocking, created on
// first use): the host-buffer products move data on it while the caller's
// stream computes, joined to that stream through events.
cudaError_t copy_stream(cudaStream_t* cs) {
    static std::mutex mu;
    static cudaStream_t streams[kMaxPoolDevices] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxPoolDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (streams[dev] == nullptr) {
        err = cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
        if (err != cudaSuccess) return err;
    }
    *cs = streams[dev];
    return cudaSuccess;
}

// dd_gemm_tc with host operands, its copies overlapped with the work: A goes
// up in blocks of rows on the copy stream (the first block, then all of B,
// then the other blocks); the caller's stream splits B once, then for each
// block of rows splits it, multiplies it by B and recombines its rows of C,
// and the copy stream brings each finished block of C back while the next
// one is computed.  A row of C depends only on its row of A (whose exponent
// is its own) and on all of B, so the blocks give the one-shot product's
// result bit for bit.  Device memory from the library's pool; returns after
// C is in the host buffers (synchronises `st`).
ddgemm_status tc_host_pipelined(int64_t M, int64_t N, int64_t K, const double* h_A_hi, const double* h_A_lo,
                                int64_t lda, const double* h_B_hi, const double* h_B_lo, int64_t ldb,
                                double* h_C_hi, double* h_C_lo, int64_t ldc, cudaStream_t st) {
    constexpr int kBlocks = 4;
    const int64_t rows = round_up((M + kBlocks - 1) / kBlocks, kTcM);  // rows per block, a multiple of 256
    const int64_t nb = (M + rows - 1) / rows;
    const TcLayout LF = make_tc_layout(rows, N, K);                      // a full block
    const TcLayout LL = make_tc_layout(M - (nb - 1) * rows, N, K);      // the last block
    const int64_t Np = LF.Np, Kp = LF.Kp;
    const int64_t a = round_up(M * K * 8, kAlign), b = round_up(K * N * 8, kAlign), c = round_up(M * N * 8, kAlign);
    const int64_t ee = round_up(M * 4, kAlign), ff = round_up(Np * 4, kAlign);
    const int64_t pb = round_up((int64_t)kTcParts * Np * Kp * 2, kAlign);
    const int64_t pa = round_up((int64_t)kTcParts * LF.Mp * Kp * 2, kAlign);
    const int64_t pp = round_up((int64_t)std::max(LF.splits, LL.splits) * kTcParts * LF.Mp * Np * 4, kAlign);
    const int64_t total = 2 * a + 2 * b + 2 * c + ee + ff + pb + pa + pp;

    unsigned int timeouts_before = 0;
    if (peek_wait_timeouts_tc(&timeouts_before, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_CUDA;
    }
    cudaStream_t cs = nullptr;
    if (copy_stream(&cs) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_CUDA;
    }
    char* dev = nullptr;
    if (pool_alloc(reinterpret_cast<void**>(&dev), (size_t)total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    double* dA_hi = reinterpret_cast<double*>(dev);
    double* dA_lo = reinterpret_cast<double*>(dev + a);
    double* dB_hi = reinterpret_cast<double*>(dev + 2 * a);
    double* dB_lo = reinterpret_cast<double*>(dev + 2 * a + b);
    double* dC_hi = reinterpret_cast<double*>(dev + 2 * a + 2 * b);
    double* dC_lo = reinterpret_cast<double*>(dev + 2 * a + 2 * b + c);
    int32_t* e = reinterpret_cast<int32_t*>(dev + 2 * a + 2 * b + 2 * c);
    int32_t* f = reinterpret_cast<int32_t*>(dev + 2 * a + 2 * b + 2 * c + ee);
    uint16_t* pB = reinterpret_cast<uint16_t*>(dev + 2 * a + 2 * b + 2 * c + ee + ff);
    uint16_t* pA = reinterpret_cast<uint16_t*>(dev + 2 * a + 2 * b + 2 * c + ee + ff + pb);
    int32_t* P = reinterpret_cast<int32_t*>(dev + 2 * a + 2 * b + 2 * c + ee + ff + pb + pa);

    // events: [0] start (st), [1] B up, [2 .. 2+nb) A blocks up, [2+nb .. 2+2nb) C blocks done, [2+2nb] all down
    std::vector<cudaEvent_t> ev((size_t)(3 + 2 * nb), nullptr);
    cudaError_t err = cudaSuccess;
    for (auto& x : ev)
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
    auto up = [&](double* dst, const double* src, int64_t r, int64_t cols, int64_t ld) {
        if (err == cudaSuccess && r > 0 && cols > 0)
            err = cudaMemcpy2DAsync(dst, (size_t)cols * 8, src, (size_t)ld * 8, (size_t)cols * 8, (size_t)r,
                                    cudaMemcpyHostToDevice, cs);
    };
    auto block_rows = [&](int64_t i) { return std::min(rows, M - i * rows); };
    if (err == cudaSuccess) err = cudaEventRecord(ev[0], st);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(cs, ev[0], 0);
    for (int64_t i = 0; i < nb; ++i) {
        up(dA_hi + i * rows * K, h_A_hi + i * rows * lda, block_rows(i), K, lda);
        up(dA_lo + i * rows * K, h_A_lo + i * rows * lda, block_rows(i), K, lda);
        if (err == cudaSuccess) err = cudaEventRecord(ev[2 + i], cs);
        if (i == 0) {
            up(dB_hi, h_B_hi, K, N, ldb);
            up(dB_lo, h_B_lo, K, N, ldb);
            if (err == cudaSuccess) err = cudaEventRecord(ev[1], cs);
        }
    }
    // the caller's stream: B's exponents and parts once, then block by block
    if (err == cudaSuccess) err = cudaStreamWaitEvent(st, ev[1], 0);
    if (err == cudaSuccess) err = run_split_tc(0, N, K, Kp, nullptr, nullptr, 1, nullptr, nullptr, dB_hi, dB_lo, N, f, pB, st);
    for (int64_t i = 0; i < nb && err == cudaSuccess; ++i) {
        const int64_t r0 = i * rows, mb = block_rows(i);
        const TcLayout& L = i + 1 < nb ? LF : LL;
        err = cudaStreamWaitEvent(st, ev[2 + i], 0);
        if (err == cudaSuccess)
            err = run_split_tc(mb, 0, K, Kp, dA_hi + r0 * K, dA_lo + r0 * K, K, e + r0, pA, nullptr, nullptr, 1,
                               nullptr, nullptr, st);
        if (err == cudaSuccess) err = launch_slice_gemm_tc(pA, pB, L.Mp, Np, Kp, L.splits, P, st);
        if (err == cudaSuccess)
            err = launch_recombine_tc(P, L.splits, L.Mp, Np, e + r0, f, mb, N, dC_hi + r0 * N, dC_lo + r0 * N, N, st);
        if (err == cudaSuccess) err = cudaEventRecord(ev[2 + nb + i], st);
    }
    // the copy stream: each block of C back as soon as it is done
    for (int64_t i = 0; i < nb && err == cudaSuccess; ++i) {
        const int64_t r0 = i * rows, mb = block_rows(i);
        err = cudaStreamWaitEvent(cs, ev[2 + nb + i], 0);
        if (err == cudaSuccess)
            err = cudaMemcpy2DAsync(h_C_hi + r0 * ldc, (size_t)ldc * 8, dC_hi + r0 * N, (size_t)N * 8, (size_t)N * 8,
                                    (size_t)mb, cudaMemcpyDeviceToHost, cs);
        if (err == cudaSuccess)
            err = cudaMemcpy2DAsync(h_C_lo + r0 * ldc, (size_t)ldc * 8, dC_lo + r0 * N, (size_t)N * 8, (size_t)N * 8,
                                    (size_t)mb, cudaMemcpyDeviceToHost, cs);
    }
    // join, release, wait
    cudaError_t je = ev[2 + 2 * nb] ? cudaEventRecord(ev[2 + 2 * nb], cs) : cudaErrorInvalidValue;
    if (je == cudaSuccess) je = cudaStreamWaitEvent(st, ev[2 + 2 * nb], 0);
    if (je != cudaSuccess) je = cudaStreamSynchronize(cs);  // the copy stream must be idle before the memory goes
    cudaError_t fe = cudaFreeAsync(dev, st);
    cudaError_t se = cudaStreamSynchronize(st);
    for (auto& x : ev)
        if (x) cudaEventDestroy(x);
    ddgemm_status s = (err == cudaSuccess && je == cudaSuccess && fe == cudaSuccess && se == cudaSuccess)
                          ? DDGEMM_OK : DDGEMM_ERR_CUDA;
    unsigned int timeouts_after = 0;
    if (s == DDGEMM_OK && (peek_wait_timeouts_tc(&timeouts_after, st) != cudaSuccess || timeouts_after != timeouts_before))
        s = DDGEMM_ERR_CUDA;
    if (s != DDGEMM_OK) cudaGetLastError();
    return s;
}

}  // namespace

extern "C" {

ddgemm_status dd_gemm_tc_layout(int64_t M, int64_t N, int64_t K, int64_t* Mp, int64_t* Np, int64_t* Kp,
                                int* splits) {
    ddgemm_status s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    TcLayout L = make_tc_layout(M, N, K);
    if (Mp) *Mp = L.Mp;
    if (Np) *Np = L.Np;
    if (Kp) *Kp = L.Kp;
    if (splits) *splits = L.splits;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_tc_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (bytes == nullptr) return DDGEMM_ERR_INVALID_ARG;
    ddgemm_status s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    *bytes = (size_t)make_tc_layout(M, N, K).total;
    return DDGEMM_OK;
}

ddgemm_status dd_gemm_tc(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                         const double* B_hi, const double* B_lo, int64_t ldb, double* C_hi, double* C_lo,
                         int64_t ldc, void* workspace, size_t workspace_bytes, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s == DDGEMM_OK) s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TcLayout L = make_tc_layout(M, N, K);
    const int64_t c = span_bytes(M, N, ldc);
    if (workspace != nullptr) {
        if ((uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)L.total) return DDGEMM_ERR_INVALID_ARG;
        if (ranges_overlap(workspace, L.total, C_hi, c) || ranges_overlap(workspace, L.total, C_lo, c))
            return DDGEMM_ERR_INVALID_ARG;
        return run_gemm_tc(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc,
                           static_cast<char*>(workspace), st);
    }
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)L.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_gemm_tc(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status dd_gemm_tc_host(int64_t M, int64_t N, int64_t K, const double* h_A_hi, const double* h_A_lo,
                              int64_t lda, const double* h_B_hi, const double* h_B_lo, int64_t ldb, double* h_C_hi,
                              double* h_C_lo, int64_t ldc, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, h_A_hi, h_A_lo, lda, h_B_hi, h_B_lo, ldb, h_C_hi, h_C_lo, ldc);
    if (s == DDGEMM_OK) s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (M >= 4 * kTcM && K > 0)  // enough rows for blocks of at least 256 to overlap the copies
        return tc_host_pipelined(M, N, K, h_A_hi, h_A_lo, lda, h_B_hi, h_B_lo, ldb, h_C_hi, h_C_lo, ldc,
                                 static_cast<cudaStream_t>(stream));
    TcLayout L = make_tc_layout(M, N, K);
    return host_product(M, N, K, h_A_hi, h_A_lo, lda, h_B_hi, h_B_lo, ldb, h_C_hi, h_C_lo, ldc, L.total,
                        static_cast<cudaStream_t>(stream),
                        [&](const double* a_hi, const double* a_lo, const double* b_hi, const double* b_lo,
                            double* c_hi, double* c_lo, char* ws, cudaStream_t st) {
                            return run_gemm_tc(L, M, N, K, a_hi, a_lo, std::max<int64_t>(K, 1), b_hi, b_lo, N,
                                               c_hi, c_lo, N, ws, st);
                        },
                        peek_wait_timeouts_tc);
}

ddgemm_status dd_split_bf16(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo, int64_t lda,
                            const double* B_hi, const double* B_lo, int64_t ldb, uint16_t* planesA, int32_t* e,
                            uint16_t* planesB, int32_t* f, void* stream) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, std::max<int64_t>(1, N));
    if (s == DDGEMM_OK) s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    if (M > 0 && (e == nullptr || (K > 0 && (A_hi == nullptr || A_lo == nullptr || planesA == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if (N > 0 && (f == nullptr || (K > 0 && (B_hi == nullptr || B_lo == nullptr || planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Kp = round_up(K, kTcK);
    return from_cuda(run_split_tc(M, N, K, Kp, A_hi, A_lo, lda, M > 0 ? e : nullptr, planesA, B_hi, B_lo, ldb,
                                  N > 0 ? f : nullptr, planesB, static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_split_bf16_with_exponents(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                                           int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb,
                                           const int32_t* e, const int32_t* f, uint16_t* planesA, uint16_t* planesB,
                                           void* stream) {
    ddgemm_status s = check_shapes(M, N, K, lda, ldb, std::max<int64_t>(1, N));
    if (s == DDGEMM_OK) s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    if (M > 0 && (e == nullptr || (K > 0 && (A_hi == nullptr || A_lo == nullptr || planesA == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if (N > 0 && (f == nullptr || (K > 0 && (B_hi == nullptr || B_lo == nullptr || planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    SplitOperand a{A_hi, A_lo, lda, M, const_cast<int32_t*>(e), true};
    SplitOperand b{B_hi, B_lo, ldb, N, const_cast<int32_t*>(f), true};
    return from_cuda(launch_split_bf16(M > 0 ? &a : nullptr, N > 0 ? &b : nullptr, K, round_up(K, kTcK),
                                       M > 0 ? planesA : nullptr, N > 0 ? planesB : nullptr,
                                       static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_slice_gemm_tc(int64_t M, int64_t N, int64_t K, const uint16_t* planesA, const uint16_t* planesB,
                               int splits, int32_t* P, void* stream) {
    ddgemm_status s = check_tc_shapes(M, N, K);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, kTcM), Np = round_up(N, kTcN), Kp = round_up(K, kTcK), KB = Kp / kTcK;
    if (splits < 1 || splits > kTcMaxSplits || (KB > 0 && splits > KB) || (KB == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (KB > 0 && ((KB + splits - 1) / splits) * kTcK > DDGEMM_TC_MAX_K_SPLIT) return DDGEMM_ERR_INVALID_ARG;
    if (P == nullptr || (K > 0 && (planesA == nullptr || planesB == nullptr))) return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0 || (uintptr_t)P % 16 != 0)
        return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(launch_slice_gemm_tc(planesA, planesB, Mp, Np, Kp, splits, P, static_cast<cudaStream_t>(stream)));
}

ddgemm_status dd_recombine_tc(int64_t M, int64_t N, const int32_t* P, int splits, const int32_t* e,
                              const int32_t* f, double* C_hi, double* C_lo, int64_t ldc, void* stream) {
    if (M < 0 || N < 0 || ldc < std::max<int64_t>(1, N)) return DDGEMM_ERR_INVALID_ARG;
    if (splits < 1 || splits > kTcMaxSplits) return DDGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (P == nullptr || e == nullptr || f == nullptr || C_hi == nullptr || C_lo == nullptr)
        return DDGEMM_ERR_INVALID_ARG;
    const int64_t Mp = round_up(M, kTcM), Np = round_up(N, kTcN);
    return from_cuda(launch_recombine_tc(P, splits, Mp, Np, e, f, M, N, C_hi, C_lo, ldc,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---- quad doubles with 27 bf16 parts ----

namespace {

constexpr int kTcQdParts = DDGEMM_TC_QD_SLICES;

ddgemm_status check_tc_qd_args(int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                               const double* const* B, int64_t ldb, double* const* C, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((round_up(M, kTcM) / kTcM) * (round_up(N, kTcN) / kTcN) > kMaxTiles) return DDGEMM_ERR_UNSUPPORTED;
    if (!tc_part_rows_ok(M, N, K, kTcQdParts)) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (A == nullptr || B == nullptr || C == nullptr) return DDGEMM_ERR_INVALID_ARG;
    const int64_t a = span_bytes(M, K, lda), b = span_bytes(K, N, ldb), c = span_bytes(M, N, ldc);
    for (int p = 0; p < 4; ++p) {
        if (C[p] == nullptr || (K > 0 && (A[p] == nullptr || B[p] == nullptr))) return DDGEMM_ERR_INVALID_ARG;
        for (int q = 0; q < 4; ++q) {
            if (ranges_overlap(C[p], c, A[q], a) || ranges_overlap(C[p], c, B[q], b)) return DDGEMM_ERR_INVALID_ARG;
            if (q != p && ranges_overlap(C[p], c, C[q], c)) return DDGEMM_ERR_INVALID_ARG;
        }
    }
    return DDGEMM_OK;
}

cudaError_t run_split_tc_qd(int64_t M, int64_t N, int64_t K, int64_t Kp, const double* const* A, int64_t lda,
                            int32_t* e, uint16_t* pA, const double* const* B, int64_t ldb, int32_t* f, uint16_t* pB,
                            cudaStream_t st) {
    const bool has_a = A != nullptr && e != nullptr && M > 0, has_b = B != nullptr && f != nullptr && N > 0;
    SplitOperand a{has_a ? A[0] : nullptr, nullptr, lda, M, e}, b{has_b ? B[0] : nullptr, nullptr, ldb, N, f};
    cudaError_t err = launch_shared_exponents(has_a ? &a : nullptr, has_b ? &b : nullptr, K, 0, st);
    if (err == cudaSuccess)
        err = launch_split_bf16_qd(has_a ? A : nullptr, lda, M, e, has_b ? B : nullptr, ldb, N, f, K, Kp, pA, pB, st);
    return err;
}

ddgemm_status run_qd_tc(const TcLayout& L, int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                        const double* const* B, int64_t ldb, double* const* C, int64_t ldc, char* ws,
                        cudaStream_t st) {
    int32_t* e = reinterpret_cast<int32_t*>(ws + L.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + L.off_f);
    uint16_t* pA = reinterpret_cast<uint16_t*>(ws + L.off_A);
    uint16_t* pB = reinterpret_cast<uint16_t*>(ws + L.off_B);
    int32_t* P = reinterpret_cast<int32_t*>(ws + L.off_P);
    DDG_STEP("qd_tc/split", run_split_tc_qd(M, N, K, L.Kp, A, lda, e, pA, B, ldb, f, pB, st));
    DDG_STEP("qd_tc/slice_gemm", launch_slice_gemm_tc_qd(pA, pB, L.Mp, L.Np, L.Kp, L.splits, P, st));
    DDG_STEP("qd_tc/recombine", launch_recombine_tc_qd(P, L.splits, L.Mp, L.Np, e, f, M, N, C, ldc, st));
    return DDGEMM_OK;
}

}  // namespace

extern "C" {

ddgemm_status qd_gemm_tc_layout(int64_t M, int64_t N, int64_t K, int64_t* Mp, int64_t* Np, int64_t* Kp,
                                int* splits) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K || !tc_part_rows_ok(M, N, K, kTcQdParts)) return DDGEMM_ERR_UNSUPPORTED;
    TcLayout L = make_tc_layout(M, N, K, kTcQdParts);
    if (Mp) *Mp = L.Mp;
    if (Np) *Np = L.Np;
    if (Kp) *Kp = L.Kp;
    if (splits) *splits = L.splits;
    return DDGEMM_OK;
}

ddgemm_status qd_gemm_tc_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (bytes == nullptr || M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K || !tc_part_rows_ok(M, N, K, kTcQdParts)) return DDGEMM_ERR_UNSUPPORTED;
    *bytes = (size_t)make_tc_layout(M, N, K, kTcQdParts).total;
    return DDGEMM_OK;
}

ddgemm_status qd_gemm_tc(int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                         const double* const* B, int64_t ldb, double* const* C, int64_t ldc, void* workspace,
                         size_t workspace_bytes, void* stream) {
    ddgemm_status s = check_tc_qd_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (s != DDGEMM_OK || M == 0 || N == 0) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TcLayout L = make_tc_layout(M, N, K, kTcQdParts);
    if (workspace != nullptr) {
        if ((uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)L.total) return DDGEMM_ERR_INVALID_ARG;
        return run_qd_tc(L, M, N, K, A, lda, B, ldb, C, ldc, static_cast<char*>(workspace), st);
    }
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)L.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_qd_tc(L, M, N, K, A, lda, B, ldb, C, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status qd_split_bf16(int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                            const double* const* B, int64_t ldb, uint16_t* planesA, int32_t* e, uint16_t* planesB,
                            int32_t* f, void* stream) {
    if (M < 0 || N < 0 || K < 0 || lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((M > 0 && (e == nullptr || A == nullptr || (K > 0 && planesA == nullptr))) ||
        (N > 0 && (f == nullptr || B == nullptr || (K > 0 && planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Kp = round_up(K, kTcK);
    return from_cuda(run_split_tc_qd(M, N, K, Kp, M > 0 ? A : nullptr, lda, e, planesA, N > 0 ? B : nullptr, ldb, f,
                                     planesB, static_cast<cudaStream_t>(stream)));
}

ddgemm_status qd_slice_gemm_tc(int64_t M, int64_t N, int64_t K, const uint16_t* planesA, const uint16_t* planesB,
                               int splits, int32_t* P, void* stream) {
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, kTcM), Np = round_up(N, kTcN), Kp = round_up(K, kTcK), KB = Kp / kTcK;
    if (splits < 1 || splits > kTcMaxSplits || (KB > 0 && splits > KB) || (KB == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (KB > 0 && ((KB + splits - 1) / splits) * kTcK > DDGEMM_TC_QD_MAX_K_SPLIT) return DDGEMM_ERR_INVALID_ARG;
    if (!tc_part_rows_ok(M, N, K, kTcQdParts)) return DDGEMM_ERR_UNSUPPORTED;
    if (P == nullptr || (K > 0 && (planesA == nullptr || planesB == nullptr))) return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0 || (uintptr_t)P % 16 != 0)
        return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(launch_slice_gemm_tc_qd(planesA, planesB, Mp, Np, Kp, splits, P,
                                             static_cast<cudaStream_t>(stream)));
}

ddgemm_status qd_recombine_tc(int64_t M, int64_t N, const int32_t* P, int splits, const int32_t* e,
                              const int32_t* f, double* const* C, int64_t ldc, void* stream) {
    if (M < 0 || N < 0 || ldc < std::max<int64_t>(1, N) || splits < 1 || splits > kTcMaxSplits)
        return DDGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (P == nullptr || e == nullptr || f == nullptr || C == nullptr) return DDGEMM_ERR_INVALID_ARG;
    for (int p = 0; p < 4; ++p)
        if (C[p] == nullptr) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Mp = round_up(M, kTcM), Np = round_up(N, kTcN);
    return from_cuda(launch_recombine_tc_qd(P, splits, Mp, Np, e, f, M, N, C, ldc, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---- octo and hexa doubles with bf16 parts ----

namespace {

int md_parts(int nparts) {
    return nparts == 8 ? DDGEMM_TC_OD_SLICES : nparts == 16 ? DDGEMM_TC_HD_SLICES : 0;
}

ddgemm_status check_tc_md_args(int nparts, int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                               const double* const* B, int64_t ldb, double* const* C, int64_t ldc) {
    if (md_parts(nparts) == 0) return DDGEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((round_up(M, kTcM) / kTcM) * (round_up(N, kTcN) / kTcN) > kMaxTiles) return DDGEMM_ERR_UNSUPPORTED;
    if (!tc_part_rows_ok(M, N, K, md_parts(nparts))) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (A == nullptr || B == nullptr || C == nullptr) return DDGEMM_ERR_INVALID_ARG;
    const int64_t a = span_bytes(M, K, lda), b = span_bytes(K, N, ldb), c = span_bytes(M, N, ldc);
    for (int p = 0; p < nparts; ++p) {
        if (C[p] == nullptr || (K > 0 && (A[p] == nullptr || B[p] == nullptr))) return DDGEMM_ERR_INVALID_ARG;
        for (int q = 0; q < nparts; ++q) {
            if (ranges_overlap(C[p], c, A[q], a) || ranges_overlap(C[p], c, B[q], b)) return DDGEMM_ERR_INVALID_ARG;
            if (q != p && ranges_overlap(C[p], c, C[q], c)) return DDGEMM_ERR_INVALID_ARG;
        }
    }
    return DDGEMM_OK;
}

cudaError_t run_split_tc_md(int nparts, int64_t M, int64_t N, int64_t K, int64_t Kp, const double* const* A,
                            int64_t lda, int32_t* e, uint16_t* pA, const double* const* B, int64_t ldb, int32_t* f,
                            uint16_t* pB, cudaStream_t st) {
    const bool has_a = A != nullptr && e != nullptr && M > 0, has_b = B != nullptr && f != nullptr && N > 0;
    SplitOperand a{has_a ? A[0] : nullptr, nullptr, lda, M, e}, b{has_b ? B[0] : nullptr, nullptr, ldb, N, f};
    cudaError_t err = launch_shared_exponents(has_a ? &a : nullptr, has_b ? &b : nullptr, K, 0, st);
    if (err == cudaSuccess)
        err = launch_split_bf16_md(nparts, has_a ? A : nullptr, lda, M, e, has_b ? B : nullptr, ldb, N, f, K, Kp, pA,
                                   pB, st);
    return err;
}

ddgemm_status run_md_tc(int nparts, const TcLayout& L, int64_t M, int64_t N, int64_t K, const double* const* A,
                        int64_t lda, const double* const* B, int64_t ldb, double* const* C, int64_t ldc, char* ws,
                        cudaStream_t st) {
    int32_t* e = reinterpret_cast<int32_t*>(ws + L.off_e);
    int32_t* f = reinterpret_cast<int32_t*>(ws + L.off_f);
    uint16_t* pA = reinterpret_cast<uint16_t*>(ws + L.off_A);
    uint16_t* pB = reinterpret_cast<uint16_t*>(ws + L.off_B);
    int32_t* P = reinterpret_cast<int32_t*>(ws + L.off_P);
    DDG_STEP("md_tc/split", run_split_tc_md(nparts, M, N, K, L.Kp, A, lda, e, pA, B, ldb, f, pB, st));
    DDG_STEP("md_tc/slice_gemm", launch_slice_gemm_tc_md(nparts, pA, pB, L.Mp, L.Np, L.Kp, L.splits, P, st));
    DDG_STEP("md_tc/recombine", launch_recombine_tc_md(nparts, P, L.splits, L.Mp, L.Np, e, f, M, N, C, ldc, st));
    return DDGEMM_OK;
}

}  // namespace

extern "C" {

ddgemm_status md_gemm_tc_layout(int nparts, int64_t M, int64_t N, int64_t K, int64_t* Mp, int64_t* Np, int64_t* Kp,
                                int* splits) {
    if (md_parts(nparts) == 0) return DDGEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K || !tc_part_rows_ok(M, N, K, md_parts(nparts))) return DDGEMM_ERR_UNSUPPORTED;
    TcLayout L = make_tc_layout(M, N, K, md_parts(nparts));
    if (Mp) *Mp = L.Mp;
    if (Np) *Np = L.Np;
    if (Kp) *Kp = L.Kp;
    if (splits) *splits = L.splits;
    return DDGEMM_OK;
}

ddgemm_status md_gemm_tc_workspace_size(int nparts, int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (md_parts(nparts) == 0) return DDGEMM_ERR_UNSUPPORTED;
    if (bytes == nullptr || M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K || !tc_part_rows_ok(M, N, K, md_parts(nparts))) return DDGEMM_ERR_UNSUPPORTED;
    *bytes = (size_t)make_tc_layout(M, N, K, md_parts(nparts)).total;
    return DDGEMM_OK;
}

ddgemm_status md_gemm_tc(int nparts, int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                         const double* const* B, int64_t ldb, double* const* C, int64_t ldc, void* workspace,
                         size_t workspace_bytes, void* stream) {
    ddgemm_status s = check_tc_md_args(nparts, M, N, K, A, lda, B, ldb, C, ldc);
    if (s != DDGEMM_OK || M == 0 || N == 0) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TcLayout L = make_tc_layout(M, N, K, md_parts(nparts));
    if (workspace != nullptr) {
        if ((uintptr_t)workspace % kAlign != 0 || workspace_bytes < (size_t)L.total) return DDGEMM_ERR_INVALID_ARG;
        return run_md_tc(nparts, L, M, N, K, A, lda, B, ldb, C, ldc, static_cast<char*>(workspace), st);
    }
    void* ws = nullptr;
    if (pool_alloc(&ws, (size_t)L.total, st) != cudaSuccess) {
        cudaGetLastError();
        return DDGEMM_ERR_ALLOC;
    }
    s = run_md_tc(nparts, L, M, N, K, A, lda, B, ldb, C, ldc, static_cast<char*>(ws), st);
    cudaError_t fe = cudaFreeAsync(ws, st);
    if (s == DDGEMM_OK && fe != cudaSuccess) s = DDGEMM_ERR_CUDA;
    return s;
}

ddgemm_status md_split_bf16(int nparts, int64_t M, int64_t N, int64_t K, const double* const* A, int64_t lda,
                            const double* const* B, int64_t ldb, uint16_t* planesA, int32_t* e, uint16_t* planesB,
                            int32_t* f, void* stream) {
    if (md_parts(nparts) == 0) return DDGEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0 || lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N))
        return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if ((M > 0 && (e == nullptr || A == nullptr || (K > 0 && planesA == nullptr))) ||
        (N > 0 && (f == nullptr || B == nullptr || (K > 0 && planesB == nullptr))))
        return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Kp = round_up(K, kTcK);
    return from_cuda(run_split_tc_md(nparts, M, N, K, Kp, M > 0 ? A : nullptr, lda, e, planesA, N > 0 ? B : nullptr,
                                     ldb, f, planesB, static_cast<cudaStream_t>(stream)));
}

ddgemm_status md_slice_gemm_tc(int nparts, int64_t M, int64_t N, int64_t K, const uint16_t* planesA,
                               const uint16_t* planesB, int splits, int32_t* P, void* stream) {
    if (md_parts(nparts) == 0) return DDGEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return DDGEMM_ERR_INVALID_ARG;
    if (K > QDGEMM_MAX_K) return DDGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return DDGEMM_OK;
    const int64_t Mp = round_up(M, kTcM), Np = round_up(N, kTcN), Kp = round_up(K, kTcK), KB = Kp / kTcK;
    if (splits < 1 || splits > kTcMaxSplits || (KB > 0 && splits > KB) || (KB == 0 && splits != 1))
        return DDGEMM_ERR_INVALID_ARG;
    if (KB > 0 && ((KB + splits - 1) / splits) * kTcK > tc_max_k_split(md_parts(nparts))) return DDGEMM_ERR_INVALID_ARG;
    if (!tc_part_rows_ok(M, N, K, md_parts(nparts))) return DDGEMM_ERR_UNSUPPORTED;
    if (P == nullptr || (K > 0 && (planesA == nullptr || planesB == nullptr))) return DDGEMM_ERR_INVALID_ARG;
    if ((uintptr_t)planesA % 16 != 0 || (uintptr_t)planesB % 16 != 0 || (uintptr_t)P % 16 != 0)
        return DDGEMM_ERR_INVALID_ARG;
    return from_cuda(launch_slice_gemm_tc_md(nparts, planesA, planesB, Mp, Np, Kp, splits, P,
                                             static_cast<cudaStream_t>(stream)));
}

ddgemm_status md_recombine_tc(int nparts, int64_t M, int64_t N, const int32_t* P, int splits, const int32_t* e,
                              const int32_t* f, double* const* C, int64_t ldc, void* stream) {
    if (md_parts(nparts) == 0) return DDGEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || ldc < std::max<int64_t>(1, N) || splits < 1 || splits > kTcMaxSplits)
        return DDGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DDGEMM_OK;
    if (P == nullptr || e == nullptr || f == nullptr || C == nullptr) return DDGEMM_ERR_INVALID_ARG;
    for (int p = 0; p < nparts; ++p)
        if (C[p] == nullptr) return DDGEMM_ERR_INVALID_ARG;
    const int64_t Mp = round_up(M, kTcM), Np = round_up(N, kTcN);
    return from_cuda(launch_recombine_tc_md(nparts, P, splits, Mp, Np, e, f, M, N, C, ldc,
                                            static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dd_gemm_noalloc: the product with a fixed, library-owned scratch buffer, for
// callers that cannot allocate device memory while they run.
// ---------------------------------------------------------------------------

namespace {

// The scratch buffer.  In host code this name only stands in for the device
// array: its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DDGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device (looked up on
// the first call for that device).
ddgemm_status noalloc_scratch(char** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();  // leave no error behind for the caller's next CUDA call
        return DDGEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return DDGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return DDGEMM_ERR_CUDA;
        }
        g_noalloc_addr[dev] = p;
    }
    *addr = static_cast<char*>(g_noalloc_addr[dev]);
    return DDGEMM_OK;
}

}  // namespace

extern "C" ddgemm_status dd_gemm_noalloc(int64_t M, int64_t N, int64_t K, const double* A_hi,
                                         const double* A_lo, int64_t lda, const double* B_hi,
                                         const double* B_lo, int64_t ldb, double* C_hi, double* C_lo,
                                         int64_t ldc, void* stream) {
    ddgemm_status s = check_gemm_args(M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc);
    if (s != DDGEMM_OK) return s;
    if (M == 0 || N == 0) return DDGEMM_OK;
    Layout L = make_layout(M, N, K);
    if (L.total > (int64_t)DDGEMM_NOALLOC_SCRATCH_BYTES) return DDGEMM_ERR_TOO_LARGE;
    char* ws = nullptr;
    s = noalloc_scratch(&ws);
    if (s != DDGEMM_OK) return s;
    // Every region of the workspace is written before it is read within the
    // call (exponents by their init kernel, part planes including padding by
    // the split kernels, P by the slice GEMM), so no clearing is needed.
    return run_gemm(L, M, N, K, A_hi, A_lo, lda, B_hi, B_lo, ldb, C_hi, C_lo, ldc, ws,
                    static_cast<cudaStream_t>(stream));
}
