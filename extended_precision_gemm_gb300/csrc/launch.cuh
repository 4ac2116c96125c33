// launch.cuh -- host-side launchers of the dd GEMM kernels (one per step).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace ddg {

// Launch `kernel` on `st` with programmatic stream serialisation: the grid
// may be scheduled before the previous kernel on the stream has finished; the
// kernel must call pdl_wait() (common.cuh) before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Step 1: exponents and part planes.  An operand is A (its rows) or B (its
// columns); `rows` counts rows of A or columns of B; element (r, k) is
// hi[r * ld + k] for A and hi[k * ld + r] for B.  Exponent arrays are
// accumulated with atomicMax (launch_shared_exponents resets them first).
// Either operand may be null.  The split kernels turn the sentinel
// EXP_NONE of an all-zero row into its final exponent 0 in place, unless
// exp_given is set (exponents supplied by the caller, read only).
struct SplitOperand {
    const double* hi;
    const double* lo;
    int64_t ld;
    int64_t rows;
    int32_t* exp;
    bool exp_given;
};
// Set every exponent to `value` (EXP_NONE before launch_exponents when the
// raw maxima, sentinel included, are wanted).
cudaError_t launch_reset_exponents(int32_t* e, int64_t M, int32_t* f, int64_t N, int32_t value,
                                   cudaStream_t st);
// The shared exponents of A's rows and B's columns (either may be null):
// e[i] = smallest e with max_k |A_hi[i,k]| < 2^e, EXP_NONE for a row without
// a nonzero element (a reset, then the atomicMax kernel over k-chunks); with
// K = 0 every exponent is set to zero_k_value.
cudaError_t launch_shared_exponents(const SplitOperand* A, const SplitOperand* B, int64_t K, int32_t zero_k_value,
                                    cudaStream_t st);
cudaError_t launch_exponents(const SplitOperand* A, const SplitOperand* B, int64_t K, cudaStream_t st);
// FP64 parts in the tiled layout of the mma.sync slice GEMM.
cudaError_t launch_split_f64(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                             double* planesA, double* planesB, cudaStream_t st);
// int16 parts for the integer-pipe slice GEMM (layout
// [tile][k-chunk][k in chunk][row in tile][part]).
cudaError_t launch_split_i16(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                             int16_t* planesA, int16_t* planesB, cudaStream_t st);

// Step 2: slice-pair GEMM into `splits` partial sets of 8 planes Mp x Np.
cudaError_t launch_slice_gemm(const double* planesA, const double* planesB, int64_t Mp,
                              int64_t Np, int64_t Kp, int splits, double* P, cudaStream_t st);
int slice_gemm_ctas_per_sm();

// Step 2 with the recombination in the epilogue (one k-split): C directly.
cudaError_t launch_slice_gemm_recombine(const double* planesA, const double* planesB, int64_t Mp, int64_t Np,
                                        int64_t Kp, const int32_t* e, const int32_t* f, int64_t M, int64_t N,
                                        double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st);

// Step 2 with step 1's split fused into the prologue: the parts are formed
// from hi/lo tiles of A (rows, leading dimension lda) and B (K x N, ldb)
// against the exponents e, f (EXP_NONE reads as 0); no part planes.
struct FusedSrc {
    const double* A_hi; const double* A_lo; int64_t lda;
    const double* B_hi; const double* B_lo; int64_t ldb;
    const int32_t* e; const int32_t* f;
    int64_t M, N, K;
    bool a_vec;  // A_hi, A_lo 16-byte aligned and lda even: 16-byte loads
};
FusedSrc make_fused_src(const double* A_hi, const double* A_lo, int64_t lda, const double* B_hi, const double* B_lo,
                        int64_t ldb, const int32_t* e, const int32_t* f, int64_t M, int64_t N, int64_t K);
cudaError_t launch_slice_gemm_fused(const FusedSrc& g, int64_t Mp, int64_t Np, int64_t Kp, int splits, double* P,
                                    cudaStream_t st);
// ... and the recombination in the epilogue as well (one k-split): C directly.
cudaError_t launch_slice_gemm_fused_recombine(const FusedSrc& g, int64_t Mp, int64_t Np, int64_t Kp,
                                              double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st);
int slice_gemm_fused_ctas_per_sm();

// Step 2 on the integer pipe: the same P from int16 parts, exact int64 sums.
cudaError_t launch_slice_gemm_i64(const int16_t* planesA, const int16_t* planesB, int64_t Mp,
                                  int64_t Np, int64_t Kp, int splits, double* P, cudaStream_t st);
int slice_gemm_i64_ctas_per_sm();
cudaError_t read_and_reset_wait_timeouts_i64(unsigned int* count);

// Step 3: recombination of the (split) planes into C = C_hi + C_lo.
cudaError_t launch_recombine(const double* P, int splits, int64_t Mp, int64_t Np,
                             const int32_t* e, const int32_t* f, int64_t M, int64_t N,
                             double* C_hi, double* C_lo, int64_t ldc, cudaStream_t st);

// Rate of a register-only mma.sync.m8n8k4.f64 loop over the whole device
// (TFLOP/s); synchronises `st`.
cudaError_t measure_dmma_roof(double* tflops, cudaStream_t st);

// The comparator: double-double GEMM on the FP64 ALUs, one accumulator per
// output, k in order.
cudaError_t launch_simt_dd_gemm(const double* A_hi, const double* A_lo, int64_t lda, const double* B_hi,
                                const double* B_lo, int64_t ldb, double* C_hi, double* C_lo, int64_t ldc,
                                int64_t M, int64_t N, int64_t K, cudaStream_t st);

// Quad doubles on the integer pipe: 16 int16 parts per element, 136 pairs,
// exact sums rounded once into 4 doubles.  A / B / C are arrays of 4 plane
// pointers.
cudaError_t launch_split_qd(const double* const* A, int64_t lda, int64_t M, const int32_t* e,
                            const double* const* B, int64_t ldb, int64_t N, const int32_t* f, int64_t K,
                            int64_t Kp, int16_t* planesA, int16_t* planesB, cudaStream_t st);
cudaError_t launch_slice_gemm_qd(const int16_t* planesA, const int16_t* planesB, int64_t Mp, int64_t Np,
                                 int64_t Kp, int splits, double* P, cudaStream_t st);
int slice_gemm_qd_ctas_per_sm();
cudaError_t launch_recombine_qd(const double* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                const int32_t* f, int64_t M, int64_t N, double* const* C, int64_t ldc,
                                cudaStream_t st);
cudaError_t read_and_reset_wait_timeouts_qd(unsigned int* count);

// The variant with 8-bit parts on the bf16 tensor cores (tcgen05): 13 bf16
// parts per element in swizzled blocks, 91 pairs accumulated in tensor
// memory, int32 part sums per k-split, exact sum rounded once.
cudaError_t launch_split_bf16(const SplitOperand* A, const SplitOperand* B, int64_t K, int64_t Kp,
                              uint16_t* planesA, uint16_t* planesB, cudaStream_t st);
cudaError_t launch_slice_gemm_tc(const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                 int64_t Kp, int splits, int32_t* P, cudaStream_t st);
cudaError_t launch_recombine_tc(const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                const int32_t* f, int64_t M, int64_t N, double* C_hi, double* C_lo, int64_t ldc,
                                cudaStream_t st);
cudaError_t read_and_reset_wait_timeouts_tc(unsigned int* count);
// CTA pairs of the tensor-core GEMM resident at once (its persistent grid;
// the same for every part count).
int tc_resident_pairs();
// Quad doubles with 27 bf16 parts (same block layout, 378 pairs).
cudaError_t launch_split_bf16_qd(const double* const* A, int64_t lda, int64_t M, int32_t* e, const double* const* B,
                                 int64_t ldb, int64_t N, int32_t* f, int64_t K, int64_t Kp, uint16_t* planesA,
                                 uint16_t* planesB, cudaStream_t st);
cudaError_t launch_slice_gemm_tc_qd(const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                    int64_t Kp, int splits, int32_t* P, cudaStream_t st);
cudaError_t launch_recombine_tc_qd(const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                   const int32_t* f, int64_t M, int64_t N, double* const* C, int64_t ldc,
                                   cudaStream_t st);

// Octo (nin = 8) and hexa (nin = 16) doubles with 54 / 107 bf16 parts.
cudaError_t launch_split_bf16_md(int nin, const double* const* A, int64_t lda, int64_t M, int32_t* e,
                                 const double* const* B, int64_t ldb, int64_t N, int32_t* f, int64_t K, int64_t Kp,
                                 uint16_t* planesA, uint16_t* planesB, cudaStream_t st);
cudaError_t launch_slice_gemm_tc_md(int nin, const uint16_t* planesA, const uint16_t* planesB, int64_t Mp, int64_t Np,
                                    int64_t Kp, int splits, int32_t* P, cudaStream_t st);
cudaError_t launch_recombine_tc_md(int nin, const int32_t* P, int splits, int64_t Mp, int64_t Np, const int32_t* e,
                                   const int32_t* f, int64_t M, int64_t N, double* const* C, int64_t ldc,
                                   cudaStream_t st);
cudaError_t read_and_reset_wait_timeouts_tc_md(unsigned int* count);

// The bounds-check records of the translation units with checks (all zero
// unless the library was built with -DDDGEMM_CHECKED); each synchronises the
// device, reads its record and clears it.
cudaError_t check_record_split(CheckRecord* out);
cudaError_t check_record_slice_gemm(CheckRecord* out);
cudaError_t check_record_fused(CheckRecord* out);
cudaError_t check_record_recombine(CheckRecord* out);
cudaError_t check_record_tc(CheckRecord* out);
cudaError_t check_record_tc_md(CheckRecord* out);

// Diagnostics of the bounded waits inside the slice GEMM.
cudaError_t read_and_reset_wait_timeouts(unsigned int* count);
// The counts of the FP64 slice GEMM / the bf16 dd slice GEMM without
// clearing them, read after the work on `st` (synchronises `st`).
cudaError_t peek_wait_timeouts(unsigned int* count, cudaStream_t st);
cudaError_t peek_wait_timeouts_tc(unsigned int* count, cudaStream_t st);

}  // namespace ddg
