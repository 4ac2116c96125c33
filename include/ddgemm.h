/*
 * ddgemm.h -- double-double matrix product on the FP64 tensor pipe of GB300.
 *
 * C = A * B for double-double matrices (A = A_hi + A_lo, M x K; B = B_hi +
 * B_lo, K x N; C = C_hi + C_lo, M x N), following "Multiple Double Arithmetic
 * on NVIDIA Tensor Cores" (arXiv 2607.06881v1), Section 2: every double
 * double is split into 8 parts of 13 bits ("quarters": 4 of the high double,
 * 4 of the low double), the products of the parts run as ordinary FP64 matrix
 * products that are exact, and the parts of the product are added back into a
 * double double.  Here the 13-bit parts of a row of A (a column of B) share
 * one exponent, so that every part of the row lies on one grid (the balancing
 * goal of Section 3, Problems 3.2 and 3.4).
 *
 * Conventions shared by every entry point below:
 *   - Matrices are row-major.  lda, ldb, ldc are leading dimensions in
 *     elements: lda >= K, ldb >= N, ldc >= N (and >= 1).
 *   - Pointers named d_* / A_hi ... are DEVICE pointers on the current device,
 *     owned by the caller; the library keeps no reference after the call.
 *     Pointers named h_* are host pointers.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) unless stated otherwise.  Argument errors are returned
 *     before anything is launched.  Errors raised by the device surface at the
 *     next synchronising call, as with any CUDA work.
 *   - Inputs must be finite, normalised double doubles (|lo| <= ulp(hi)/2 and
 *     lo = 0 where hi = 0).  Other inputs give unspecified values (no fault,
 *     no hang); they are not checked.
 *   - K <= DDGEMM_MAX_K (2^24): every slice-pair sum then stays below 2^53 and
 *     is exact (the argument of eq. (5) of the paper, for 13-bit parts and
 *     8 index sums).  Larger K returns DDGEMM_ERR_UNSUPPORTED.
 *   - M, N or K = 0 is valid; K = 0 writes C = +0.
 *   - Every wait inside a slice GEMM on its operand copies is bounded in
 *     time.  A block that gives up stops early, leaves its part of the result
 *     incomplete and counts itself in a device counter; the asynchronous
 *     entry points cannot see this and still return DDGEMM_OK.  A result
 *     counts only if dd_wait_timeouts (which synchronises) reads 0 after it;
 *     the blocking host-buffer entry points (dd_gemm_host, dd_gemm_tc_host)
 *     check the counter themselves and return DDGEMM_ERR_CUDA when it is not
 *     0.  (It stays 0 in normal operation.)
 */
#ifndef DDGEMM_H
#define DDGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DDGEMM_SLICES 8          /* parts per double double (4 + 4 quarters) */
#define DDGEMM_DIGIT_BITS 13     /* bits per quarter */
#define DDGEMM_MAX_K (1 << 24)   /* exactness bound on the inner dimension */
#define DDGEMM_TILE_M 32         /* row tile of the part planes of A / of P */
#define DDGEMM_TILE_N 32         /* column tile of the part planes of B / of P */
#define DDGEMM_CHUNK_K 8         /* k-chunk of the part planes */
#define DDGEMM_EXP_NONE (-4096)  /* raw exponent of an all-zero row / column (dd_exponents) */

typedef enum {
    DDGEMM_OK = 0,
    DDGEMM_ERR_INVALID_ARG = 1,  /* bad size, leading dimension, pointer or overlap */
    DDGEMM_ERR_UNSUPPORTED = 2,  /* K beyond DDGEMM_MAX_K */
    DDGEMM_ERR_ALLOC = 3,        /* device allocation failed */
    DDGEMM_ERR_CUDA = 4,         /* a CUDA call or launch failed */
    DDGEMM_ERR_TOO_LARGE = 5     /* needs more scratch than dd_gemm_noalloc's fixed buffer */
} ddgemm_status;

/* Human-readable name of a status code (static string). */
const char* dd_status_string(int status);

/* ------------------------------------------------------------------ */
/* Whole product                                                        */
/* ------------------------------------------------------------------ */

/*
 * Padded extents and the k-split of the slice GEMM chosen for this shape on
 * the current device: Mp = M rounded up to DDGEMM_TILE_M, Np = N rounded up to
 * DDGEMM_TILE_N, Kp = K rounded up to DDGEMM_CHUNK_K; splits >= 1.  Any output
 * pointer may be NULL.
 */
ddgemm_status dd_gemm_layout(int64_t M, int64_t N, int64_t K,
                             int64_t* Mp, int64_t* Np, int64_t* Kp, int* splits);

/* Bytes of device workspace dd_gemm_ws needs for this shape on the current
 * device (written to *bytes). */
ddgemm_status dd_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * C = A * B (double double), caller-provided workspace.
 * The paper's five steps (Section 2): split into 8 parts, rewrite, multiply on
 * the tensor cores, extract, add the parts into a double double; here run as
 * five kernels on `stream`: exponent reset, row / column exponents, split of
 * both operands into part planes, the slice-pair GEMM (FP64 mma.sync), and
 * the recombination.  `workspace` is a device buffer of at least
 * dd_gemm_workspace_size() bytes, 256-byte aligned; its contents on entry do
 * not matter and it must not be used by anything else until the work on
 * `stream` completes.  C must not overlap A, B or the workspace.
 */
ddgemm_status dd_gemm_ws(int64_t M, int64_t N, int64_t K,
                         const double* A_hi, const double* A_lo, int64_t lda,
                         const double* B_hi, const double* B_lo, int64_t ldb,
                         double* C_hi, double* C_lo, int64_t ldc,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * C = A * B (double double).  As dd_gemm_ws, with the workspace taken from the
 * library's stream-ordered memory pool on the current device (allocated and
 * freed on `stream`).  The pool keeps freed memory for the next call instead
 * of unmapping it at every synchronisation (mapping gigabytes anew on every
 * call costs a visible part of a product); dd_pool_trim returns it to the
 * device.  Every entry point below whose workspace may be NULL, and the
 * host-buffer entry points, allocate from the same pool.  Returns
 * DDGEMM_ERR_ALLOC when the allocation fails.
 */
ddgemm_status dd_gemm(int64_t M, int64_t N, int64_t K,
                      const double* A_hi, const double* A_lo, int64_t lda,
                      const double* B_hi, const double* B_lo, int64_t ldb,
                      double* C_hi, double* C_lo, int64_t ldc, void* stream);

/*
 * C = A * B with HOST operands and result: copies A and B to the current
 * device, runs dd_gemm, copies C back, and returns only after the result is
 * in h_C_hi / h_C_lo (it synchronises `stream`).  Host buffers are read and
 * written as dense row-major arrays with the given leading dimensions;
 * page-locked (pinned) buffers make the copies faster.  The device memory of
 * the call (dense copies of A, B and C plus the workspace) comes from the
 * library's pool (see dd_gemm); dd_pool_trim returns it to the device.
 */
ddgemm_status dd_gemm_host(int64_t M, int64_t N, int64_t K,
                           const double* h_A_hi, const double* h_A_lo, int64_t lda,
                           const double* h_B_hi, const double* h_B_lo, int64_t ldb,
                           double* h_C_hi, double* h_C_lo, int64_t ldc, void* stream);

/*
 * Options of dd_gemm_ex.  A zero-initialised struct (or a NULL pointer) asks
 * for what dd_gemm does.
 *   slices:         parts per double double: 0 or 8 (the only count built;
 *                   other values return DDGEMM_ERR_UNSUPPORTED).
 *   pairs:          part pairs kept: 0 or 36, every pair with index sum
 *                   s + t <= 7 (others: DDGEMM_ERR_UNSUPPORTED).
 *   split_k:        k-splits of the slice GEMM: 0 = automatic (as
 *                   dd_gemm_layout), else 1 .. min(64, Kp / 8) (1 when K = 0);
 *                   any count gives the same result bit for bit.
 *   fuse_recombine: 1 = the recombination (steps 4-5 of Section 2) runs in
 *                   the slice GEMM's epilogue, which writes C directly: no
 *                   part-sum planes P.  It needs all of k in one block: with
 *                   split_k = 1 it always applies; with split_k = 0 it applies
 *                   when the automatic choice is one split (dd_gemm_ex_plan
 *                   tells); split_k > 1 returns DDGEMM_ERR_UNSUPPORTED.
 *   fuse_split:     1 = the 13-bit parts are formed inside the slice GEMM from
 *                   hi/lo tiles of A and B (the conversion pipelined behind
 *                   the MMAs; "Ozaki 2.5: Engineering the Deconstruction Path
 *                   of fp64-Emulated Dense Matrix Multiplication on FP8 Tensor
 *                   Cores", summary): no part planes.  The exponents are still
 *                   found first (one pass over A_hi and B_hi).
 * Every combination gives C identical bit for bit to dd_gemm's.
 */
typedef struct {
    int slices;
    int pairs;
    int split_k;
    int fuse_recombine;
    int fuse_split;
} ddgemm_opts;

/*
 * What dd_gemm_ex does with these options for this shape on the current
 * device: its workspace bytes, its k-split count, and whether the
 * recombination runs in the slice GEMM (1) or as its own kernel (0).  Any
 * output pointer may be NULL.  Errors as dd_gemm_ex's option checks.
 */
ddgemm_status dd_gemm_ex_plan(int64_t M, int64_t N, int64_t K, const ddgemm_opts* opts,
                              size_t* workspace_bytes, int* splits, int* fused_recombine);

/*
 * C = A * B (double double) with options (ddgemm_opts; NULL = defaults).
 * `workspace` (dd_gemm_ex_plan's bytes, 256-byte aligned) may be NULL: then
 * it comes from the library's pool (see dd_gemm; DDGEMM_ERR_ALLOC on failure).
 * With both fusions the workspace holds only the exponents (4 (Mp + Np)
 * bytes).  Otherwise as dd_gemm_ws.
 */
ddgemm_status dd_gemm_ex(int64_t M, int64_t N, int64_t K,
                         const double* A_hi, const double* A_lo, int64_t lda,
                         const double* B_hi, const double* B_lo, int64_t ldb,
                         double* C_hi, double* C_lo, int64_t ldc,
                         const ddgemm_opts* opts, void* workspace, size_t workspace_bytes, void* stream);

/*
 * C = A * B (double double) without allocating any memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that must not allocate device memory while they run: an application that
 * hands all GPU memory to its own allocator at start-up, a plug-in whose host
 * forbids allocations, or a latency-critical loop where cudaMalloc / cudaFree
 * could wait for the whole device.  Instead of a workspace it uses one fixed
 * scratch buffer of DDGEMM_NOALLOC_SCRATCH_BYTES (64 MiB), a static device
 * array of the library; every GPU on which the library's device code is
 * loaded holds that buffer until the process exits.
 *
 * Same arguments and results as dd_gemm.  Shapes whose workspace
 * (dd_gemm_workspace_size) exceeds the buffer return DDGEMM_ERR_TOO_LARGE
 * before anything runs; M = N = K = 256 fits, for example.
 * The first call on a device looks up the buffer's device address
 * (cudaGetSymbolAddress, which may also make the driver load the module that
 * holds it); make that first call on each device before any stream capture.
 * All calls on a device share the one buffer, which keeps whatever the last
 * call left in it.  Each call writes every part of the buffer it reads before
 * reading it, so leftovers never change a result and nothing needs clearing;
 * but calls whose work can overlap on the same GPU (issued on different
 * streams, or from different host threads) race on the buffer: order them,
 * for example by issuing them on one stream.  Device ordinals 0..63 are
 * served; a current device of 64 or more returns DDGEMM_ERR_CUDA.
 */
#define DDGEMM_NOALLOC_SCRATCH_BYTES (64u << 20)
ddgemm_status dd_gemm_noalloc(int64_t M, int64_t N, int64_t K,
                              const double* A_hi, const double* A_lo, int64_t lda,
                              const double* B_hi, const double* B_lo, int64_t ldb,
                              double* C_hi, double* C_lo, int64_t ldc, void* stream);

/*
 * Return the device memory the library's pool keeps on the current device
 * (workspaces of calls without one, device copies of the host-buffer entry
 * points) to the device; synchronises the device.  DDGEMM_OK also when
 * nothing was allocated on it.
 */
ddgemm_status dd_pool_trim(void);

/* ------------------------------------------------------------------ */
/* The steps of the path, one entry point each                          */
/* ------------------------------------------------------------------ */

/*
 * Step 1a (rows of A): shared exponents and part planes.
 *   e[i] = smallest integer with max_k |A_hi[i,k]| < 2^e[i]; 0 for a zero row.
 *   The parts of x = A_hi[i,k] + A_lo[i,k] are the 8 truncating base-2^13
 *   digits of |x| * 2^-e[i], most significant first, with the sign of x:
 *       x * 2^-e[i] = sum_s D_s 2^(-13 (s+1)) + r,   |r| < 2^-104,
 *   each D_s an integer in (-2^13, 2^13) stored as a double (the quarters of
 *   Section 2 of the paper, on a grid shared by the row).  When hi and lo
 *   have opposite signs the truncation of their sum borrows from the higher
 *   digits, the value-preserving move of Problem 3.3, eq. (7).
 * Output layout (tiled for the slice GEMM; entries outside M x K are 0):
 *   planes[((((mt * KC + kc) * 8 + s) * 2 + q) * 32 + mi) * 4 + r]
 *     holds D_s of element (i, k) with mt = i / 32, mi = i % 32,
 *     kc = k / 8, q = (k % 8) / 4, r = k % 4, KC = Kp / 8
 *   (8 * Mp * Kp doubles; Mp, Kp from dd_gemm_layout).  e: M int32.
 */
ddgemm_status dd_split_rows(int64_t M, int64_t K,
                            const double* A_hi, const double* A_lo, int64_t lda,
                            double* planes, int32_t* e, void* stream);

/*
 * Step 1b (columns of B): as dd_split_rows, for the columns of B (K x N,
 * row-major, leading dimension ldb): f[j] from max_k |B_hi[k,j]|, and
 *   planes[((((nt * KC + kc) * 8 + t) * 2 + q) * 32 + ni) * 4 + r]
 *     holds D_t of element (k, j) with nt = j / 32, ni = j % 32
 *   (8 * Np * Kp doubles).  f: N int32.
 */
ddgemm_status dd_split_cols(int64_t K, int64_t N,
                            const double* B_hi, const double* B_lo, int64_t ldb,
                            double* planes, int32_t* f, void* stream);

/*
 * Step 1 for both operands at once (what dd_gemm runs): dd_split_rows on A
 * and dd_split_cols on B, in three launches (exponent reset, exponents of
 * both, split of both).  Same outputs and layouts as the two calls.
 */
ddgemm_status dd_split(int64_t M, int64_t N, int64_t K,
                       const double* A_hi, const double* A_lo, int64_t lda,
                       const double* B_hi, const double* B_lo, int64_t ldb,
                       double* planesA, int32_t* e, double* planesB, int32_t* f, void* stream);

/*
 * The k-split of the product across devices or passes (each holds a slab of
 * the inner dimension: columns k0..k1-1 of A and the same rows of B).  The
 * paper's method splits each row of A / column of B on one exponent grid
 * (Section 2; Problems 3.2 and 3.4 of Section 3); for the slab products to add
 * up to the unsplit ones every slab must use the exponents of the WHOLE row /
 * column, the maximum over the slabs.  Pattern: dd_exponents on each slab ->
 * elementwise MAX of the e (and f) arrays over the slabs (an all-reduce MAX
 * across devices) -> dd_split_with_exponents on each slab with those maxima
 * -> dd_slice_gemm on each slab -> the P of all slabs, side by side as
 * k-splits (or summed: an all-reduce SUM, exact because every partial sum is
 * an integer below 2^53) -> one dd_recombine with the same maxima.  The
 * result is identical bit for bit to dd_gemm on the unsplit operands.
 *
 * dd_exponents: the raw shared exponents of the rows of A (e, M int32) and
 *   the columns of B (f, N int32): e[i] = smallest integer with
 *   max_k |A_hi[i,k]| < 2^e[i], and DDGEMM_EXP_NONE (below every other value)
 *   for a row without a nonzero element, including every row when K = 0, so
 *   that the elementwise maximum over slabs is the exponent of the whole row.
 *   M = 0 (N = 0) skips A (B); A_hi / B_hi may then be NULL.
 * dd_split_with_exponents: the part planes of dd_split_rows / dd_split_cols
 *   (same layouts) against caller-supplied exponents e, f (read only; a value
 *   of DDGEMM_EXP_NONE stands for 0).  Every e[i] must be at least the
 *   exponent of row i of this slab (the maximum over slabs is), otherwise the
 *   parts are unspecified (no fault).  M = 0 (N = 0) skips A (B).
 * Errors as for dd_split.  Both are asynchronous on `stream`.
 */
ddgemm_status dd_exponents(int64_t M, int64_t N, int64_t K,
                           const double* A_hi, int64_t lda, const double* B_hi, int64_t ldb,
                           int32_t* e, int32_t* f, void* stream);
ddgemm_status dd_split_with_exponents(int64_t M, int64_t N, int64_t K,
                                      const double* A_hi, const double* A_lo, int64_t lda,
                                      const double* B_hi, const double* B_lo, int64_t ldb,
                                      const int32_t* e, const int32_t* f,
                                      double* planesA, double* planesB, void* stream);

/*
 * Step 2 (slice-pair GEMM, eqs. (3)-(4) of the paper grouped by index sum):
 *   P[z][d][i][j] = sum_{s+t=d} sum_{k in split z} A_s[i,k] * B_t[k,j],
 *   d = 0..7, for the 36 pairs s + t <= 7, on the FP64 tensor pipe
 *   (mma.sync m8n8k4 f64), with every sum an exact integer below 2^53.
 * planesA / planesB: the outputs of dd_split_rows / dd_split_cols for the same
 * M, N, K.  P: splits x 8 x Mp x Np doubles, row-major per plane; split z
 * covers the k-chunks [z * KC / splits, (z + 1) * KC / splits).  splits must
 * be in [1, KC] (or 1 when KC = 0); dd_gemm_layout gives the automatic choice.
 */
ddgemm_status dd_slice_gemm(int64_t M, int64_t N, int64_t K,
                            const double* planesA, const double* planesB,
                            int splits, double* P, void* stream);

/*
 * Step 2 with step 1's split fused in: P exactly as dd_slice_gemm produces
 * from dd_split's planes, but the parts are formed inside the GEMM from the
 * hi/lo of A (M x K, lda) and B (K x N, ldb) against the exponents e (M) and
 * f (N) -- from dd_split, dd_exponents, or the maximum over k-slabs of
 * dd_exponents (DDGEMM_EXP_NONE reads as 0; see dd_split_with_exponents for
 * the contract on slab exponents).  P: splits x 8 x Mp x Np doubles, 16-byte
 * aligned; splits as for dd_slice_gemm.  No part planes are read or written.
 */
ddgemm_status dd_slice_gemm_fused(int64_t M, int64_t N, int64_t K,
                                  const double* A_hi, const double* A_lo, int64_t lda,
                                  const double* B_hi, const double* B_lo, int64_t ldb,
                                  const int32_t* e, const int32_t* f,
                                  int splits, double* P, void* stream);

/*
 * Step 3 (recombination, steps 4-5 of the paper's algorithm):
 *   P_d = sum_z P[z][d][i][j] (exact), then, from d = 7 down to 0,
 *   (h, l) <- quick_two_sum(two_sum(h, P_d 2^(-13(d+2))) with l added to its
 *   error), starting from h = P_7 2^-117, l = 0; finally
 *   C_hi = h * 2^(e[i] + f[j]), C_lo = l * 2^(e[i] + f[j]) (ldexp, correctly
 *   rounded; +0 for zero).  P as produced by dd_slice_gemm.
 */
ddgemm_status dd_recombine(int64_t M, int64_t N, const double* P, int splits,
                           const int32_t* e, const int32_t* f,
                           double* C_hi, double* C_lo, int64_t ldc, void* stream);

/* ------------------------------------------------------------------ */
/* Comparator                                                           */
/* ------------------------------------------------------------------ */

/*
 * C = A * B with plain double-double arithmetic on the FP64 ALUs, no
 * splitting: the second method of Section 4.2 of the paper (one thread per
 * inner product, double-double multiply and add).  Per k, in order:
 *   p = a_hi b_hi; e = fma(a_hi, b_hi, -p); e += a_hi b_lo + a_lo b_hi;
 *   (s, t) = two_sum(c_hi, p); t = (t + c_lo) + e;
 *   (c_hi, c_lo) = quick_two_sum(s, t).
 * Not the method under evaluation: it is the reference point the paper
 * compares against.  Same argument checks as dd_gemm (including K <=
 * DDGEMM_MAX_K); M <= 2097120.
 */
ddgemm_status dd_gemm_simt(int64_t M, int64_t N, int64_t K,
                           const double* A_hi, const double* A_lo, int64_t lda,
                           const double* B_hi, const double* B_lo, int64_t ldb,
                           double* C_hi, double* C_lo, int64_t ldc, void* stream);

/* ------------------------------------------------------------------ */
/* Integer-pipe variant of the slice-pair GEMM                          */
/* ------------------------------------------------------------------ */

/*
 * The same product, with the slice-pair GEMM (step 2) on the integer pipe:
 * the 13-bit parts are stored as int16 and every pair product is a 32-bit
 * integer multiply-add into an int32 partial sum, added into an exact int64
 * total before it could overflow.  The paper
 * runs these products on FP64 tensor cores because they are exact there
 * (eq. (5)); on GB300 the FP64 pipe, which also executes mma.sync f64, is the
 * narrowest unit, while the exactness needs only integer arithmetic.  The
 * part sums P_d are the same integers, so C is identical bit for bit to
 * dd_gemm's.
 *
 * dd_gemm_i64: as dd_gemm_ws; `workspace` may be NULL, in which case it is
 * taken from the library's pool (see dd_gemm; DDGEMM_ERR_ALLOC on failure).
 * dd_gemm_i64_workspace_size / dd_gemm_i64_layout: its workspace bytes and
 * automatic k-split for this shape on the current device.
 */
ddgemm_status dd_gemm_i64_layout(int64_t M, int64_t N, int64_t K, int* splits);
ddgemm_status dd_gemm_i64_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);
ddgemm_status dd_gemm_i64(int64_t M, int64_t N, int64_t K,
                          const double* A_hi, const double* A_lo, int64_t lda,
                          const double* B_hi, const double* B_lo, int64_t ldb,
                          double* C_hi, double* C_lo, int64_t ldc,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Step 1 for the integer pipe: exponents e (f) exactly as dd_split_rows
 * (dd_split_cols), parts as int16 in the layout
 *   planes[((((tile * KC + kc) * 8 + kk) * 32 + ti) * 8) + s]
 * holding D_s of element (row or column tile * 32 + ti, k = kc * 8 + kk)
 * (8 * Mp * Kp int16 for A, 8 * Np * Kp for B; 0 outside the matrix).
 */
ddgemm_status dd_split_rows_i16(int64_t M, int64_t K,
                                const double* A_hi, const double* A_lo, int64_t lda,
                                int16_t* planes, int32_t* e, void* stream);
ddgemm_status dd_split_cols_i16(int64_t K, int64_t N,
                                const double* B_hi, const double* B_lo, int64_t ldb,
                                int16_t* planes, int32_t* f, void* stream);

/* Both operands at once, as dd_split, with int16 parts. */
ddgemm_status dd_split_i16(int64_t M, int64_t N, int64_t K,
                           const double* A_hi, const double* A_lo, int64_t lda,
                           const double* B_hi, const double* B_lo, int64_t ldb,
                           int16_t* planesA, int32_t* e, int16_t* planesB, int32_t* f, void* stream);

/*
 * Step 2 on the integer pipe: P exactly as dd_slice_gemm (splits x 8 x Mp x
 * Np doubles holding the int64 sums, which are below 2^53), from the int16
 * part planes of dd_split_rows_i16 / dd_split_cols_i16.
 */
ddgemm_status dd_slice_gemm_i64(int64_t M, int64_t N, int64_t K,
                                const int16_t* planesA, const int16_t* planesB,
                                int splits, double* P, void* stream);

/* ------------------------------------------------------------------ */
/* Quad doubles (4 doubles per number) on the integer pipe              */
/* ------------------------------------------------------------------ */

/*
 * C = A * B for quad-double matrices: every number is x0 + x1 + x2 + x3, four
 * non-overlapping doubles (|x_{p+1}| <= ulp(x_p)/2), passed as four row-major
 * planes sharing one leading dimension (A, B, C: host arrays of 4 device
 * pointers).  The method of Section 2 of the paper for more parts ("a
 * quartered quad double matrix has 16 times the size", Table 2): 16 parts of
 * 13 bits on a shared row / column exponent, the 136 index-sum pairs
 * s + t <= 15 as exact integer sums on the integer pipe, and the 16 parts of
 * the product summed exactly and rounded once into four doubles
 * (c0 = RN(X), c1 = RN(X - c0), ...).  K <= QDGEMM_MAX_K (2^23) keeps every
 * part sum below 2^53.  `workspace` (qd_gemm_workspace_size bytes, 256-byte
 * aligned) may be NULL: then it comes from the library's pool (see dd_gemm).
 */
#define QDGEMM_MAX_K (1 << 23)
ddgemm_status qd_gemm_layout(int64_t M, int64_t N, int64_t K, int* splits);
ddgemm_status qd_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);
ddgemm_status qd_gemm(int64_t M, int64_t N, int64_t K,
                      const double* const* A, int64_t lda,
                      const double* const* B, int64_t ldb,
                      double* const* C, int64_t ldc,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * The steps of qd_gemm.  qd_split: exponents e (M) and f (N) as for double
 * doubles (from the leading planes) and the 16 int16 parts of every element,
 * layout planes[((((tile * KC + kc) * 8 + kk) * 32 + ti) * 16) + s]
 * (16 * Mp * Kp int16 for A, 16 * Np * Kp for B).  qd_slice_gemm: P
 * (splits x 16 x Mp x Np doubles holding exact integers).  qd_recombine: the
 * four output planes from P and the exponents.
 */
ddgemm_status qd_split(int64_t M, int64_t N, int64_t K,
                       const double* const* A, int64_t lda, const double* const* B, int64_t ldb,
                       int16_t* planesA, int32_t* e, int16_t* planesB, int32_t* f, void* stream);
ddgemm_status qd_slice_gemm(int64_t M, int64_t N, int64_t K, const int16_t* planesA,
                            const int16_t* planesB, int splits, double* P, void* stream);
ddgemm_status qd_recombine(int64_t M, int64_t N, const double* P, int splits, const int32_t* e,
                           const int32_t* f, double* const* C, int64_t ldc, void* stream);

/* ------------------------------------------------------------------ */
/* Double doubles with 8-bit parts on the bf16 tensor cores (tcgen05)   */
/* ------------------------------------------------------------------ */

/*
 * C = A * B (double double) with the slice-pair products on GB300's bf16
 * tensor cores.  The paper relates its rewriting to the Ozaki scheme, which
 * computes accurate products with lower precision arithmetic (Section 1), and
 * its exactness argument (Section 2, eqs. (1)-(5)) only needs parts with few
 * nonzero bits on a shared grid; "Ozaki 2.5: Engineering the Deconstruction
 * Path of fp64-Emulated Dense Matrix Multiplication on FP8 Tensor Cores"
 * (summary) applies the idea to 8-bit tensor pipes.  The paper has no bf16
 * variant; this one keeps its steps and changes the width of a part:
 *   - shared exponent e' = e + 1 (e as for dd_gemm, one bit of headroom);
 *     X = trunc((hi + lo) 2^(104 - e')); 13 balanced base-256 digits of X
 *     (least significant first, D = ((X + 128) mod 256) - 128, the top digit
 *     the rest): every part is an integer in [-128, 128], exact in bf16;
 *   - P_d = sum_{s+t=d} A_s B_t for d = 0..12 (91 pairs) with tcgen05.mma
 *     (bf16 in, f32 accumulators in tensor memory), exact: 1024 products of
 *     at most 2^14 are summed in f32 (every partial sum an integer of at most
 *     2^24) and then added into exact int32 totals;
 *   - Z = sum_d P_d 2^(8 (12 - d)) (exact) rounded once to the nearest double
 *     double of Z 2^(e'_i + f'_j - 112) (ties to even; zeros are +0).
 * Its result is not bit-identical to dd_gemm's (other parts, one rounding);
 * both are within the same normwise bound of the exact product.
 * Same arguments and conventions as dd_gemm; K <= DDGEMM_MAX_K.  `workspace`
 * (dd_gemm_tc_workspace_size bytes, 256-byte aligned) may be NULL: then it
 * comes from the library's pool (see dd_gemm; DDGEMM_ERR_ALLOC on failure).
 */
#define DDGEMM_TC_SLICES 13         /* parts per double double */
#define DDGEMM_TC_DIGIT_BITS 8      /* bits per part */
#define DDGEMM_TC_TILE_M 256        /* rows of C per output block (a CTA pair); Mp is a multiple */
#define DDGEMM_TC_BLOCK_M 128       /* rows of A per part block */
#define DDGEMM_TC_TILE_N 256        /* columns of B per part block / of C per output block */
#define DDGEMM_TC_CHUNK_K 64        /* k per part block (one 128-byte row) */
#define DDGEMM_TC_MAX_K_SPLIT 8192  /* k per slice-GEMM block: int32 part sums stay exact */
#define DDGEMM_TC_QD_SLICES 27      /* parts per quad double (216 bits) */
#define DDGEMM_TC_QD_MAX_K_SPLIT 4096 /* k per slice-GEMM block for quad doubles */
#define DDGEMM_TC_OD_SLICES 54      /* parts per octo double (432 bits) */
#define DDGEMM_TC_HD_SLICES 107     /* parts per hexa double (856 bits) */

/*
 * Padded extents (Mp = M rounded up to 256, Np = N rounded up to 256, Kp = K
 * rounded up to 64) and the k-split of the slice GEMM (every split covers at
 * most DDGEMM_TC_MAX_K_SPLIT of k; more splits only where they balance the
 * persistent CTA pairs of the GEMM, e.g. for long K over few output blocks).
 * Any output pointer may be NULL.  DDGEMM_ERR_UNSUPPORTED for K >
 * DDGEMM_MAX_K, or when Mp (or Np) x parts x Kp / 64 reaches 2^31: the
 * tensor copies address the part blocks as 128-byte rows with 32-bit
 * coordinates (2^31 rows are 256 GiB of parts).  The same limits apply to the
 * quad- and multiple-double variants below with their part counts.
 */
ddgemm_status dd_gemm_tc_layout(int64_t M, int64_t N, int64_t K,
                                int64_t* Mp, int64_t* Np, int64_t* Kp, int* splits);
ddgemm_status dd_gemm_tc_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);
ddgemm_status dd_gemm_tc(int64_t M, int64_t N, int64_t K,
                         const double* A_hi, const double* A_lo, int64_t lda,
                         const double* B_hi, const double* B_lo, int64_t ldb,
                         double* C_hi, double* C_lo, int64_t ldc,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * dd_gemm_tc with HOST operands and result, as dd_gemm_host: copies A and B
 * to the current device (memory from the library's pool, see dd_gemm),
 * runs dd_gemm_tc, copies C back, and returns after the result is in h_C_hi /
 * h_C_lo (it synchronises `stream`).  Pinned host buffers make the copies
 * faster.
 */
ddgemm_status dd_gemm_tc_host(int64_t M, int64_t N, int64_t K,
                              const double* h_A_hi, const double* h_A_lo, int64_t lda,
                              const double* h_B_hi, const double* h_B_lo, int64_t ldb,
                              double* h_C_hi, double* h_C_lo, int64_t ldc, void* stream);

/*
 * The steps of dd_gemm_tc (all device pointers; used by the parity tests).
 *
 * dd_split_bf16: e (M int32) and f (N int32) receive the exponents e, f of
 * dd_split (the parts use e + 1, f + 1), and the parts as bf16 bit patterns:
 *   planesA: 13 * Mp * Kp uint16, block (mb, s, kb) of 128 x 64 (rows
 *            128 mb .. 128 mb + 127) at element ((mb * 13 + s) * (Kp / 64) + kb) * 8192;
 *   planesB: 13 * Np * Kp uint16, block (nt, t, kb) of 256 x 64 at element
 *            ((nt * 13 + t) * (Kp / 64) + kb) * 16384;
 *   inside a block, element (row r, k) is at byte
 *            r * 128 + (((k / 8) ^ (r % 8)) * 16) + (k % 8) * 2
 *   (rows of B's blocks are columns of B; padding rows / k hold 0).
 * dd_slice_gemm_tc: P, splits x 13 x Mp x Np int32 (row-major Mp x Np per
 *   split and part): the exact part sums of each k-split; splits as given by
 *   dd_gemm_tc_layout (1 <= splits, and ceil(Kp/64 / splits) * 64 <= 8192).
 *   planesA, planesB and P must be 16-byte aligned (tensor copies read the
 *   parts, 16-byte stores write P); any split count in that range gives the
 *   same sums.
 * dd_recombine_tc: C from P and the exponents of dd_split_bf16 (P of any
 *   alignment; 16-byte aligned P and C are read and written 16 bytes at a
 *   time).
 * Errors as for the dd_gemm steps.
 */
ddgemm_status dd_split_bf16(int64_t M, int64_t N, int64_t K,
                            const double* A_hi, const double* A_lo, int64_t lda,
                            const double* B_hi, const double* B_lo, int64_t ldb,
                            uint16_t* planesA, int32_t* e, uint16_t* planesB, int32_t* f, void* stream);
/*
 * The k-split of the bf16 variant across slabs (see dd_exponents): the parts
 * of dd_split_bf16 (same layouts; exponents plus one bit of headroom) against
 * caller-supplied exponents e, f in the form dd_exponents returns (the
 * maximum over the slabs; DDGEMM_EXP_NONE stands for 0).  The int32 part sums
 * of the slabs, side by side as k-splits, go to one dd_recombine_tc with the
 * same e, f; the result equals dd_gemm_tc's bit for bit.
 */
ddgemm_status dd_split_bf16_with_exponents(int64_t M, int64_t N, int64_t K,
                                           const double* A_hi, const double* A_lo, int64_t lda,
                                           const double* B_hi, const double* B_lo, int64_t ldb,
                                           const int32_t* e, const int32_t* f,
                                           uint16_t* planesA, uint16_t* planesB, void* stream);
ddgemm_status dd_slice_gemm_tc(int64_t M, int64_t N, int64_t K, const uint16_t* planesA,
                               const uint16_t* planesB, int splits, int32_t* P, void* stream);
ddgemm_status dd_recombine_tc(int64_t M, int64_t N, const int32_t* P, int splits, const int32_t* e,
                              const int32_t* f, double* C_hi, double* C_lo, int64_t ldc, void* stream);

/*
 * Quad doubles (four doubles per number, as for qd_gemm) with the parts on the
 * bf16 tensor cores: the scheme of dd_gemm_tc with 27 balanced 8-bit parts
 * (X = trunc(x 2^(216 - e')) for x the sum of the four doubles, e' = e + 1 with
 * e from the leading doubles), the 378 pairs s + t <= 26 with tcgen05.mma on
 * CTA pairs, and the exact sum of the 27 part sums rounded once into four
 * non-overlapping doubles (c0 = RN(X), c1 = RN(X - c0), ...).  The paper
 * applies its rewriting to general multiple doubles (Section 2, Tables 1-2);
 * this is that rewriting with 8-bit parts.  Arguments as qd_gemm;
 * K <= QDGEMM_MAX_K; a k-split covers at most DDGEMM_TC_QD_MAX_K_SPLIT of k.
 * Steps: qd_split_bf16 (parts in the block layout of dd_split_bf16 with 27
 * parts), qd_slice_gemm_tc (P: splits x 27 x Mp x Np int32), qd_recombine_tc.
 */
ddgemm_status qd_gemm_tc_layout(int64_t M, int64_t N, int64_t K,
                                int64_t* Mp, int64_t* Np, int64_t* Kp, int* splits);
ddgemm_status qd_gemm_tc_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);
ddgemm_status qd_gemm_tc(int64_t M, int64_t N, int64_t K,
                         const double* const* A, int64_t lda,
                         const double* const* B, int64_t ldb,
                         double* const* C, int64_t ldc,
                         void* workspace, size_t workspace_bytes, void* stream);
ddgemm_status qd_split_bf16(int64_t M, int64_t N, int64_t K,
                            const double* const* A, int64_t lda, const double* const* B, int64_t ldb,
                            uint16_t* planesA, int32_t* e, uint16_t* planesB, int32_t* f, void* stream);
ddgemm_status qd_slice_gemm_tc(int64_t M, int64_t N, int64_t K, const uint16_t* planesA,
                               const uint16_t* planesB, int splits, int32_t* P, void* stream);
ddgemm_status qd_recombine_tc(int64_t M, int64_t N, const int32_t* P, int splits, const int32_t* e,
                              const int32_t* f, double* const* C, int64_t ldc, void* stream);

/*
 * Octo doubles (nparts = 8) and hexa doubles (nparts = 16) with the parts on
 * the bf16 tensor cores: the scheme of qd_gemm_tc with DDGEMM_TC_OD_SLICES =
 * 54 / DDGEMM_TC_HD_SLICES = 107 balanced 8-bit parts (X = trunc(x 2^(8 NP -
 * e'))), the NP (NP + 1) / 2 pairs (1485 / 5778) on the tensor cores, and the
 * exact sum of the part sums rounded once into nparts non-overlapping doubles
 * (with gradual underflow; a zero or infinite part ends the expansion and the
 * rest are +0).  The paper's Table 2 gives the dimensions of quartered octo
 * and hexa doubles.  A, B, C are host arrays of nparts device pointers to
 * row-major planes sharing one leading dimension.  K <= QDGEMM_MAX_K; a
 * k-split covers at most 2048 (octo) / 1024 (hexa) of k.  Other nparts values
 * return DDGEMM_ERR_UNSUPPORTED (quad doubles: qd_gemm_tc; double doubles:
 * dd_gemm_tc).  Steps as for quad doubles, with NP parts.
 */
ddgemm_status md_gemm_tc_layout(int nparts, int64_t M, int64_t N, int64_t K,
                                int64_t* Mp, int64_t* Np, int64_t* Kp, int* splits);
ddgemm_status md_gemm_tc_workspace_size(int nparts, int64_t M, int64_t N, int64_t K, size_t* bytes);
ddgemm_status md_gemm_tc(int nparts, int64_t M, int64_t N, int64_t K,
                         const double* const* A, int64_t lda,
                         const double* const* B, int64_t ldb,
                         double* const* C, int64_t ldc,
                         void* workspace, size_t workspace_bytes, void* stream);
ddgemm_status md_split_bf16(int nparts, int64_t M, int64_t N, int64_t K,
                            const double* const* A, int64_t lda, const double* const* B, int64_t ldb,
                            uint16_t* planesA, int32_t* e, uint16_t* planesB, int32_t* f, void* stream);
ddgemm_status md_slice_gemm_tc(int nparts, int64_t M, int64_t N, int64_t K, const uint16_t* planesA,
                               const uint16_t* planesB, int splits, int32_t* P, void* stream);
ddgemm_status md_recombine_tc(int nparts, int64_t M, int64_t N, const int32_t* P, int splits, const int32_t* e,
                              const int32_t* f, double* const* C, int64_t ldc, void* stream);

/* ------------------------------------------------------------------ */
/* Diagnostics                                                          */
/* ------------------------------------------------------------------ */

/*
 * Measured rate of the FP64 tensor pipe on the current device, in TFLOP/s
 * (2 * 8 * 8 * 4 flops per mma.sync.m8n8k4.f64): a register-only loop of
 * that instruction on every SM, timed with CUDA events on `stream`.  This is
 * the roof of the slice-pair GEMM.  Synchronises `stream`.
 */
ddgemm_status dd_fp64_tensor_roof(double* tflops, void* stream);

/*
 * The bounds-checked build.  libddgemm_checked.so (the same sources compiled
 * with -DDDGEMM_CHECKED) tests the global accesses of the split, slice-GEMM
 * and recombination kernels of the double-double paths (FP64 planes, fused,
 * bf16 tensor cores) against the extents of their buffers before making
 * them: an access out of bounds is skipped (its result is wrong, nothing
 * faults) and counted, and the first one is recorded.  It stands in for a
 * memory checker where none can run.  dd_checked_build returns 1 in that
 * library and 0 in libddgemm.so.  dd_check_report synchronises the device
 * and returns, since its previous call, the number of accesses refused
 * (*count), the check site of the first one (*site: 1xx split, 2xx slice
 * GEMM, 3xx recombination, 4xx fused GEMM, 5xx-7xx bf16 split, recombination
 * and GEMM, 8xx exponents) and its element offset (*index); all zero in the
 * normal build.
 */
int dd_checked_build(void);
ddgemm_status dd_check_report(unsigned int* count, unsigned int* site, int64_t* index);

/*
 * Number of times a slice-GEMM thread block (any variant) gave up waiting
 * for its operand copies on the current device (each wait is bounded in time; a block that
 * gives up stops early and its P tile is incomplete).  Synchronises the
 * device, reads the counter and resets it to 0.  Zero in normal operation.
 */
ddgemm_status dd_wait_timeouts(unsigned int* count);

#ifdef __cplusplus
}
#endif

#endif /* DDGEMM_H */
