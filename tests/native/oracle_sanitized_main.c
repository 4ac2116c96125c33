/* Drives the exact oracle (oracle/exact_ddgemm.c, compiled into this program
 * with AddressSanitizer and UndefinedBehaviorSanitizer) through closed forms,
 * cancellation, subnormals and selected rows/columns; exits non-zero on a
 * wrong value (the sanitizers abort on memory or UB errors). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

int oracle_dd_gemm_block(int64_t M, int64_t N, int64_t K, const double* A_hi, const double* A_lo,
                         int64_t lda, const double* B_hi, const double* B_lo, int64_t ldb, int64_t nrows,
                         const int64_t* rows, int64_t ncols, const int64_t* cols, double* out_hi,
                         double* out_lo, int nthreads);
int oracle_md_gemm_block(int np, int64_t M, int64_t N, int64_t K, const double* const* Apart, int64_t lda,
                         const double* const* Bpart, int64_t ldb, int64_t nrows, const int64_t* rows,
                         int64_t ncols, const int64_t* cols, double* const* out, int nthreads);

static int fail(const char* what) {
    fprintf(stderr, "FAIL: %s\n", what);
    return 1;
}

int main(void) {
    enum { M = 5, N = 4, K = 37 };
    double *Ah = malloc(sizeof(double) * M * K), *Al = malloc(sizeof(double) * M * K);
    double *Bh = malloc(sizeof(double) * K * N), *Bl = malloc(sizeof(double) * K * N);
    double *Ch = malloc(sizeof(double) * M * N), *Cl = malloc(sizeof(double) * M * N);
    int64_t rows[M], cols[N];
    for (int i = 0; i < M; ++i) rows[i] = i;
    for (int j = 0; j < N; ++j) cols[j] = j;
    /* (1 + 2^-60)^2 summed K times = (K, K 2^-59) */
    for (int t = 0; t < M * K; ++t) { Ah[t] = 1.0; Al[t] = ldexp(1.0, -60); }
    for (int t = 0; t < K * N; ++t) { Bh[t] = 1.0; Bl[t] = ldexp(1.0, -60); }
    if (oracle_dd_gemm_block(M, N, K, Ah, Al, K, Bh, Bl, N, M, rows, N, cols, Ch, Cl, 2) != 0) return fail("rc");
    for (int t = 0; t < M * N; ++t)
        if (Ch[t] != K || Cl[t] != K * ldexp(1.0, -59)) return fail("closed form");
    /* exact cancellation and subnormal products */
    for (int i = 0; i < M; ++i)
        for (int k = 0; k < K; ++k) {
            Ah[i * K + k] = (k % 2 ? -1.0 : 1.0) * ldexp(1.0, -600 + i);
            Al[i * K + k] = 0.0;
        }
    for (int t = 0; t < K * N; ++t) { Bh[t] = ldexp(1.0, -500); Bl[t] = 0.0; }
    if (oracle_dd_gemm_block(M, N, K, Ah, Al, K, Bh, Bl, N, M, rows, N, cols, Ch, Cl, 2) != 0) return fail("rc2");
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            const double want = ldexp(1.0, -1100 + i); /* K odd: one term survives */
            if (Ch[i * N + j] != want || Cl[i * N + j] != 0.0) return fail("cancellation / subnormal");
        }
    /* four-part path with selected rows and columns */
    const double* Ap[4] = {Ah, Al, Al, Al};
    const double* Bp[4] = {Bh, Bl, Bl, Bl};
    double* Cp[4] = {Ch, Cl, malloc(sizeof(double) * M * N), malloc(sizeof(double) * M * N)};
    int64_t r2[2] = {4, 1}, c2[3] = {3, 0, 2};
    if (oracle_md_gemm_block(4, M, N, K, Ap, K, Bp, N, 2, r2, 3, c2, Cp, 2) != 0) return fail("rc3");
    for (int t = 0; t < 6; ++t)
        if (Cp[0][t] != ldexp(1.0, -1100 + (int)r2[t / 3]) || Cp[1][t] != 0.0) return fail("md");
    /* argument errors are reported, not acted on */
    if (oracle_dd_gemm_block(-1, N, K, Ah, Al, K, Bh, Bl, N, M, rows, N, cols, Ch, Cl, 1) != 1) return fail("arg");
    free(Cp[2]); free(Cp[3]);
    free(Ah); free(Al); free(Bh); free(Bl); free(Ch); free(Cl);
    puts("ok");
    return 0;
}
