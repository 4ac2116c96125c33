/*
 * exact_ddgemm.c -- exact double-double matrix product, rounded once.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference ("oracle") that the
 * GPU path is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header
 * or constant with the CUDA library.
 *
 * What it computes (the plain definition of the product of double-double
 * matrices; "Multiple Double Arithmetic on NVIDIA Tensor Cores", Definition
 * 1.1 (a multiple double is an unevaluated sum of doubles) and the final step
 * of the Section 2 algorithm (the parts are summed into one double double)):
 *
 *     X_ij = sum_k (A_hi[i,k] + A_lo[i,k]) * (B_hi[k,j] + B_lo[k,j])
 *
 * formed EXACTLY, then rounded once to the nearest double double:
 *
 *     C_hi = RN(X),  C_lo = RN(X - C_hi)       (round to nearest, ties to even)
 *
 * Method: every double is an integer mantissa times a power of two.  Each of
 * the four products per k is an exact 106-bit integer (unsigned __int128)
 * times a power of two; it is added, with its sign, into a fixed-point
 * accumulator whose least significant bit is 2^-2208 (below the smallest
 * product of two subnormals, 2^-2148) and which spans 140 limbs of 32 bits
 * (up to 2^2272, above the largest product sum of finite doubles for
 * K <= 2^26).  Limbs are int64 and take signed 32-bit digits with deferred
 * carries, so 2^30 deposits cannot overflow them.  The result is independent
 * of the order of k and of the number of threads.
 *
 * Non-finite inputs are rejected (return code 2).  A result beyond the double
 * range is returned as +-inf in hi (never reached by the workloads).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LIMB_BITS 32
#define NLIMBS 140
#define BASE_EXP (-2208) /* weight of bit 0 of limb 0 is 2^BASE_EXP */
#define MAX_K (1LL << 26)

typedef struct {
    uint64_t m; /* integer mantissa, < 2^53 */
    int32_t e;  /* value = (-1)^neg * m * 2^e */
    int32_t neg;
} dec_t;

/* Split a finite double into sign, integer mantissa and exponent (IEEE 754
 * binary64 bit layout; subnormals have no hidden bit and exponent -1074). */
static int decompose(double x, dec_t* d) {
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint32_t biased = (uint32_t)((bits >> 52) & 0x7FF);
    uint64_t frac = bits & ((1ULL << 52) - 1);
    if (biased == 0x7FF) return -1;
    d->neg = (int32_t)(bits >> 63);
    if (biased == 0) {
        d->m = frac;
        d->e = -1074;
    } else {
        d->m = frac | (1ULL << 52);
        d->e = (int32_t)biased - 1075;
    }
    return 0;
}

typedef struct {
    int64_t limb[NLIMBS];
    int lo, hi; /* touched limb range [lo, hi] */
} acc_t;

static void acc_clear(acc_t* a) {
    memset(a->limb, 0, sizeof a->limb);
    a->lo = NLIMBS;
    a->hi = -1;
}

/* Add (-1)^neg * m1 * m2 * 2^(e1 + e2) exactly. */
static void acc_add_product(acc_t* a, const dec_t* x, const dec_t* y) {
    if (x->m == 0 || y->m == 0) return;
    unsigned __int128 p = (unsigned __int128)x->m * y->m; /* < 2^106 */
    int pos = x->e + y->e - BASE_EXP;                       /* >= 60 */
    int L = pos / LIMB_BITS, off = pos % LIMB_BITS;
    unsigned __int128 low = p << off; /* bits that stay below 2^128 */
    uint64_t top = off ? (uint64_t)(p >> (128 - off)) : 0;
    uint64_t w[5];
    w[0] = (uint64_t)low & 0xFFFFFFFFu;
    w[1] = (uint64_t)(low >> 32) & 0xFFFFFFFFu;
    w[2] = (uint64_t)(low >> 64) & 0xFFFFFFFFu;
    w[3] = (uint64_t)(low >> 96) & 0xFFFFFFFFu;
    w[4] = top;
    int neg = x->neg ^ y->neg;
    for (int i = 0; i < 5; ++i) {
        if (w[i] == 0) continue;
        int idx = L + i;
        a->limb[idx] += neg ? -(int64_t)w[i] : (int64_t)w[i];
        if (idx < a->lo) a->lo = idx;
        if (idx > a->hi) a->hi = idx;
    }
}

/* Propagate carries so that every limb is in [0, 2^32), except that the sign
 * of the whole number is returned: on return the limbs hold |X| and *neg is
 * set when X < 0. */
static void acc_normalize(acc_t* a, int* neg) {
    *neg = 0;
    if (a->hi < 0) return;
    int64_t carry = 0;
    for (int i = a->lo; i < NLIMBS; ++i) {
        int64_t v = a->limb[i] + carry;
        int64_t low = v & 0xFFFFFFFFLL;
        carry = (v - low) / 4294967296LL; /* exact floor division */
        a->limb[i] = low;
        if (low != 0 && i > a->hi) a->hi = i;
        if (i >= a->hi && carry == 0) break;
    }
    if (carry < 0) {
        /* X = carry * 2^(32*NLIMBS) + limbs < 0: take the magnitude. */
        *neg = 1;
        for (int i = a->lo; i < NLIMBS; ++i) a->limb[i] = -a->limb[i];
        a->hi = NLIMBS - 1;
        carry = 0;
        for (int i = a->lo; i < NLIMBS; ++i) {
            int64_t v = a->limb[i] + carry;
            int64_t low = v & 0xFFFFFFFFLL;
            carry = (v - low) / 4294967296LL;
            a->limb[i] = low;
        }
    }
    while (a->hi >= a->lo && a->limb[a->hi] == 0) --a->hi;
    if (a->hi < a->lo) { a->lo = NLIMBS; a->hi = -1; }
}

/* Bit b (absolute index from bit 0 of limb 0) of the normalised magnitude. */
static int get_bit(const acc_t* a, long b) {
    if (b < 0) return 0;
    long L = b / LIMB_BITS;
    if (L >= NLIMBS) return 0;
    return (int)((a->limb[L] >> (b % LIMB_BITS)) & 1);
}

/* Is any bit with index < b set? */
static int any_below(const acc_t* a, long b) {
    if (b <= 0 || a->hi < 0) return 0;
    long L = b / LIMB_BITS;
    for (long i = a->lo; i < L && i <= a->hi; ++i)
        if (a->limb[i]) return 1;
    if (L <= a->hi && L < NLIMBS) {
        int r = (int)(b % LIMB_BITS);
        if (r && (a->limb[L] & ((1LL << r) - 1))) return 1;
    }
    return 0;
}

/* Round the normalised magnitude (with sign neg) to the nearest double,
 * ties to even, with gradual underflow. */
static double acc_round(const acc_t* a, int neg) {
    if (a->hi < 0) return 0.0; /* exact zero -> +0 */
    int64_t top = a->limb[a->hi];
    int msb = 63 - __builtin_clzll((unsigned long long)top);
    long tbit = (long)a->hi * LIMB_BITS + msb; /* index of the leading bit */
    long texp = tbit + BASE_EXP;               /* its weight exponent */
    long qexp = texp - 52;                     /* weight of the last kept bit */
    if (qexp < -1074) qexp = -1074;
    long qbit = qexp - BASE_EXP;
    uint64_t m = 0;
    for (long b = tbit; b >= qbit; --b) m = (m << 1) | (uint64_t)get_bit(a, b);
    int rbit = get_bit(a, qbit - 1);
    int sticky = any_below(a, qbit - 1);
    if (rbit && (sticky || (m & 1))) m += 1;
    double r;
    /* The largest finite double is (2^53 - 1) * 2^971. */
    if (qexp > 971 || (qexp == 971 && m >= (1ULL << 53))) {
        r = INFINITY;
    } else {
        r = ldexp((double)m, (int)qexp); /* m <= 2^53: exact */
    }
    return neg ? -r : r;
}

/* Exact value of one output entry, rounded once to the nearest dd.  `arow`
 * holds the 2K decompositions (hi, lo) of row i of A, `bcol` those of column
 * j of B, interleaved as [k][hi, lo]. */
static void entry(const dec_t* arow, const dec_t* bcol, int64_t K, acc_t* acc,
                  double* out_hi, double* out_lo) {
    acc_clear(acc);
    for (int64_t k = 0; k < K; ++k) {
        const dec_t* x = arow + 2 * k;
        const dec_t* y = bcol + 2 * k;
        acc_add_product(acc, &x[0], &y[0]);
        acc_add_product(acc, &x[0], &y[1]);
        acc_add_product(acc, &x[1], &y[0]);
        acc_add_product(acc, &x[1], &y[1]);
    }
    int neg;
    acc_normalize(acc, &neg);
    double hi = acc_round(acc, neg);
    double lo = 0.0;
    if (hi != 0.0 && isfinite(hi)) {
        /* Subtract hi exactly (its bits lie on the accumulator grid), then
         * round the remainder.  The accumulator holds |X|; undo the sign. */
        if (neg)
            for (int i = acc->lo; i <= acc->hi; ++i) acc->limb[i] = -acc->limb[i];
        dec_t h, one;
        decompose(-hi, &h);
        one.m = 1; one.e = 0; one.neg = 0;
        acc_add_product(acc, &h, &one);
        acc_normalize(acc, &neg);
        lo = acc_round(acc, neg);
    }
    *out_hi = hi + 0.0; /* +0 for a zero result */
    *out_lo = lo + 0.0;
}

/*
 * C[r, c] for r in rows[0..nrows), c in cols[0..ncols): the block of the exact
 * product at the chosen rows and columns of C, written row-major to
 * out_hi/out_lo (nrows x ncols).  A is M x K row-major with leading dimension
 * lda (hi and lo planes), B is K x N row-major with leading dimension ldb.
 * nthreads <= 0 uses the OpenMP default.
 * Returns 0 on success, 1 on a bad argument, 2 on a non-finite input,
 * 3 when out of host memory.
 */
int oracle_dd_gemm_block(int64_t M, int64_t N, int64_t K,
                         const double* A_hi, const double* A_lo, int64_t lda,
                         const double* B_hi, const double* B_lo, int64_t ldb,
                         int64_t nrows, const int64_t* rows,
                         int64_t ncols, const int64_t* cols,
                         double* out_hi, double* out_lo, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || K > MAX_K || nrows < 0 || ncols < 0) return 1;
    if (nrows == 0 || ncols == 0) return 0;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 1;
    for (int64_t c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N) return 1;
    if (K == 0) {
        for (int64_t t = 0; t < nrows * ncols; ++t) { out_hi[t] = 0.0; out_lo[t] = 0.0; }
        return 0;
    }
    size_t kk = (size_t)(2 * K);
    dec_t* adec = (dec_t*)malloc(sizeof(dec_t) * kk * (size_t)nrows);
    dec_t* bdec = (dec_t*)malloc(sizeof(dec_t) * kk * (size_t)ncols);
    if (!adec || !bdec) { free(adec); free(bdec); return 3; }
    int bad = 0;
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            bad |= decompose(A_hi[rows[r] * lda + k], &adec[r * kk + 2 * k]);
            bad |= decompose(A_lo[rows[r] * lda + k], &adec[r * kk + 2 * k + 1]);
        }
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t k = 0; k < K; ++k) {
            bad |= decompose(B_hi[k * ldb + cols[c]], &bdec[c * kk + 2 * k]);
            bad |= decompose(B_lo[k * ldb + cols[c]], &bdec[c * kk + 2 * k + 1]);
        }
    if (bad) { free(adec); free(bdec); return 2; }
    int64_t total = nrows * ncols;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        acc_t* acc = (acc_t*)malloc(sizeof(acc_t));
#pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < total; ++t) {
            int64_t r = t / ncols, c = t % ncols;
            entry(adec + r * kk, bdec + c * kk, K, acc, &out_hi[t], &out_lo[t]);
        }
        free(acc);
    }
    free(adec);
    free(bdec);
    return 0;
}

/*
 * Multiple doubles with `np` parts (2: double double, 4: quad double, 8: octo
 * double, 16: hexa double -- the sizes of the paper's Table 2): the
 * exact value X_ij = sum_k (sum_p A_p[i,k]) (sum_q B_q[k,j]) rounded once to
 * np non-overlapping doubles, x_0 = RN(X), x_1 = RN(X - x_0), ...,
 * x_{np-1} = RN(X - x_0 - ... - x_{np-2}) ("Multiple Double Arithmetic on
 * NVIDIA Tensor Cores", Definition 1.1: a multiple double is an unevaluated
 * sum of non-overlapping doubles).  Apart[p] / Bpart[p] are the part planes
 * (row-major, leading dimensions lda / ldb); out[p] receives part p of the
 * nrows x ncols block.  Return codes as oracle_dd_gemm_block.
 */
#define MAX_PARTS 16  /* every product of two parts stays inside the accumulator's range */

static void entry_md(const dec_t* arow, const dec_t* bcol, int64_t K, int np, acc_t* acc,
                     double* const* out, int64_t t) {
    acc_clear(acc);
    for (int64_t k = 0; k < K; ++k) {
        const dec_t* x = arow + np * k;
        const dec_t* y = bcol + np * k;
        for (int p = 0; p < np; ++p)
            for (int q = 0; q < np; ++q) acc_add_product(acc, &x[p], &y[q]);
    }
    int neg;
    acc_normalize(acc, &neg);
    for (int p = 0; p < np; ++p) {
        double v = acc_round(acc, neg);
        out[p][t] = v + 0.0;
        if (v == 0.0 || !isfinite(v)) {
            for (int r = p + 1; r < np; ++r) out[r][t] = 0.0;
            return;
        }
        /* subtract v exactly and continue with the remainder */
        if (neg)
            for (int i = acc->lo; i <= acc->hi; ++i) acc->limb[i] = -acc->limb[i];
        dec_t h, one;
        decompose(-v, &h);
        one.m = 1; one.e = 0; one.neg = 0;
        acc_add_product(acc, &h, &one);
        acc_normalize(acc, &neg);
    }
}

int oracle_md_gemm_block(int np, int64_t M, int64_t N, int64_t K,
                         const double* const* Apart, int64_t lda,
                         const double* const* Bpart, int64_t ldb,
                         int64_t nrows, const int64_t* rows,
                         int64_t ncols, const int64_t* cols,
                         double* const* out, int nthreads) {
    if (np < 1 || np > MAX_PARTS) return 1;
    if (M < 0 || N < 0 || K < 0 || (int64_t)np * np * K > 4 * MAX_K || nrows < 0 || ncols < 0) return 1;
    if (nrows == 0 || ncols == 0) return 0;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 1;
    for (int64_t c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N) return 1;
    if (K == 0) {
        for (int p = 0; p < np; ++p)
            for (int64_t t = 0; t < nrows * ncols; ++t) out[p][t] = 0.0;
        return 0;
    }
    size_t kk = (size_t)np * (size_t)K;
    dec_t* adec = (dec_t*)malloc(sizeof(dec_t) * kk * (size_t)nrows);
    dec_t* bdec = (dec_t*)malloc(sizeof(dec_t) * kk * (size_t)ncols);
    if (!adec || !bdec) { free(adec); free(bdec); return 3; }
    int bad = 0;
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t k = 0; k < K; ++k)
            for (int p = 0; p < np; ++p)
                bad |= decompose(Apart[p][rows[r] * lda + k], &adec[r * kk + (size_t)np * k + p]);
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t k = 0; k < K; ++k)
            for (int p = 0; p < np; ++p)
                bad |= decompose(Bpart[p][k * ldb + cols[c]], &bdec[c * kk + (size_t)np * k + p]);
    if (bad) { free(adec); free(bdec); return 2; }
    int64_t total = nrows * ncols;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        acc_t* acc = (acc_t*)malloc(sizeof(acc_t));
#pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < total; ++t) {
            int64_t r = t / ncols, c = t % ncols;
            entry_md(adec + r * kk, bdec + c * kk, K, np, acc, out, t);
        }
        free(acc);
    }
    free(adec);
    free(bdec);
    return 0;
}

/* Number of threads an OpenMP parallel region uses by default. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
