/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the FP8 rowwise-scaled
 * grouped GEMM f8f8bf16_rowwise_grouped: stacked, dynamic, offsets, batched, ragged-N
 * and ragged-K layouts, and the block-scaled (groupwise) stacked, dynamic and batched
 * variants.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark may build, load or call this file.  It shares no code, header,
 * table or constant with the CUDA library and includes nothing from it.
 *
 * What it computes (MSLK #471 "Back the FP8 rowwise grouped GEMM ops with FlyDSL on
 * ROCm", commit introducing the rowwise scaling scheme, and the PR Summary table):
 *
 *     out[r, n] = bf16_rne( scale_a[r] * scale_b[g, n] * sum_k A[r, k] * B[g, n, k] )
 *
 * for every row r that belongs to group g.  A and B hold OCP FP8 E4M3 ("fn") codes,
 * scale_a / scale_b are fp32, out is bf16.  The rowwise scales are constant along K,
 * so the sum is taken unscaled and both scales are applied once afterwards.
 *
 * Exactness.  Every E4M3 value is an integer multiple of 2^-9 with magnitude <= 448,
 * so every product is a multiple of 2^-18 below 2^17.62, and any partial sum over
 * K <= 2^14 terms is a multiple of 2^-18 below 2^31.62: it needs fewer than 53 bits,
 * so the fp64 sum is exact in any order.  The product of two fp32 scales is exact in
 * fp64.  The last product ab*S is rounded once to fp64; its exact error is recovered
 * with fma, and the bf16 rounding uses it to break the only case where rounding the
 * fp64 value could differ from rounding the exact value (an fp64 value that sits
 * exactly on a bf16 rounding midpoint).  The result is therefore the correctly
 * rounded bf16 of the exact mathematical value.
 *
 * Layouts (MSLK #471, commits adding the packed "sizes" layout and the padded
 * "dynamic" layout; PR Summary table):
 *   stacked : groups packed along M; group g owns rows [off_g, off_g + m_g), with
 *             off_0 = 0 and off_{g+1} = off_g + m_g (exclusive prefix in group order).
 *   dynamic : group g owns the slab of rows [g*E, (g+1)*E); only its first
 *             min(max(zsi[g], 0), E) rows are valid; every other slab row is +0.0.
 * Readings of points the pages leave open:
 *   - m_sizes entries are clamped into [0, total_M - off_g], so the groups never
 *     reach past total_M; the return value reports whether any clamping happened.
 *     Rows of a stacked output past the last group are not written.
 *   - A reduction over K = 0 yields +0.0 for every owned row (MSLK #471, commit that
 *     zeroes the output of an empty reduction).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fopenmp -shared -fPIC oracle.c
 * (-ffp-contract=off keeps every multiply and add separately rounded as written.)
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake; the test suite
 * compiles the mutants to show that its pins catch each of them.  0 is the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ------------------------------------------------------------------------------ */
/* OCP 8-bit floating point specification (OFP8), format E4M3:                     */
/* sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, a single */
/* NaN mantissa pattern S.1111.111, largest finite magnitude 448.                   */
/* ------------------------------------------------------------------------------ */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
#if ORACLE_MUTANT == 6
    sign = 0; /* mutant: sign bit ignored */
#endif
    if (e == 15 && m == 7) return NAN;
    double mag;
    if (e == 0) {
        mag = ldexp((double)m, -9); /* subnormal: 2^(1-7) * m/8 */
    } else {
#if ORACLE_MUTANT == 5
        mag = ldexp((double)(8 + m), e - 11); /* mutant: bias 8 */
#else
        mag = ldexp((double)(8 + m), e - 10); /* normal: 2^(e-7) * (1 + m/8) */
#endif
    }
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------------------ */
/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits; the same exponent     */
/* range as binary32, subnormal spacing 2^-133.  Round to nearest, ties to even.   */
/* The value rounded is hi + lo exactly, where hi is a double and lo its exact     */
/* error term (|lo| <= half an ulp of hi); pass lo = 0 for a plain double.         */
/* NaN encodes as 0x7FC0 (sign kept).                                               */
/* ------------------------------------------------------------------------------ */
uint16_t oracle_bf16_round(double hi, double lo)
{
    if (isnan(hi)) return (uint16_t)(signbit(hi) ? 0xFFC0u : 0x7FC0u);
    uint16_t sign = signbit(hi) ? 0x8000u : 0u;
    double a = fabs(hi);
    double alo = signbit(hi) ? -lo : lo; /* error term of |x| */
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) {
        /* hi == 0 with a nonzero error cannot come from a correctly rounded product
         * of finite doubles unless it underflowed; treat the sign of lo as decisive. */
        if (alo == 0.0) return sign;
        /* |x| = |lo| is far below the smallest bf16 subnormal (2^-133): rounds to 0. */
        return sign;
    }

#if ORACLE_MUTANT == 4
    /* mutant: double rounding through binary32 first */
    a = (double)(float)a;
    alo = 0.0;
#endif

    int ex;
    frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;         /* floor(log2(a)) */
    int subnormal = (E < -126);
    int qexp = subnormal ? -133 : E - 7;
    double t = ldexp(a, -qexp); /* exact: scaling by a power of two, no underflow */
    double r = floor(t);
    double frac = t - r;        /* exact */
    if (frac > 0.5) {
        r += 1.0;
    } else if (frac == 0.5) {
        if (alo > 0.0) {
            r += 1.0;
        } else if (alo < 0.0) {
            /* below the midpoint: keep r */
        } else {
#if ORACLE_MUTANT == 9
            r += 1.0; /* mutant: ties away from zero */
#else
            if (fmod(r, 2.0) != 0.0) r += 1.0; /* ties to even */
#endif
        }
    }
    /* r is an integer: in [0, 128] for subnormals, [128, 256] for normals. */
    uint32_t bits;
    if (subnormal) {
        bits = (uint32_t)r;                      /* r == 128 carries into exponent 1 */
    } else {
        bits = ((uint32_t)(E + 127) << 7) + ((uint32_t)r - 128u); /* r == 256 carries */
    }
    if (bits >= 0x7F80u) bits = 0x7F80u;         /* overflow to infinity */
    return (uint16_t)(sign | bits);
}

double oracle_bf16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xFF;
    int m = bits & 0x7F;
    double mag;
    if (e == 0xFF) mag = (m == 0) ? INFINITY : NAN;
    else if (e == 0) mag = ldexp((double)m, -133);
    else mag = ldexp((double)(128 + m), e - 127 - 7);
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------------------ */
/* Group row ranges of the stacked layout: exclusive prefix of m_sizes in group     */
/* order, each count clamped into [0, total_M - off_g].  Returns 1 if any entry was */
/* clamped, else 0.  off has G+1 entries.                                           */
/* ------------------------------------------------------------------------------ */
int oracle_stacked_offsets(const int64_t *m_sizes, int64_t G, int64_t total_M, int64_t *off)
{
    int clamped = 0;
    off[0] = 0;
    for (int64_t g = 0; g < G; ++g) {
        int64_t m = m_sizes[g];
        int64_t room = total_M - off[g];
        if (m < 0) { m = 0; clamped = 1; }
        if (m > room) { m = room; clamped = 1; }
#if ORACLE_MUTANT == 7
        off[g + 1] = off[g] + m + (g == 0 ? 1 : 0); /* mutant: prefix off by one */
        if (off[g + 1] > total_M) off[g + 1] = total_M;
#else
        off[g + 1] = off[g] + m;
#endif
    }
    return clamped;
}

/* Unscaled dot product of two code rows, summed in fp64 in k order (exact). */
static double dot_lut(const uint8_t *arow, const uint8_t *brow, int64_t K, const double *lut)
{
    double s = 0.0;
    int64_t kend = K;
#if ORACLE_MUTANT == 1
    if (kend > 0) kend -= 1; /* mutant: last K term dropped */
#endif
    for (int64_t k = 0; k < kend; ++k) s += lut[arow[k]] * lut[brow[k]];
    return s;
}

/* One output element: exact fp64 dot product, scales applied once, one rounding.
 * An empty reduction (K = 0) is +0.0 whatever the scales: the op zeroes its output
 * for a contraction of length zero (MSLK #471, commit zeroing an empty reduction). */
static uint16_t oracle_element(const uint8_t *arow, const uint8_t *brow, int64_t K,
                               float sa, float sb, const double *lut)
{
    if (K == 0) return 0x0000u;
    double s = dot_lut(arow, brow, K, lut);
#if ORACLE_MUTANT == 10
    double ab = (double)sa; (void)sb; /* mutant: scale_b forgotten */
#else
    double ab = (double)sa * (double)sb; /* exact: 24 + 24 significant bits */
#endif
    double p = ab * s;
    double err = fma(ab, s, -p);         /* exact error of the rounded product */
    return oracle_bf16_round(p, err);
}

static void fill_lut(double *lut)
{
    for (int c = 0; c < 256; ++c) lut[c] = oracle_e4m3_to_double((uint8_t)c);
}

/* The fp64 dot product used for every output element (before scaling). */
double oracle_dot(const uint8_t *arow, const uint8_t *brow, int64_t K)
{
    double lut[256];
    fill_lut(lut);
    return dot_lut(arow, brow, K, lut);
}

/* Element-wise oracle_bf16_round over arrays (lo may be NULL for all zeros). */
void oracle_bf16_round_array(const double *hi, const double *lo, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(hi[i], lo ? lo[i] : 0.0);
}

static const uint8_t *b_row(const uint8_t *B, int64_t g, int64_t n, int64_t N, int64_t K)
{
    return B + ((size_t)g * (size_t)N + (size_t)n) * (size_t)K;
}

static uint16_t element_gn(const uint8_t *arow, const uint8_t *B, const float *scale_b,
                           int64_t g, int64_t n, int64_t N, int64_t K, float sa, const double *lut)
{
#if ORACLE_MUTANT == 2
    if (K == 0) return 0x0000u;
    double s = 0.0;
    const uint8_t *bg = B + (size_t)g * (size_t)N * (size_t)K;
    for (int64_t k = 0; k < K; ++k) {
        size_t idx = ((size_t)k * (size_t)N + (size_t)n) % ((size_t)N * (size_t)K);
        s += lut[arow[k]] * lut[bg[idx]];
    }
    double ab = (double)sa * (double)scale_b[g * N + n];
    double p = ab * s;
    return oracle_bf16_round(p, fma(ab, s, -p));
#else
    float sb;
#if ORACLE_MUTANT == 3
    sb = scale_b[n]; /* mutant: scale_b of group 0 used for every group */
#else
    sb = scale_b[g * N + n];
#endif
    return oracle_element(arow, b_row(B, g, n, N, K), K, sa, sb, lut);
#endif
}

/* ------------------------------------------------------------------------------ */
/* Stacked layout.  A [total_M, K], B [G, N, K], scale_a [total_M], scale_b [G, N], */
/* m_sizes [G] (int64), out [total_M, N] bf16 bits.  Rows past the last group are  */
/* left untouched.  Returns the clamp flag of oracle_stacked_offsets.               */
/* ------------------------------------------------------------------------------ */
int oracle_stacked(const uint8_t *A, const uint8_t *B, const float *scale_a,
                   const float *scale_b, const int64_t *m_sizes, int64_t G, int64_t N,
                   int64_t K, int64_t total_M, uint16_t *out, int nthreads)
{
    double lut[256];
    fill_lut(lut);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    if (!off) return -1;
    int clamped = oracle_stacked_offsets(m_sizes, G, total_M, off);
    int64_t rows = off[G];
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int64_t g = 0;
        while (!(r >= off[g] && r < off[g + 1])) ++g;
        const uint8_t *arow = A + (size_t)r * (size_t)K;
        for (int64_t n = 0; n < N; ++n)
            out[(size_t)r * (size_t)N + (size_t)n] =
                element_gn(arow, B, scale_b, g, n, N, K, scale_a[r], lut);
    }
    free(off);
    return clamped;
}

/* Stacked layout, a chosen subset of rows: out_rows[i, :] = out[rows[i], :].       */
/* A row that belongs to no group gets every element set to 0xFFFF (a marker: the  */
/* stacked output leaves such rows untouched).                                      */
int oracle_stacked_rows(const uint8_t *A, const uint8_t *B, const float *scale_a,
                        const float *scale_b, const int64_t *m_sizes, int64_t G, int64_t N,
                        int64_t K, int64_t total_M, const int64_t *rows, int64_t nrows,
                        uint16_t *out_rows, int nthreads)
{
    double lut[256];
    fill_lut(lut);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    if (!off) return -1;
    int clamped = oracle_stacked_offsets(m_sizes, G, total_M, off);
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        int64_t g = -1;
        for (int64_t h = 0; h < G; ++h)
            if (r >= off[h] && r < off[h + 1]) { g = h; break; }
        uint16_t *o = out_rows + (size_t)i * (size_t)N;
        if (g < 0) {
            for (int64_t n = 0; n < N; ++n) o[n] = 0xFFFFu;
            continue;
        }
        const uint8_t *arow = A + (size_t)r * (size_t)K;
        for (int64_t n = 0; n < N; ++n)
            o[n] = element_gn(arow, B, scale_b, g, n, N, K, scale_a[r], lut);
    }
    free(off);
    return clamped;
}

/* ------------------------------------------------------------------------------ */
/* Dynamic (padded) layout.  A [G*E, K], B [G, N, K], scale_a [G*E], scale_b [G, N], */
/* zero_start_index_M [G] (int64), out [G*E, N] bf16 bits.  Every output row is     */
/* written: valid rows with the product, padding rows with +0.0.                    */
/* ------------------------------------------------------------------------------ */
void oracle_dynamic(const uint8_t *A, const uint8_t *B, const float *scale_a,
                    const float *scale_b, const int64_t *zsi, int64_t G, int64_t E,
                    int64_t N, int64_t K, uint16_t *out, int nthreads)
{
    double lut[256];
    fill_lut(lut);
    int64_t rows = G * E;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t row = 0; row < rows; ++row) {
        int64_t g = row / E;
        int64_t r = row - g * E;
        int64_t v = zsi[g];
        if (v < 0) v = 0;
        if (v > E) v = E;
        uint16_t *o = out + (size_t)row * (size_t)N;
        if (r >= v) {
#if ORACLE_MUTANT == 8
            continue; /* mutant: padding rows left as they were */
#else
            for (int64_t n = 0; n < N; ++n) o[n] = 0x0000u;
            continue;
#endif
        }
        const uint8_t *arow = A + (size_t)row * (size_t)K;
        for (int64_t n = 0; n < N; ++n)
            o[n] = element_gn(arow, B, scale_b, g, n, N, K, scale_a[row], lut);
    }
}

/* Dynamic layout, a chosen subset of slab rows (global row indices in [0, G*E)). */
void oracle_dynamic_rows(const uint8_t *A, const uint8_t *B, const float *scale_a,
                         const float *scale_b, const int64_t *zsi, int64_t G, int64_t E,
                         int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                         uint16_t *out_rows, int nthreads)
{
    double lut[256];
    fill_lut(lut);
    (void)G;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t row = rows[i];
        int64_t g = row / E;
        int64_t r = row - g * E;
        int64_t v = zsi[g];
        if (v < 0) v = 0;
        if (v > E) v = E;
        uint16_t *o = out_rows + (size_t)i * (size_t)N;
        if (r >= v) {
            for (int64_t n = 0; n < N; ++n) o[n] = 0x0000u;
            continue;
        }
        const uint8_t *arow = A + (size_t)row * (size_t)K;
        for (int64_t n = 0; n < N; ++n)
            o[n] = element_gn(arow, B, scale_b, g, n, N, K, scale_a[row], lut);
    }
}

/* ------------------------------------------------------------------------------ */
/* Offsets layout (2D-3D, the torch-native grouped mm addressing; MSLK #471, commit  */
/* decoding group boundaries from an int32 inclusive prefix sum): offsets[g] is the  */
/* end row of group g, so group g owns rows [offsets[g-1], offsets[g]) with          */
/* offsets[-1] = 0 -- a row count is the step between successive offsets.  Counts    */
/* then follow the stacked rules (a negative step owns no rows; rows past total_M    */
/* are clamped).  Returns the stacked clamp flag.                                    */
/* ------------------------------------------------------------------------------ */
int oracle_offsets(const uint8_t *A, const uint8_t *B, const float *scale_a,
                   const float *scale_b, const int32_t *offsets, int64_t G, int64_t N,
                   int64_t K, int64_t total_M, uint16_t *out, int nthreads)
{
    int64_t *m = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    if (!m) return -1;
    for (int64_t g = 0; g < G; ++g)
        m[g] = (int64_t)offsets[g] - (g > 0 ? (int64_t)offsets[g - 1] : 0);
    int clamped = oracle_stacked(A, B, scale_a, scale_b, m, G, N, K, total_M, out, nthreads);
    free(m);
    return clamped;
}

/* ------------------------------------------------------------------------------ */
/* Batched layout (3D-3D; MSLK #471, commit adding the layout whose groups all carry */
/* their full complement of rows): group g owns the whole slab [g*M, (g+1)*M), every */
/* row computed, and no metadata is read.                                           */
/* ------------------------------------------------------------------------------ */
void oracle_batched(const uint8_t *A, const uint8_t *B, const float *scale_a,
                    const float *scale_b, int64_t G, int64_t M, int64_t N, int64_t K,
                    uint16_t *out, int nthreads)
{
    double lut[256];
    fill_lut(lut);
    int64_t rows = G * M;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t row = 0; row < rows; ++row) {
        int64_t g = row / M;
        const uint8_t *arow = A + (size_t)row * (size_t)K;
        uint16_t *o = out + (size_t)row * (size_t)N;
        for (int64_t n = 0; n < N; ++n)
            o[n] = element_gn(arow, B, scale_b, g, n, N, K, scale_a[row], lut);
    }
}

/* ------------------------------------------------------------------------------ */
/* Ragged-N layout (3D-2D; MSLK #471, commit adding the form whose weights are one    */
/* [total_N, K] matrix that the groups partition by row, results packed side by side */
/* into [M, total_N]).  A [G, M, K] (one slab of M rows per group), scale_a [G, M],    */
/* B [total_N, K], scale_b [total_N], offsets [G] int32 inclusive prefix over N:       */
/* group g owns the output columns [c_g, c_{g+1}), where the column counts are the     */
/* steps offsets[g] - offsets[g-1] (offsets[-1] = 0) under the stacked clamping rules. */
/*   out[m, n] = bf16(sa[g, m] * sb[n] * sum_k A[g, m, k] * B[n, k]),  n in group g    */
/* Columns past the last group are left untouched.  Returns the clamp flag.           */
/* ------------------------------------------------------------------------------ */
static int counts_from_offsets(const int32_t *offsets, int64_t G, int64_t total, int64_t *bound)
{
    int64_t *cnt = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    if (!cnt) return -1;
    for (int64_t g = 0; g < G; ++g)
        cnt[g] = (int64_t)offsets[g] - (g > 0 ? (int64_t)offsets[g - 1] : 0);
    int clamped = oracle_stacked_offsets(cnt, G, total, bound);
    free(cnt);
    return clamped;
}

int oracle_n_offsets(const uint8_t *A, const uint8_t *B, const float *scale_a,
                     const float *scale_b, const int32_t *offsets, int64_t G, int64_t M,
                     int64_t total_N, int64_t K, const int64_t *rows, int64_t nrows,
                     uint16_t *out, int nthreads)
{
    /* rows == NULL: all M output rows into out [M, total_N]; else out row i = row rows[i] */
    double lut[256];
    fill_lut(lut);
    int64_t *col = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    if (!col) return -1;
    int clamped = counts_from_offsets(offsets, G, total_N, col);
    int64_t n_out = rows ? nrows : M;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < n_out; ++i) {
        int64_t m = rows ? rows[i] : i;
        uint16_t *o = out + (size_t)i * (size_t)total_N;
        for (int64_t g = 0; g < G; ++g) {
#if ORACLE_MUTANT == 11
            const uint8_t *arow = A + (size_t)m * (size_t)K; /* mutant: slab of group 0 */
#else
            const uint8_t *arow = A + ((size_t)g * (size_t)M + (size_t)m) * (size_t)K;
#endif
            float sa = scale_a[g * M + m];
            for (int64_t n = col[g]; n < col[g + 1]; ++n)
                o[n] = oracle_element(arow, B + (size_t)n * (size_t)K, K, sa, scale_b[n], lut);
        }
    }
    free(col);
    return clamped;
}

/* ------------------------------------------------------------------------------ */
/* Ragged-K layout (2D-2D; MSLK #471, commit adding the layout whose groups slice K):   */
/* A [M, total_K], B [N, total_K], scale_a [G, M], scale_b [G, N], offsets [G] int32   */
/* inclusive prefix over K: group g contracts over k in [k_g, k_{g+1}) (counts and     */
/* clamping as above) and produces a whole [M, N] slab:                                 */
/*   out[g, m, n] = bf16(sa[g, m] * sb[g, n] * sum_{k_g <= k < k_{g+1}} A[m, k] B[n, k]) */
/* A group contracting over nothing gets +0.0 (the empty sum).  out is [G*M, N]; with   */
/* rows != NULL, out row i is slab row rows[i] (in [0, G*M)).  Returns the clamp flag.  */
/* ------------------------------------------------------------------------------ */
int oracle_k_offsets(const uint8_t *A, const uint8_t *B, const float *scale_a,
                     const float *scale_b, const int32_t *offsets, int64_t G, int64_t M,
                     int64_t N, int64_t total_K, const int64_t *rows, int64_t nrows,
                     uint16_t *out, int nthreads)
{
    double lut[256];
    fill_lut(lut);
    int64_t *ks = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    if (!ks) return -1;
    int clamped = counts_from_offsets(offsets, G, total_K, ks);
    int64_t n_out = rows ? nrows : G * M;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < n_out; ++i) {
        int64_t row = rows ? rows[i] : i;
        int64_t g = row / M;
        int64_t m = row - g * M;
#if ORACLE_MUTANT == 12
        int64_t k0 = 0, len = ks[g + 1] - ks[g]; /* mutant: every slice starts at k = 0 */
#else
        int64_t k0 = ks[g], len = ks[g + 1] - ks[g];
#endif
        const uint8_t *arow = A + (size_t)m * (size_t)total_K + (size_t)k0;
        float sa = scale_a[g * M + m];
        uint16_t *o = out + (size_t)i * (size_t)N;
        for (int64_t n = 0; n < N; ++n)
            o[n] = oracle_element(arow, B + (size_t)n * (size_t)total_K + (size_t)k0, len, sa,
                                  scale_b[g * N + n], lut);
    }
    free(ks);
    return clamped;
}

/* ------------------------------------------------------------------------------ */
/* Block-scaled (groupwise) stacked layout (MSLK #471, commit introducing the rowwise */
/* scheme beside the block scheme the kernel already had: a scale per scale block,    */
/* applied to each block's partial sum inside the K loop).  Blocks of 128 along K and */
/* 128 along N (the pages require K and N to cover whole blocks under block scaling): */
/*   scale_a [total_M, K/128]     one scale per row and K block                        */
/*   scale_b [G, N/128, K/128]    one scale per (128 columns x 128 K) block of B       */
/*   out[r, n] = bf16( sum_kb scale_a[r, kb] * scale_b[g, n/128, kb] * S_kb(r, n) )    */
/* with S_kb the exact sum over the block's 128 products.  Each term ab * S_kb is     */
/* split exactly into p + e (fma) and the terms are summed in double-double (Knuth's   */
/* TwoSum), so the bf16 rounding sees the exact value to ~106 bits.  Returns the       */
/* stacked clamp flag, or -2 if K or N is not a multiple of 128.                       */
/* ------------------------------------------------------------------------------ */
#define ORACLE_SCALE_BLOCK 128

static void two_sum(double a, double b, double *s, double *e)
{
    double x = a + b;
    double bv = x - a;
    double av = x - bv;
    *s = x;
    *e = (a - av) + (b - bv);
}

static uint16_t blockwise_element(const uint8_t *arow, const uint8_t *brow, int64_t K,
                                  const float *sa_row, const float *sb_blk, const double *lut)
{
    int64_t nkb = K / ORACLE_SCALE_BLOCK;
    if (nkb == 0) return 0x0000u;
    double hi = 0.0, lo = 0.0;
    for (int64_t kb = 0; kb < nkb; ++kb) {
        double S = dot_lut(arow + kb * ORACLE_SCALE_BLOCK, brow + kb * ORACLE_SCALE_BLOCK,
                           ORACLE_SCALE_BLOCK, lut);
#if ORACLE_MUTANT == 13
        double ab = (double)sa_row[0] * (double)sb_blk[0]; /* mutant: block 0's scales */
#else
        double ab = (double)sa_row[kb] * (double)sb_blk[kb]; /* exact */
#endif
        double p = ab * S;
        double pe = fma(ab, S, -p);
        double t;
        two_sum(hi, p, &hi, &t);
        lo += t + pe;
    }
    double e;
    two_sum(hi, lo, &hi, &e);
    return oracle_bf16_round(hi, e);
}

int oracle_blockwise_stacked(const uint8_t *A, const uint8_t *B, const float *scale_a,
                             const float *scale_b, const int64_t *m_sizes, int64_t G,
                             int64_t N, int64_t K, int64_t total_M, const int64_t *rows,
                             int64_t nrows, uint16_t *out, int nthreads)
{
    /* rows == NULL: the whole output [total_M, N] (rows past the last group untouched);
     * else out row i = output row rows[i] (0xFFFF for a row of no group) */
    if (K % ORACLE_SCALE_BLOCK != 0 || N % ORACLE_SCALE_BLOCK != 0) return -2;
    double lut[256];
    fill_lut(lut);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    if (!off) return -1;
    int clamped = oracle_stacked_offsets(m_sizes, G, total_M, off);
    int64_t nkb = K / ORACLE_SCALE_BLOCK, nnb = N / ORACLE_SCALE_BLOCK;
    int64_t n_out = rows ? nrows : off[G];
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < n_out; ++i) {
        int64_t r = rows ? rows[i] : i;
        int64_t g = -1;
        for (int64_t h = 0; h < G; ++h)
            if (r >= off[h] && r < off[h + 1]) { g = h; break; }
        uint16_t *o = out + (size_t)i * (size_t)N;
        if (g < 0) {
            if (rows) for (int64_t n = 0; n < N; ++n) o[n] = 0xFFFFu;
            continue;
        }
        const uint8_t *arow = A + (size_t)r * (size_t)K;
        const float *sa_row = scale_a + (size_t)r * (size_t)nkb;
        for (int64_t n = 0; n < N; ++n) {
            const float *sb_blk = scale_b + ((size_t)g * (size_t)nnb + (size_t)(n / ORACLE_SCALE_BLOCK)) * (size_t)nkb;
            o[n] = blockwise_element(arow, b_row(B, g, n, N, K), K, sa_row, sb_blk, lut);
        }
    }
    free(off);
    return clamped;
}

/* ------------------------------------------------------------------------------ */
/* Block-scaled (groupwise) dynamic and batched layouts: the slabs of the dynamic    */
/* layout (group g owns rows [g*E, (g+1)*E); the first min(max(zsi[g], 0), E) are    */
/* valid and every other slab row is +0.0) with the block scaling above:             */
/*   scale_a [G*E, K/128]         one scale per slab row and K block                 */
/*   scale_b [G, N/128, K/128]    one scale per (128 columns x 128 K) block of B     */
/* zsi == NULL: every slab row is valid (the batched layout, no metadata).            */
/* rows == NULL: the whole output [G*E, N]; else out row i = slab row rows[i].        */
/* Returns -2 if K or N is not a multiple of 128, else 0.                             */
/* ------------------------------------------------------------------------------ */
int oracle_blockwise_dynamic(const uint8_t *A, const uint8_t *B, const float *scale_a,
                             const float *scale_b, const int64_t *zsi, int64_t G, int64_t E,
                             int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                             uint16_t *out, int nthreads)
{
    if (K % ORACLE_SCALE_BLOCK != 0 || N % ORACLE_SCALE_BLOCK != 0) return -2;
    double lut[256];
    fill_lut(lut);
    int64_t nkb = K / ORACLE_SCALE_BLOCK, nnb = N / ORACLE_SCALE_BLOCK;
    int64_t n_out = rows ? nrows : G * E;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < n_out; ++i) {
        int64_t row = rows ? rows[i] : i;
        int64_t g = row / E;
        int64_t r = row - g * E;
        int64_t v = zsi ? zsi[g] : E;
        if (v < 0) v = 0;
        if (v > E) v = E;
        uint16_t *o = out + (size_t)i * (size_t)N;
        if (r >= v) {
            for (int64_t n = 0; n < N; ++n) o[n] = 0x0000u;
            continue;
        }
        const uint8_t *arow = A + (size_t)row * (size_t)K;
#if ORACLE_MUTANT == 14
        const float *sa_row = scale_a + (size_t)r * (size_t)nkb; /* mutant: slab-local row */
#else
        const float *sa_row = scale_a + (size_t)row * (size_t)nkb;
#endif
        for (int64_t n = 0; n < N; ++n) {
            const float *sb_blk = scale_b + ((size_t)g * (size_t)nnb + (size_t)(n / ORACLE_SCALE_BLOCK)) * (size_t)nkb;
            o[n] = blockwise_element(arow, b_row(B, g, n, N, K), K, sa_row, sb_blk, lut);
        }
    }
    return 0;
}

/* Exact unscaled dot products as integers: S * 2^18 for one (row, n) pair, using   */
/* the integer form of each code (value * 2^9).  Lets a test check the fp64 sum     */
/* against integer arithmetic.  NaN codes yield INT64_MIN.                          */
int64_t oracle_dot_int(const uint8_t *arow, const uint8_t *brow, int64_t K)
{
    int64_t s = 0;
    for (int64_t k = 0; k < K; ++k) {
        uint8_t ca = arow[k], cb = brow[k];
        if ((ca & 0x7F) == 0x7F || (cb & 0x7F) == 0x7F) return INT64_MIN;
        int ea = (ca >> 3) & 15, ma = ca & 7, eb = (cb >> 3) & 15, mb = cb & 7;
        int64_t ia = (ea == 0) ? ma : ((int64_t)(8 + ma) << (ea - 1)); /* value * 2^9 */
        int64_t ib = (eb == 0) ? mb : ((int64_t)(8 + mb) << (eb - 1));
        if (ca & 0x80) ia = -ia;
        if (cb & 0x80) ib = -ib;
        s += ia * ib;
    }
    return s;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
