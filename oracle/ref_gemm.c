/*
 * CPU oracle for the FP8 fine-grained-scaled GEMM (NT layout, bf16 output).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this code.  It shares nothing with the CUDA path:
 * no headers, helpers, tables or constants.  It is plain and slow on purpose,
 * so that a reader can check it against the method's definition by eye.
 *
 * What it computes (DeepGEMM: "clean and efficient FP8 GEMM kernels with
 * fine-grained scaling", es.news.hada.io/topic?id=19459, section
 * "Interfaz GEMM y restricciones de layout"; DeepSeek-V3 fine-grained scaling
 * as summarised on es.news.hada.io/topic?id=19444, first list):
 *
 *   D[m,n] = bf16_rne( sum over K groups g of
 *              ( sum_{k in g} dec(A[m,k]) * dec(B[n,k]) ) * sa[m,g] * sb[n/128,g] )
 *
 *   A  : e4m3 codes, [M][K] row-major (the non-transposed LHS of "NT")
 *   B  : e4m3 codes, [N][K] row-major (the transposed RHS of "NT")
 *   g  : a 128-wide slice of K
 *   sa : fp32, one per (row, K group), stored K-group-major ("transposed",
 *        TMA-aligned): sa[g * ld_sa + m]
 *   sb : fp32, one per 128x128 block of B: sb[(n/128) * kb + g]
 *   D  : bf16 bit patterns, [M][N] row-major
 *
 * Arithmetic: each group's dot product is summed in double, which is exact
 * (every product of two e4m3 values is a multiple of 2^-18 below 2^18, and
 * 128 of them fit in 53 bits).  The scale products and the sum over groups
 * round in double (relative error ~1e-16).  The result is rounded once, from
 * double straight to bf16, round-to-nearest-even.
 *
 * The file also holds the other storage layouts (nn, tn, tt) and the
 * K-grouped form (dg_ref_gemm_layout, dg_ref_k_grouped_tn, with their
 * readings) and the activation quantiser that produces A and sa
 * (dg_ref_quantize_1x128, at the end, with its own reading).
 *
 * The M-grouped forms (same pages, section "Dense y Grouped GEMM"):
 *  - contiguous: rows of all experts are concatenated along M; m_indices[m]
 *    names the expert of row m, and -1 marks a padding row, whose output is
 *    written as +0;
 *  - masked: A is [G][max_m][K]; only the first masked_m[g] rows of group g
 *    are computed; the other output rows are left as they were.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC ref_gemm.c -o libdgref.so -lm
 * (oracle/build.py does this).  OpenMP only splits rows across threads; the
 * arithmetic of every output element is the same with any thread count.
 *
 * DG_REF_MUTANT (test-only): when defined to a nonzero value, one deliberate
 * mistake is compiled in, so that the pin tests can show they catch it.  The
 * normal build never defines it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef DG_REF_MUTANT
#define DG_REF_MUTANT 0
#endif

/* ---------------------------------------------------------------- e4m3 -- */
/* OCP FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits.  Exponent field 0 holds subnormals (f/8 * 2^-6).  There is
 * no infinity; S.1111.111 is NaN, so the largest finite value is 448. */
double dg_ref_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int f = code & 0x7;
    double mag;
    if (e == 0xF && f == 0x7)
        return NAN;
#if DG_REF_MUTANT == 4
    if (e == 0)
        mag = 0.0;                       /* mutant: subnormals flushed */
    else
#else
    if (e == 0)
        mag = ldexp((double)f / 8.0, -6); /* subnormal */
    else
#endif
        mag = ldexp(1.0 + (double)f / 8.0, e - 7);
#if DG_REF_MUTANT == 7
    (void)sign;
    return mag;                          /* mutant: sign dropped */
#else
    return sign ? -mag : mag;
#endif
}

/* ---------------------------------------------------------------- bf16 -- */
/* bf16: 1 sign bit, 8 exponent bits (bias 127, as fp32), 7 stored mantissa
 * bits.  Normal values are (1 + f/128) * 2^(e-127); below 2^-126 the spacing
 * stays 2^-133 (subnormals).  The rounding is to nearest, ties to even, done
 * once from the double value.  Every bf16 value is also an fp32 value, so the
 * rounded number is built as a float and its upper 16 bits are returned. */
uint16_t dg_ref_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    double q; /* spacing of bf16 values around a */
    if (a == 0.0 || isinf(a)) {
        float f = (float)x;
        uint32_t u;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    if (a < ldexp(1.0, -126)) {
        q = ldexp(1.0, -133);
    } else {
        int ex;
        frexp(a, &ex);                   /* a = fr * 2^ex with fr in [0.5, 1) */
        q = ldexp(1.0, (ex - 1) - 7);    /* 8 significant bits */
    }
    double r = a / q;                    /* exact: q is a power of two */
#if DG_REF_MUTANT == 5
    double n = floor(r);                 /* mutant: truncation instead of RNE */
#else
    double n = nearbyint(r);             /* default mode: nearest, ties to even */
#endif
    double v = n * q;                    /* exact */
    float f = (float)v;                  /* exact, or +inf past the bf16 range */
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t h = (uint16_t)(u >> 16);
    if (neg)
        h |= 0x8000;
    return h;
}

/* ------------------------------------------------------- one output row -- */
/* Computes row m of A (row pointer a_row) against all N rows of B (b_base) and
 * returns the unrounded double accumulators in acc[N]. */
static void ref_row_f64(const uint8_t *a_row, const float *sa, int ld_sa, int m,
                        const uint8_t *b_base, const float *sb,
                        int N, int K, double *acc)
{
    int kb = K / 128;
    int ng = kb;
#if DG_REF_MUTANT == 1
    ng = kb - 1;                          /* mutant: last K group dropped */
#endif
    for (int n = 0; n < N; ++n) {
        const uint8_t *b_row = b_base + (size_t)n * K;
        double total = 0.0;
        for (int g = 0; g < ng; ++g) {
            double dot = 0.0;
            for (int k = 128 * g; k < 128 * g + 128; ++k) {
#if DG_REF_MUTANT == 6
                /* mutant: B read as if it were stored [K][N] */
                double bv = dg_ref_e4m3_to_double(b_base[(size_t)k * N + n]);
                (void)b_row;
#else
                double bv = dg_ref_e4m3_to_double(b_row[k]);
#endif
                dot += dg_ref_e4m3_to_double(a_row[k]) * bv;
            }
#if DG_REF_MUTANT == 3
            double s_a = (double)sa[(size_t)m * kb + g];   /* mutant: sa read row-major */
#else
            double s_a = (double)sa[(size_t)g * ld_sa + m];
#endif
#if DG_REF_MUTANT == 2
            double s_b = (double)sb[(size_t)g * ((N + 127) / 128) + n / 128]; /* mutant: sb transposed */
#else
            double s_b = (double)sb[(size_t)(n / 128) * kb + g];
#endif
#if DG_REF_MUTANT == 8
            total += dot * s_a;                  /* mutant: B scale dropped */
            (void)s_b;
#else
            total += dot * s_a * s_b;
#endif
        }
        acc[n] = total;
    }
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int dg_ref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* -------------------------------------------------------------- dense ---- */
/* Unrounded accumulators, [M][N] doubles.  Used by the pins that compare the
 * oracle with a library closed form before the final rounding. */
void dg_ref_gemm_nt_f64(const uint8_t *A, const float *sa, int ld_sa,
                        const uint8_t *B, const float *sb,
                        double *acc, int M, int N, int K, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; ++m)
        ref_row_f64(A + (size_t)m * K, sa, ld_sa, m, B, sb, N, K,
                    acc + (size_t)m * N);
}

/* Rows rows[0..nrows-1] of the dense product, written to D[i][N] (row i of D
 * holds output row rows[i]). */
void dg_ref_gemm_nt_rows(const uint8_t *A, const float *sa, int ld_sa,
                         const uint8_t *B, const float *sb,
                         uint16_t *D, int N, int K,
                         const int64_t *rows, int nrows, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        int m = (int)rows[i];
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        ref_row_f64(A + (size_t)m * K, sa, ld_sa, m, B, sb, N, K, acc);
        for (int n = 0; n < N; ++n)
            D[(size_t)i * N + n] = dg_ref_bf16_rne(acc[n]);
        free(acc);
    }
}

void dg_ref_gemm_nt(const uint8_t *A, const float *sa, int ld_sa,
                    const uint8_t *B, const float *sb,
                    uint16_t *D, int M, int N, int K, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; ++m) {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        ref_row_f64(A + (size_t)m * K, sa, ld_sa, m, B, sb, N, K, acc);
        for (int n = 0; n < N; ++n)
            D[(size_t)m * N + n] = dg_ref_bf16_rne(acc[n]);
        free(acc);
    }
}

/* ------------------------------------------------- with an addend C ----- */
/* D = C + A @ B^T (the GEMM naming convention of DeepGEMM,
 * es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de layout"),
 * here with C and D bf16 [M][N]: the bf16 C value, exact in double, is added
 * to the unrounded double sum, and the total is rounded once to bf16. */
void dg_ref_gemm_nt_c(const uint8_t *A, const float *sa, int ld_sa,
                      const uint8_t *B, const float *sb, const uint16_t *C,
                      uint16_t *D, int M, int N, int K, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; ++m) {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        ref_row_f64(A + (size_t)m * K, sa, ld_sa, m, B, sb, N, K, acc);
        for (int n = 0; n < N; ++n) {
            uint32_t u = (uint32_t)C[(size_t)m * N + n] << 16;
            float c;
            memcpy(&c, &u, 4);
#if DG_REF_MUTANT == 13
            (void)c;
            D[(size_t)m * N + n] = dg_ref_bf16_rne(acc[n]);   /* mutant: C dropped */
#else
            D[(size_t)m * N + n] = dg_ref_bf16_rne((double)c + acc[n]);
#endif
        }
        free(acc);
    }
}

/* ------------------------------------------------- grouped, contiguous --- */
/* A: [M_total][K]; B: [G][N][K]; sa: [kb][ld_sa]; sb: [G][nb][kb];
 * m_indices: [M_total], expert of each row or -1 (padding -> +0).
 * Computes the rows listed in rows[] (all rows when rows == NULL, nrows ==
 * M_total) into D[i][N]. */
void dg_ref_grouped_contiguous_rows(const uint8_t *A, const float *sa, int ld_sa,
                                    const uint8_t *B, const float *sb,
                                    const int32_t *m_indices,
                                    uint16_t *D, int N, int K, int num_groups,
                                    const int64_t *rows, int nrows, int nthreads)
{
    int kb = K / 128;
    int nb = (N + 127) / 128;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        int m = rows ? (int)rows[i] : i;
        int e = m_indices[m];
        uint16_t *drow = D + (size_t)i * N;
#if DG_REF_MUTANT == 9
        if (e < 0) e = 0;                 /* mutant: padding rows computed */
#endif
        if (e < 0 || e >= num_groups) {
            for (int n = 0; n < N; ++n)
                drow[n] = 0x0000;         /* +0 */
            continue;
        }
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        ref_row_f64(A + (size_t)m * K, sa, ld_sa, m,
                    B + (size_t)e * N * K, sb + (size_t)e * nb * kb, N, K, acc);
        for (int n = 0; n < N; ++n)
            drow[n] = dg_ref_bf16_rne(acc[n]);
        free(acc);
    }
}

/* --------------------------------------------------- grouped, masked ----- */
/* A: [G][max_m][K]; B: [G][N][K]; sa: [G][kb][ld_sa]; sb: [G][nb][kb];
 * D: [G][max_m][N], updated in place: rows m < masked_m[g] are computed, the
 * others keep whatever D held. */
void dg_ref_grouped_masked(const uint8_t *A, const float *sa, int ld_sa,
                           const uint8_t *B, const float *sb,
                           const int32_t *masked_m,
                           uint16_t *D, int num_groups, int max_m, int N, int K,
                           int nthreads)
{
    int kb = K / 128;
    int nb = (N + 127) / 128;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int g = 0; g < num_groups; ++g) {
        for (int m = 0; m < max_m; ++m) {
            int valid = masked_m[g];
#if DG_REF_MUTANT == 10
            valid = max_m;                /* mutant: mask ignored */
#endif
            if (m >= valid)
                continue;
            double *acc = (double *)malloc(sizeof(double) * (size_t)N);
            ref_row_f64(A + ((size_t)g * max_m + m) * K,
                        sa + (size_t)g * kb * ld_sa, ld_sa, m,
                        B + (size_t)g * N * K, sb + (size_t)g * nb * kb, N, K, acc);
            uint16_t *drow = D + ((size_t)g * max_m + m) * N;
            for (int n = 0; n < N; ++n)
                drow[n] = dg_ref_bf16_rne(acc[n]);
            free(acc);
        }
    }
}

/* ------------------------------------------- operand layouts ----------- */
/* The four storage layouts of the non-grouped GEMM, named after DeepGEMM's
 * fp8_gemm_{nt, nn, tn, tt} (es.news.hada.io/topic?id=19459, "Dense y Grouped
 * GEMM"; all four exist on SM100, "Interfaz GEMM y restricciones de layout").
 * The naming convention is D = C + A @ B with the letters saying whether each
 * stored operand enters transposed: "nt" is D = C + A @ B.T.  So
 *   A "n": stored [M][K], element (m, k) at A[m*K + k]
 *   A "t": stored [K][M], element (m, k) at A[k*M + m]
 *   B "t": stored [N][K], element (n, k) at B[n*K + k]
 *   B "n": stored [K][N], element (n, k) at B[k*N + n]
 * The scales do not depend on the storage: sa[g*ld_sa + m] per (row, K group),
 * sb[(n/128)*kb + g] per 128x128 block of (n, k). */
static double ref_elem(const uint8_t *A, int a_t, const float *sa, int ld_sa,
                       const uint8_t *B, int b_n, const float *sb, int kb_all,
                       int M, int N, int K, int m, int n, int g0, int g1)
{
    double total = 0.0;
    for (int g = g0; g < g1; ++g) {
        double dot = 0.0;
        for (int k = 128 * g; k < 128 * g + 128; ++k) {
#if DG_REF_MUTANT == 15
            uint8_t a = A[(size_t)m * K + k];        /* mutant: A's storage ignored */
            (void)a_t;
#else
            uint8_t a = a_t ? A[(size_t)k * M + m] : A[(size_t)m * K + k];
#endif
            uint8_t b = b_n ? B[(size_t)k * N + n] : B[(size_t)n * K + k];
            dot += dg_ref_e4m3_to_double(a) * dg_ref_e4m3_to_double(b);
        }
        total += dot * (double)sa[(size_t)g * ld_sa + m] * (double)sb[(size_t)(n / 128) * kb_all + g];
    }
    return total;
}

static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* D [M][N] = bf16(C + A @ B) in the layout (a_t, b_n) above; C [M][N] bf16 or
 * NULL (no addend). */
void dg_ref_gemm_layout(const uint8_t *A, int a_t, const float *sa, int ld_sa,
                        const uint8_t *B, int b_n, const float *sb,
                        const uint16_t *C, uint16_t *D, int M, int N, int K, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = ref_elem(A, a_t, sa, ld_sa, B, b_n, sb, K / 128, M, N, K, m, n, 0, K / 128);
            double c = C ? bf16_bits_to_double(C[(size_t)m * N + n]) : 0.0;
            D[(size_t)m * N + n] = dg_ref_bf16_rne(c + acc);
        }
}

/* ----------------------------------------------- K-grouped ("tn") -------- */
/* The K-grouped GEMM for the MoE weight gradient (k_grouped_fp8_gemm_tn_contiguous,
 * same page, "Dense y Grouped GEMM": M and N fixed, the groups concatenated
 * along K).  Group g owns K rows [k0_g, k0_g + ks[g]) with k0_g = ks[0] + ... +
 * ks[g-1], each ks[g] a multiple of 128 (whole K groups):
 *   D[g][m][n] = bf16( C[g][m][n] + sum over the K groups j of group g of
 *                      (sum_{k in j} dec(A[k][m]) dec(B[k][n])) sa[j][m] sb[n/128][j] )
 * A: [K_all][M] ("t"), B: [K_all][N] ("n"), sa: [K_all/128][ld_sa],
 * sb: [ceil(N/128)][K_all/128], C and D: [G][M][N] (C may be NULL).  A group
 * with ks[g] = 0 gives D = C (or +0). */
void dg_ref_k_grouped_tn(const uint8_t *A, const float *sa, int ld_sa,
                         const uint8_t *B, const float *sb, const uint16_t *C,
                         uint16_t *D, int M, int N, const int32_t *ks, int num_groups,
                         int nthreads)
{
    int K_all = 0;
    for (int g = 0; g < num_groups; ++g)
        K_all += ks[g];
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int g = 0; g < num_groups; ++g)
        for (int m = 0; m < M; ++m) {
            int k0 = 0;
            for (int h = 0; h < g; ++h)
                k0 += ks[h];
#if DG_REF_MUTANT == 14
            if (g > 0 && k0 >= 128)
                k0 -= 128;                /* mutant: segment starts a K group early */
#endif
            int g0 = k0 / 128, g1 = (k0 + ks[g]) / 128;
            for (int n = 0; n < N; ++n) {
                double acc = ref_elem(A, 1, sa, ld_sa, B, 1, sb, K_all / 128, M, N, K_all, m, n,
                                      g0, g1);
                size_t o = ((size_t)g * M + m) * N + n;
                double c = C ? bf16_bits_to_double(C[o]) : 0.0;
                D[o] = dg_ref_bf16_rne(c + acc);
            }
        }
}

/* ------------------------------------------------ activation quantiser -- */
/* The step that produces the GEMM's left operand: each row of a bf16
 * activation matrix is cut into 128-wide K groups, and each (row, group) gets
 * one fp32 scale and 128 e4m3 codes.  The pages state the layout of the
 * result (the LHS scales fp32 and K-group-major, "transposed", TMA-aligned:
 * es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de layout")
 * and, in the same section, leave the FP8 conversion to the caller, without
 * fixing its arithmetic.  The reading taken here, all in fp32:
 *
 *   amax     = max |x[m,k]| over the group              (exact)
 *   a        = max(amax, 1e-4)
 *   sa[g][m] = a / 448                                   (fp32 division)
 *   q[m,k]   = e4m3_rne_satfinite( x[m,k] * (448 / a) )   (fp32 division once,
 *                                                          fp32 multiply each)
 *
 * 448 is the largest finite e4m3 value, so the largest |x| of a group maps to
 * code magnitude 448.  Inputs are finite. */

/* fp32 -> e4m3 ("fn"): round to nearest, ties to even, saturating to +-448
 * (the format has no infinity); NaN gives 0x7F.  Written from the format
 * definition: normal values (1 + f/8) * 2^(e-7) have spacing 2^(E-3) in
 * [2^E, 2^(E+1)); below 2^-6 the spacing stays 2^-9 (subnormals). */
uint8_t dg_ref_e4m3_from_float(float v)
{
    if (isnan(v))
        return 0x7F;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs((double)v);          /* exact */
    uint8_t code;
    if (a >= 448.0) {
        code = 0x7E;                     /* saturate: S.1111.110 = 448 */
    } else if (a < ldexp(1.0, -6)) {
        /* subnormal range; n = 8 is the smallest normal value, code 0x08 */
#if DG_REF_MUTANT == 12
        double n = floor(a / ldexp(1.0, -9));    /* mutant: truncation */
#else
        double n = nearbyint(a / ldexp(1.0, -9));
#endif
        code = (uint8_t)n;
    } else {
        int ex;
        frexp(a, &ex);                   /* a in [2^(ex-1), 2^ex) */
        int E = ex - 1;
#if DG_REF_MUTANT == 12
        double n = floor(a / ldexp(1.0, E - 3)); /* mutant: truncation */
#else
        double n = nearbyint(a / ldexp(1.0, E - 3));   /* 8..16, exact division */
#endif
        if (n >= 16.0) {                 /* rounded up into the next binade */
            E += 1;
            n = 8.0;
        }
        code = (uint8_t)(((E + 7) << 3) | ((int)n - 8));   /* a < 448: E <= 8 */
    }
    return neg ? (uint8_t)(code | 0x80) : code;
}

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* X: bf16 bit patterns [G][M][K]; Q: e4m3 codes [G][M][K];
 * sa: [G][K/128][ld_sa], columns m < M written. */
void dg_ref_quantize_1x128(const uint16_t *X, uint8_t *Q, float *sa, int num_groups, int M,
                           int K, int ld_sa, int nthreads)
{
    int kb = K / 128;
    set_threads(nthreads);
#pragma omp parallel for schedule(static) collapse(2)
    for (int z = 0; z < num_groups; ++z) {
        for (int m = 0; m < M; ++m) {
            for (int g = 0; g < kb; ++g) {
                const uint16_t *x = X + ((size_t)z * M + m) * K + (size_t)g * 128;
                uint8_t *q = Q + ((size_t)z * M + m) * K + (size_t)g * 128;
                float amax = 0.0f;
                for (int k = 0; k < 128; ++k) {
                    float v = fabsf(bf16_bits_to_float(x[k]));
                    if (v > amax)
                        amax = v;
                }
                float a = amax > 1e-4f ? amax : 1e-4f;
#if DG_REF_MUTANT == 11
                float scale = a;                  /* mutant: 448 left out */
                float factor = 1.0f / a;
#else
                float scale = a / 448.0f;
                float factor = 448.0f / a;
#endif
                for (int k = 0; k < 128; ++k)
                    q[k] = dg_ref_e4m3_from_float(bf16_bits_to_float(x[k]) * factor);
                sa[((size_t)z * kb + g) * ld_sa + m] = scale;
            }
        }
    }
}

/* ------------------------------------------------ UE8M0 packed scales ---- */
/* The scale format of DeepGEMM's SM100 kernels (es.news.hada.io/topic?id=19459,
 * "Interfaz GEMM y restricciones de layout": packed UE8M0, four per 32-bit
 * integer).  UE8M0 is an unsigned 8-bit exponent with bias 127 (the E8M0
 * scale type of the OCP microscaling formats): code e is 2^(e - 127), and
 * 0xFF is NaN.  Packing: the four K groups 4i .. 4i+3 of one row share a
 * 32-bit word, group 4i + j in bits 8j .. 8j+7.
 *   sfa: [ceil(kb/4)][ld] words, word (i, m) = groups 4i.. of row m
 *   sfb: [nb][ceil(kb/4)] words, word (b, i) = groups 4i.. of the 128-row block b
 * The decoders below turn them into the fp32 scales of the main formula
 * (every UE8M0 value but NaN is exact in fp32, 2^-127 as a subnormal). */
double dg_ref_ue8m0_to_double(uint8_t e)
{
    if (e == 0xFF)
        return NAN;
#if DG_REF_MUTANT == 16
    return ldexp(1.0, (int)e - 128);      /* mutant: bias 128 */
#else
    return ldexp(1.0, (int)e - 127);
#endif
}

static uint8_t packed_byte(int32_t word, int j)
{
#if DG_REF_MUTANT == 17
    j = 3 - j;                            /* mutant: bytes taken in reverse order */
#endif
    return (uint8_t)(((uint32_t)word >> (8 * j)) & 0xFFu);
}

/* sa[g*ld + m] = scale of (row m, K group g), for g < kb and m < ld */
void dg_ref_decode_sfa(const int32_t *sfa, float *sa, int kb, int ld)
{
    for (int g = 0; g < kb; ++g)
        for (int m = 0; m < ld; ++m)
            sa[(size_t)g * ld + m] =
                (float)dg_ref_ue8m0_to_double(packed_byte(sfa[(size_t)(g / 4) * ld + m], g % 4));
}

/* sb[b*kb + g] = scale of (block b, K group g) */
void dg_ref_decode_sfb(const int32_t *sfb, float *sb, int nb, int kb)
{
    int kbp = (kb + 3) / 4;
    for (int b = 0; b < nb; ++b)
        for (int g = 0; g < kb; ++g)
            sb[(size_t)b * kb + g] =
                (float)dg_ref_ue8m0_to_double(packed_byte(sfb[(size_t)b * kbp + g / 4], g % 4));
}

/* The 1x128 quantiser with UE8M0 scales (the scale rounded up to a power of
 * two, so that it is exact in the packed format).  In fp32, per row and
 * K group: a = max(amax, 1e-4); t = a / 448 (one rounding); s = the smallest
 * power of two >= t; Q = e4m3 (round to nearest even, saturating) of x / s,
 * exact division by a power of two.  The exponent byte 127 + log2(s) goes to
 * byte g % 4 of word sfa[g/4][m]; bytes of groups past K/128 are left as they
 * were.  X, Q as in dg_ref_quantize_1x128; sfa: [G][ceil(kb/4)][ld] words. */
void dg_ref_quantize_1x128_ue8m0(const uint16_t *X, uint8_t *Q, int32_t *sfa, int num_groups,
                                 int M, int K, int ld, int nthreads)
{
    int kb = K / 128, kbp = (kb + 3) / 4;
    set_threads(nthreads);
#pragma omp parallel for schedule(static) collapse(2)
    for (int z = 0; z < num_groups; ++z)
        for (int m = 0; m < M; ++m) {
            const uint16_t *xr = X + ((size_t)z * M + m) * K;
            uint8_t *qr = Q + ((size_t)z * M + m) * K;
            for (int g = 0; g < kb; ++g) {
                float amax = 0.0f;
                for (int k = 128 * g; k < 128 * g + 128; ++k) {
                    float v = fabsf(bf16_bits_to_float(xr[k]));
                    if (v > amax)
                        amax = v;
                }
                float a = amax > 1e-4f ? amax : 1e-4f;
                float t = a / 448.0f;
                int ex;
                float f = frexpf(t, &ex);         /* t = f * 2^ex, f in [0.5, 1) */
#if DG_REF_MUTANT == 18
                int lg = ex - 1;                  /* mutant: rounded down, not up */
                (void)f;
#else
                int lg = (f == 0.5f) ? ex - 1 : ex;   /* log2 of the power-of-two ceiling */
#endif
                float inv = ldexpf(1.0f, -lg);
                for (int k = 128 * g; k < 128 * g + 128; ++k)
                    qr[k] = dg_ref_e4m3_from_float(bf16_bits_to_float(xr[k]) * inv);
                uint8_t *word = (uint8_t *)(sfa + ((size_t)z * kbp + g / 4) * ld + m);
                word[g % 4] = (uint8_t)(127 + lg);   /* little-endian: byte j = bits 8j.. */
            }
        }
}
