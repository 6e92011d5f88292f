/*
 * CPU oracle for the shape-driven half-precision GEMM and the M=1 decode GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (plain definitions, accumulated in fp64):
 *
 *  - GEMM   C[i][j] = sum_k A[i][k] * B[k][j]
 *      "Beating hipBLASLt on a Gaming GPU", section "The result": a square
 *      fp16 GEMM, fp16 inputs with higher-precision accumulation.  A is
 *      row-major MxK, B is row-major KxN (both IEEE binary16 bit patterns).
 *      Every fp16 value is exact in fp64 and every product of two fp16 values
 *      (11 x 11 significant bits) is exact in fp64, so the only rounding is in
 *      the fp64 running sum.  Loop order i-k-j with one fp64 row accumulator.
 *
 *  - GEMV bf16   y[n] = sum_k x[k] * W[n][k]
 *      "mojo-baro", section "Four rounds on the decode shape": M=1, K=4096,
 *      N=12288 skinny GEMM with the weights stored K-major (the "B-layout"
 *      of round v1).  x and W are bfloat16 bit patterns.
 *
 *  - GEMV q8     y[n] = sum_g s[n][g] * sum_{k in group g} x[k] * q[n][k]
 *      "mojo-baro", round v2 ("K-major q8"): int8 weights with one scale per
 *      32 consecutive K-elements.  The scale is an fp16 bit pattern, one per
 *      (row, group), stored [N][K/32].  The group sum is formed first and then
 *      scaled, which is the order the description reads in.
 *
 *  - The same GEMM on bfloat16 operands (the FlyDSL pull request "Speed up
 *    the RDNA3 GEMM up to 1.85x by choosing the tile from the shape",
 *    section "Performance", measures bf16).
 *
 *  - fp16 and bf16 decoding and fp64 -> fp16 / bf16 round-to-nearest-even
 *    encoders, written from the IEEE 754 binary16 and the bfloat16
 *    definitions; they are used to compare against the GPU's 16-bit output bit
 *    for bit on integer-valued inputs.
 *
 * Build: plain C99 with OpenMP across output rows (which does not change the
 * order of any single output's sum).  Compile with -ffp-contract=off so that
 * x86 and Arm give identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- number formats ----------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double sdt_oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 1024), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
double sdt_oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest binary16, ties to even. */
uint16_t sdt_oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00u;
    if (isinf(x)) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the quantum is 2^-24; a result of 1024 quanta is
         * the smallest normal number, whose bit pattern is exactly 0x0400. */
        double q = nearbyint(ldexp(a, 24));     /* default mode: ties to even */
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    frexp(a, &e2);                              /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;                             /* a in [2^E, 2^(E+1)) */
    double q = nearbyint(ldexp(a, 10 - E));     /* significand in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024));
}

/* Round an fp64 value to the nearest bfloat16 (8 significant bits, binary32
 * exponent range), ties to even.  Written from the format's definition: the
 * significand is rounded to 8 bits at the value's binary exponent; below the
 * smallest normal (2^-126) the quantum is fixed at 2^-133. */
uint16_t sdt_oracle_f64_to_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7fc0u;
    if (isinf(x)) return (uint16_t)(sign | 0x7f80u);
    if (a < ldexp(1.0, -126)) {
        double q = nearbyint(ldexp(a, 133));      /* subnormal quantum 2^-133 */
        return (uint16_t)(sign | (uint16_t)q);    /* q == 128 is the smallest normal */
    }
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;                               /* a in [2^E, 2^(E+1)) */
    double q = nearbyint(ldexp(a, 7 - E));        /* significand in [128, 256] */
    if (q == 256.0) { q = 128.0; E += 1; }
    if (E > 127) return (uint16_t)(sign | 0x7f80u);
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)((int)q - 128));
}

void sdt_oracle_f64_array_to_bf16(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = sdt_oracle_f64_to_bf16(x[i]);
}

void sdt_oracle_f16_array_to_f64(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = sdt_oracle_f16_to_f64(h[i]);
}

void sdt_oracle_bf16_array_to_f64(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = sdt_oracle_bf16_to_f64(h[i]);
}

void sdt_oracle_f64_array_to_f16(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = sdt_oracle_f64_to_f16(x[i]);
}

/* ---- GEMM --------------------------------------------------------------- */

/*
 * C[r][j] for the requested rows only: rows[r] is the row index into A (so a
 * sample of rows can be checked at sizes where the full product is too slow).
 * rows == NULL means all M rows in order.  C is n_rows x N, fp64.
 * threads <= 0 uses the OpenMP default.  Returns 0, or -1 on bad arguments or
 * allocation failure.
 */
/* dtype 0: A and B hold IEEE binary16 patterns; dtype 1: bfloat16 patterns. */
static double sdt_oracle_decode(uint16_t v, int dtype)
{
    return dtype ? sdt_oracle_bf16_to_f64(v) : sdt_oracle_f16_to_f64(v);
}

int sdt_oracle_gemm_rows_t(int64_t M, int64_t N, int64_t K,
                           const uint16_t *A, const uint16_t *B,
                           const int64_t *rows, int64_t n_rows,
                           double *C, int threads, int dtype)
{
    if (M < 0 || N < 0 || K < 0 || n_rows < 0 || (dtype != 0 && dtype != 1)) return -1;
    if (n_rows == 0 || N == 0) return 0;
    if (!A || !B || !C) return -1;
    double *Bd = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    if (!Bd) return -1;
    for (int64_t t = 0; t < K * N; ++t) Bd[t] = sdt_oracle_decode(B[t], dtype);
    int bad = 0;
#ifdef _OPENMP
    /* the count applies to this loop only (no process-wide setting is changed) */
    const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad) num_threads(nt)
#endif
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) { bad |= 1; continue; }
        double *acc = C + r * N;
        for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = sdt_oracle_decode(A[i * K + k], dtype);
            const double *brow = Bd + k * N;
            for (int64_t j = 0; j < N; ++j) acc[j] += a * brow[j];
        }
    }
    free(Bd);
    return bad ? -1 : 0;
}

int sdt_oracle_gemm_rows(int64_t M, int64_t N, int64_t K,
                         const uint16_t *A, const uint16_t *B,
                         const int64_t *rows, int64_t n_rows,
                         double *C, int threads)
{
    return sdt_oracle_gemm_rows_t(M, N, K, A, B, rows, n_rows, C, threads, 0);
}

int sdt_oracle_gemm(int64_t M, int64_t N, int64_t K,
                    const uint16_t *A, const uint16_t *B, double *C, int threads)
{
    return sdt_oracle_gemm_rows(M, N, K, A, B, NULL, M, C, threads);
}

/* ---- GEMV (M = 1 decode) ------------------------------------------------ */

/* W is K-major: row n holds W[n][0..K-1] contiguously. */
int sdt_oracle_gemv_bf16(int64_t K, int64_t N, const uint16_t *x,
                         const uint16_t *W, double *y, int threads)
{
    if (K < 0 || N < 0) return -1;
    if (N == 0) return 0;
    if (!x || !W || !y) return -1;
    double *xd = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    if (!xd) return -1;
    for (int64_t k = 0; k < K; ++k) xd[k] = sdt_oracle_bf16_to_f64(x[k]);
#ifdef _OPENMP
    const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += xd[k] * sdt_oracle_bf16_to_f64(W[n * K + k]);
        y[n] = acc;
    }
    free(xd);
    return 0;
}

/* q is int8 [N][K]; s holds fp16 scales [N][K/32]; K must be a multiple of 32. */
int sdt_oracle_gemv_q8(int64_t K, int64_t N, const uint16_t *x,
                       const int8_t *q, const uint16_t *s, double *y, int threads)
{
    const int64_t G = 32;
    if (K < 0 || N < 0 || K % G != 0) return -1;
    if (N == 0) return 0;
    if (!x || !q || !s || !y) return -1;
    double *xd = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    if (!xd) return -1;
    for (int64_t k = 0; k < K; ++k) xd[k] = sdt_oracle_bf16_to_f64(x[k]);
    const int64_t n_groups = K / G;
#ifdef _OPENMP
    const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t g = 0; g < n_groups; ++g) {
            double part = 0.0;
            for (int64_t k = g * G; k < (g + 1) * G; ++k)
                part += xd[k] * (double)q[n * K + k];
            acc += sdt_oracle_f16_to_f64(s[n * n_groups + g]) * part;
        }
        y[n] = acc;
    }
    free(xd);
    return 0;
}

int sdt_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
