/*
 * Float64 CPU oracle for the FP32 matrix multiply C = A·B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code with the CUDA path.
 *
 * What it computes, from the pages' definition of the product:
 *   "3 · La mémoire partagée", §3.1 "Le problème que ça résout": each output
 *   C[lig][col] is the sum over k of A[lig][k]·B[k][col], one multiply and
 *   one add per k, 2N³ operations for N×N; and "共享内存与同步" (cuda-oxide),
 *   section "SharedArray —— 静态共享内存" (tiled_sgemm): general m×k times
 *   k×n with A read as a[row*k + i] and B as b[i*n + col], row-major.
 * Every kernel on those pages overwrites C (no alpha, no beta).
 *
 *   C_ref[i][j]  = sum_{k=0}^{K-1} (double)A[i][k] * (double)B[k][j]
 *   bound[i][j]  = sum_{k=0}^{K-1} |A[i][k]| * |B[k][j]|     (float64)
 *
 * The k sum runs in ascending k for every element.  The loop nest is i-k-j
 * with a float64 row accumulator; that changes no element's summation order
 * relative to the i-j-k triple loop, it only walks B by rows.
 * K = 0 gives the empty sum, 0.  M = 0 or N = 0 writes nothing.
 *
 * Build with -O2 -fno-fast-math -ffp-contract=off so no multiply-add is
 * fused: the x86 host and the aarch64 GPU host then give identical bits.
 *
 * ORACLE_MUTANT (compile-time, tests only) plants one plausible mistake so
 * the tests can show their pins catch it; 0 (the default) is the oracle.
 *   1 drops the last k term, 2 reads B transposed (B[j][k], the flat index
 *   wrapped into B's extent so the mistake stays in bounds),
 *   3 subtracts odd-k terms, 4 reads A one row too high (wraps at M-1),
 *   5 accumulates in float32 instead of float64; 6-8 break the 16-bit
 *   rounding (see oracle_round_half).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#if ORACLE_MUTANT == 5
typedef float acc_t;
#else
typedef double acc_t;
#endif

/* Element (i, k) of A and (k, j) of B as the definition reads them.  The
 * mutants change only these reads, the range of k or the sign. */
static inline double a_at(const float *A, int64_t lda, int64_t M, int64_t i,
                          int64_t k) {
#if ORACLE_MUTANT == 4
    int64_t r = (i + 1 < M) ? i + 1 : i;
    return (double)A[r * lda + k];
#else
    (void)M;
    return (double)A[i * lda + k];
#endif
}

static inline double b_at(const float *B, int64_t ldb, int64_t K, int64_t k,
                          int64_t j) {
#if ORACLE_MUTANT == 2
    return (double)B[(j * ldb + k) % (K * ldb)];
#else
    (void)K;
    return (double)B[k * ldb + j];
#endif
}

static inline int64_t k_end(int64_t K) {
#if ORACLE_MUTANT == 1
    return K > 0 ? K - 1 : 0;
#else
    return K;
#endif
}

static inline double term_sign(int64_t k) {
#if ORACLE_MUTANT == 3
    return (k & 1) ? -1.0 : 1.0;
#else
    (void)k;
    return 1.0;
#endif
}

/*
 * Full product.  C (M×N, leading dimension ldc) receives C_ref; bound, when
 * not NULL, receives the matching sum of magnitudes with the same ldc.
 * nthreads <= 0 uses the OpenMP default.  Returns the number of
 * multiply-adds performed (M·N·K for the oracle), or -1 on bad arguments.
 */
int64_t oracle_gemm_f64(int64_t M, int64_t N, int64_t K, const float *A,
                        int64_t lda, const float *B, int64_t ldb, double *C,
                        int64_t ldc, double *bound, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N) return -1;
    if (M == 0 || N == 0) return 0;
    int64_t fmas = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel reduction(+ : fmas)
    {
        acc_t *row = (acc_t *)malloc(sizeof(acc_t) * (size_t)N);
        double *mag = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < M; ++i) {
            for (int64_t j = 0; j < N; ++j) {
                row[j] = 0;
                mag[j] = 0.0;
            }
            const int64_t kend = k_end(K);
            for (int64_t k = 0; k < kend; ++k) {
                const double a = a_at(A, lda, M, i, k) * term_sign(k);
                for (int64_t j = 0; j < N; ++j) {
                    const double b = b_at(B, ldb, K, k, j);
                    row[j] += (acc_t)(a * b);
                    mag[j] += fabs(a) * fabs(b);
                }
                fmas += N;
            }
            for (int64_t j = 0; j < N; ++j) C[i * ldc + j] = (double)row[j];
            if (bound)
                for (int64_t j = 0; j < N; ++j) bound[i * ldc + j] = mag[j];
        }
        free(row);
        free(mag);
    }
    return fmas;
}

/*
 * Selected elements only: out[t] = C_ref[rows[t]][cols[t]] (and its bound),
 * for checking a few outputs of a product too large to compute whole.
 * Returns the number of multiply-adds, or -1 on bad arguments.
 */
int64_t oracle_gemm_f64_entries(int64_t M, int64_t N, int64_t K,
                                const float *A, int64_t lda, const float *B,
                                int64_t ldb, int64_t count, const int64_t *rows,
                                const int64_t *cols, double *out,
                                double *bound) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || count < 0) return -1;
    int64_t fmas = 0;
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return -1;
        acc_t s = 0;
        double m = 0.0;
        const int64_t kend = k_end(K);
        for (int64_t k = 0; k < kend; ++k) {
            const double a = a_at(A, lda, M, i, k) * term_sign(k);
            const double b = b_at(B, ldb, K, k, j);
            s += (acc_t)(a * b);
            m += fabs(a) * fabs(b);
            ++fmas;
        }
        out[t] = (double)s;
        if (bound) bound[t] = m;
    }
    return fmas;
}

/* Threads OpenMP would use for oracle_gemm_f64 with nthreads <= 0. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Epilogue of the fused product C = act(A·B + bias), applied to an oracle
 * product: out[i][j] = act(C[i][j] + bias[j]) in float64 (bias may be NULL).
 * act 0 is the identity; act 1 is GELU, x·Φ(x) = x/2·(1 + erf(x/√2)) with Φ
 * the standard normal distribution function.  The pages name GELU (its own
 * kernel in "Rendre le GPU rapide", "Les kernels fusionnés") and the fused
 * bias add (same article, "Et par rapport à PyTorch ?") without a formula;
 * this is GELU's definition.  C and out may be the same array.
 */
int oracle_epilogue_f64(int64_t M, int64_t N, const double *C, int64_t ldc,
                        const float *bias, int act, double *out,
                        int64_t ldo) {
    if (M < 0 || N < 0 || ldc < N || ldo < N || act < 0 || act > 1) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double z = C[i * ldc + j] + (bias ? (double)bias[j] : 0.0);
            if (act == 1) z = 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
            out[i * ldo + j] = z;
        }
    return 0;
}

/*
 * Operand rounding of the mixed-precision product ("Rendre le GPU rapide",
 * "Les Tensor Cores"): only the two operands of the multiply are rounded to
 * a 16-bit float; every sum and every tensor stays float32.  The oracle of
 * that product is therefore oracle_gemm_f64 applied to the operands after
 * oracle_round_half and oracle_widen_half (widening is exact).
 *
 * type 0, bfloat16: the upper 16 bits of the float32 pattern, rounded to
 *   nearest with ties to even the way the pages do it: add 0x7FFF plus the
 *   lowest kept bit to the 32-bit pattern, then drop the low 16 bits.
 *   Overflow carries into the exponent and yields ±Inf, as IEEE rounding
 *   does.  The pages do not treat NaN (the carry could turn a NaN pattern
 *   into Inf or a wrapped sign); here a NaN stays a quiet NaN.
 * type 1, IEEE binary16 (1 sign, 5 exponent bits with bias 15, 10 stored
 *   significand bits), from the format's definition: |x| >= 65520 (halfway
 *   between 65504 and 2^16, which ties to the even 2^16) gives ±Inf;
 *   otherwise |x| is rounded to the nearest multiple of its quantum
 *   2^(e-10), e = max(floor(log2|x|), -14), ties to an even multiple.
 *   Below 2^-14 the quantum stays 2^-24 (gradual underflow).
 *
 * ORACLE_MUTANT 6 rounds bfloat16 by truncation; 7 breaks binary16 ties
 * away from zero; 8 flushes values below 2^-14 to zero (no gradual
 * underflow).
 */
static uint16_t round_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);          /* NaN, quiet */
#if ORACLE_MUTANT == 6
    return (uint16_t)(u >> 16);
#else
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
#endif
}

static uint16_t round_f16(float x) {
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    const double a = fabs((double)x);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);  /* also ±Inf */
    if (a == 0.0) return sign;
    int ex;
    (void)frexp(a, &ex);               /* a = m·2^ex, m in [0.5, 1) */
    int e = ex - 1;                    /* floor(log2 a) */
#if ORACLE_MUTANT == 8
    if (e < -14) return sign;
#endif
    if (e < -14) e = -14;
    const double r = ldexp(a, 10 - e); /* a / quantum, exact */
    double n = floor(r);
    const double d = r - n;            /* exact: r has at most 24 bits */
#if ORACLE_MUTANT == 7
    if (d >= 0.5) n += 1.0;
#else
    if (d > 0.5 || (d == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
#endif
    if (e == -14 && n <= 1024.0)       /* subnormal, or 2^-14 exactly */
        return (uint16_t)(sign | (uint16_t)n);
    if (n == 2048.0) {                 /* rounded up to the next binade */
        n = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) |
                      (uint16_t)(n - 1024.0));
}

/* dst[i][j] = round(src[i][j]) for a rows×cols block; row strides in
 * elements.  Returns 0, or -1 for bad arguments. */
int oracle_round_half(int type, int64_t rows, int64_t cols, const float *src,
                      int64_t lds, uint16_t *dst, int64_t ldd) {
    if ((type != 0 && type != 1) || rows < 0 || cols < 0 || lds < cols ||
        ldd < cols)
        return -1;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j)
            dst[i * ldd + j] = type == 0 ? round_bf16(src[i * lds + j])
                                         : round_f16(src[i * lds + j]);
    return 0;
}

/* dst[t] = the float32 value of the 16-bit pattern src[t] (exact). */
int oracle_widen_half(int type, int64_t n, const uint16_t *src, float *dst) {
    if ((type != 0 && type != 1) || n < 0) return -1;
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t h = src[t];
        float v;
        if (type == 0) {
            const uint32_t u = (uint32_t)h << 16;
            memcpy(&v, &u, 4);
        } else {
            const int E = (h >> 10) & 31, F = h & 1023;
            double m;
            if (E == 0) m = ldexp((double)F, -24);
            else if (E == 31) m = F ? NAN : INFINITY;
            else m = ldexp((double)(1024 + F), E - 25);
            v = (float)((h & 0x8000u) ? -m : m);
        }
        dst[t] = v;
    }
    return 0;
}
