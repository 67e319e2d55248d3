/*
 * oracle_gemm.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the GPU path
 * computes.  Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of
 * bench.py may load this code; the library under dense_tensor_core_bf16_gb300/
 * never does, and nothing here is shared with it.
 *
 * What it follows
 *   - "10. Tensor Cores, shapes, and tile alignment", section "Shape the
 *     operation": C (M x N) = A (M x K) B (K x N); useful work 2MNK.
 *   - "The Tensor Core" lesson (0011), paragraph on mixed precision and the
 *     WMMA walk-through: low-precision inputs, products accumulated in a wider
 *     type, the k sweep starting from a zero accumulator (D = A x B + C with
 *     C = 0).
 * Reading: the exact result is the definition sum_k a_ik * b_kj.  Every bf16
 * input is widened exactly to binary64; products of two bf16 values are exact
 * in binary64 (8 x 8 significant bits), and the sum is taken left to right in
 * increasing k in binary64.  That is the reference value; the GPU's fp32
 * accumulation is judged against it with an error bound, not bit for bit
 * (except where every partial sum is an integer below 2^24).
 *
 * Pins (tests/test_oracle_pins.py): exact rational brute force on tiny
 * shapes, identity and permutation products, small-integer inputs against an
 * int64 triple loop, and numpy's binary64 matmul as an independent library
 * routine.  The binary64 -> bf16 rounding below is pinned by hand-picked bit
 * patterns and by a brute-force nearest-value search over all 65536 bf16
 * encodings.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> binary64, exact: a bf16 value is the upper half of a
 * binary32 encoding, and binary32 -> binary64 widening is exact. */
double oracle_bf16_to_f64(uint16_t h) {
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* binary64 -> bf16, round to nearest, ties to even, straight from the
 * IEEE 754 definition (never through binary32, which would round twice).
 *
 * bf16 has 8 significant bits (7 stored) and binary32's exponent range, so
 * for a finite x the spacing of representable values around |x| is
 * q = 2^(max(e, -126) - 7) where 2^e <= |x| < 2^(e+1); below 2^-126 the
 * spacing is the subnormal quantum 2^-133.  x / q is exact (q is a power of
 * two and the quotient stays in range), nearbyint() in the default rounding
 * mode rounds it to the nearest integer with ties to even, and the product
 * back by q is exact.  A result of 2^128 or more is past the largest finite
 * bf16 ((2 - 2^-7) * 2^127) and becomes infinity. */
uint16_t oracle_f64_to_bf16_rne(double x) {
    if (isnan(x)) {
        return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    }
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    double ax = fabs(x);
    if (isinf(ax)) return (uint16_t)(sign | 0x7F80u);
    if (ax == 0.0) return sign;
    int e2;
    (void)frexp(ax, &e2);          /* ax = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                 /* 2^e <= ax < 2^(e+1) */
    if (e < -126) e = -126;
    double q = ldexp(1.0, e - 7);
    double n = nearbyint(ax / q);
    double r = n * q;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    float rf = (float)r;            /* exact: r is a bf16 value */
    uint32_t w;
    memcpy(&w, &rf, sizeof w);
    return (uint16_t)(sign | (uint16_t)(w >> 16));
}

void oracle_f64_to_bf16_rne_array(const double *x, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16_rne(x[i]);
}

void oracle_bf16_to_f64_array(const uint16_t *h, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(h[i]);
}

/* Element (i, k) of A and element (k, j) of B for either storage order.
 * Row-major X with leading dimension ld: X[r][c] at X[r*ld + c].
 * Column-major: X[r][c] at X[c*ld + r]. */
static double a_elem(const uint16_t *A, int64_t lda, int a_col_major, int64_t i, int64_t k) {
    return oracle_bf16_to_f64(a_col_major ? A[k * lda + i] : A[i * lda + k]);
}
static double b_elem(const uint16_t *B, int64_t ldb, int b_col_major, int64_t k, int64_t j) {
    return oracle_bf16_to_f64(b_col_major ? B[j * ldb + k] : B[k * ldb + j]);
}

/* One output: C[i][j] = sum_{k=0}^{K-1} a_ik * b_kj, in increasing k, binary64;
 * *sabs = sum_k |a_ik * b_kj| (the scale of the error bound). */
static void dot_one(int64_t K, const uint16_t *A, int64_t lda, int a_cm,
                    const uint16_t *B, int64_t ldb, int b_cm,
                    int64_t i, int64_t j, double *c, double *sabs) {
    double acc = 0.0, abs_acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = a_elem(A, lda, a_cm, i, k) * b_elem(B, ldb, b_cm, k, j);
        acc += p;
        abs_acc += fabs(p);
    }
    *c = acc;
    if (sabs) *sabs = abs_acc;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full product.  C and Sabs (may be NULL) are row-major M x N with leading
 * dimension ldc.  Rows are spread over OpenMP threads; each output is still
 * one left-to-right sum. */
void oracle_gemm(int64_t M, int64_t N, int64_t K,
                 const uint16_t *A, int64_t lda, int a_col_major,
                 const uint16_t *B, int64_t ldb, int b_col_major,
                 double *C, double *Sabs, int64_t ldc, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double c, s;
            dot_one(K, A, lda, a_col_major, B, ldb, b_col_major, i, j, &c, &s);
            C[i * ldc + j] = c;
            if (Sabs) Sabs[i * ldc + j] = s;
        }
    }
}

/* Selected outputs (rows[t], cols[t]) for t < n, for shapes too large to
 * compute in full. */
void oracle_gemm_entries(int64_t K,
                         const uint16_t *A, int64_t lda, int a_col_major,
                         const uint16_t *B, int64_t ldb, int b_col_major,
                         const int64_t *rows, const int64_t *cols, int64_t n,
                         double *out, double *sabs, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t t = 0; t < n; ++t) {
        double c, s;
        dot_one(K, A, lda, a_col_major, B, ldb, b_col_major, rows[t], cols[t], &c, &s);
        out[t] = c;
        if (sabs) sabs[t] = s;
    }
}
