/*
 * oracle_conv.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of the 2-D convolution the
 * GPU path computes as an implicit GEMM.  Only tests/ may load it; nothing
 * here is shared with the library under dense_tensor_core_bf16_gb300/.
 *
 * What it follows
 *   - lesson "The Tensor Core", the paragraph on what work the Tensor Cores
 *     speed up: convolutions reach them through im2col / implicit GEMM, i.e.
 *     the convolution is a matrix product whose rows are output pixels and
 *     whose inner dimension runs over the filter taps and input channels.
 * Definition (forward convolution as used by neural networks, i.e. a
 * cross-correlation; NHWC activations, KRSC filters):
 *
 *   y[n][p][q][k] = sum_{r<R} sum_{s<S} sum_{c<C}
 *                   x[n][p*sh - ph + r*dh][q*sw - pw + s*dw][c] * w[k][r][s][c]
 *
 * with x taken as zero outside 0 <= h < H, 0 <= w < W (the padding), and
 * P = (H + 2 ph - dh (R-1) - 1) / sh + 1, Q likewise (integer division).
 * Every bf16 input is widened exactly to binary64; products are exact; the
 * sum is taken in increasing r, then s, then c, in binary64.  Sabs[...] is the
 * same sum of |x w|, for the error bound of an fp32 accumulation.
 *
 * Pins (tests/test_oracle_pins.py): a 1 x 1 convolution against the pinned
 * GEMM oracle, exact rational brute force on tiny shapes with stride, padding
 * and dilation, the tap count under padding with all-ones inputs, and the
 * identity filter.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double oracle_bf16_to_f64(uint16_t h);

void oracle_conv2d_fprop(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                         int64_t pad_h, int64_t pad_w, int64_t str_h, int64_t str_w, int64_t dil_h, int64_t dil_w,
                         int64_t P, int64_t Q, const uint16_t *x, const uint16_t *w, double *y, double *sabs,
                         int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const int64_t rows = N * P;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t np = 0; np < rows; ++np) {
        const int64_t n = np / P;
        const int64_t p = np % P;
        for (int64_t q = 0; q < Q; ++q) {
            for (int64_t k = 0; k < K; ++k) {
                double acc = 0.0, sa = 0.0;
                for (int64_t r = 0; r < R; ++r) {
                    const int64_t h = p * str_h - pad_h + r * dil_h;
                    if (h < 0 || h >= H) continue;
                    for (int64_t s = 0; s < S; ++s) {
                        const int64_t ww = q * str_w - pad_w + s * dil_w;
                        if (ww < 0 || ww >= W) continue;
                        const uint16_t *xp = x + ((n * H + h) * W + ww) * C;
                        const uint16_t *wp = w + ((k * R + r) * S + s) * C;
                        for (int64_t c = 0; c < C; ++c) {
                            const double prod = oracle_bf16_to_f64(xp[c]) * oracle_bf16_to_f64(wp[c]);
                            acc += prod;
                            sa += fabs(prod);
                        }
                    }
                }
                const int64_t o = ((n * P + p) * Q + q) * K + k;
                y[o] = acc;
                if (sabs) sabs[o] = sa;
            }
        }
    }
}
