/*
 * CPU oracle for Q4_0 dequantisation and MUL_MAT -- TEST INFRASTRUCTURE ONLY.
 * See q4_0_oracle.h for the definitions followed and their sources.
 * Plain scalar C; compile without fast-math or FMA contraction.
 */
#include "q4_0_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32            /* weights per block */
#define BLOCK_BYTES 18   /* 2 bytes of d, 16 bytes of qs */

size_t oracle_q4_0_nbytes(int64_t M, int64_t K)
{
    return (size_t)M * (size_t)(K / QK) * BLOCK_BYTES;
}

/*
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   e == 0:       (-1)^s * 2^-14 * (f / 1024)         (zero, subnormal)
 *   1 <= e <= 30: (-1)^s * 2^(e-15) * (1 + f / 1024)
 *   e == 31:      f == 0 ? (-1)^s * inf : NaN
 */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);                 /* f/1024 * 2^-14 */
    } else if (e == 31) {
        mag = (f == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(1024 + f), e - 25);     /* (1+f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

void oracle_half_to_float_n(const uint16_t *h, size_t n, float *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = (float)oracle_half_to_double(h[i]);
}

/* One row of K/32 blocks -> K fp32 weights, w = d * (q - 8). */
static void dequant_row(const uint8_t *row, int64_t K, float *w)
{
    int64_t nb = K / QK;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = row + b * BLOCK_BYTES;
        uint16_t d_bits = (uint16_t)(blk[0] | (blk[1] << 8));   /* little-endian */
        float d = (float)oracle_half_to_double(d_bits);
        const uint8_t *qs = blk + 2;
        for (int j = 0; j < 16; ++j) {
            int q_lo = qs[j] & 0x0F;        /* element j      */
            int q_hi = qs[j] >> 4;          /* element j + 16 */
            w[b * QK + j] = d * (float)(q_lo - 8);
            w[b * QK + j + 16] = d * (float)(q_hi - 8);
        }
    }
}

void oracle_dequant_q4_0(const uint8_t *W, int64_t M, int64_t K, float *out)
{
    size_t row_bytes = (size_t)(K / QK) * BLOCK_BYTES;
    for (int64_t m = 0; m < M; ++m)
        dequant_row(W + (size_t)m * row_bytes, K, out + (size_t)m * (size_t)K);
}

void oracle_mul_mat_q4_0(const uint8_t *W, int64_t M, int64_t K,
                         const float *X, int64_t N,
                         double *Y, double *S, int nthreads)
{
    size_t row_bytes = (size_t)(K / QK) * BLOCK_BYTES;
    if (nthreads < 1)
        nthreads = 1;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 4)
#endif
    for (int64_t m = 0; m < M; ++m) {
        float *w = (float *)malloc((size_t)(K > 0 ? K : 1) * sizeof(float));
        dequant_row(W + (size_t)m * row_bytes, K, w);
        for (int64_t n = 0; n < N; ++n) {
            const float *x = X + (size_t)n * (size_t)K;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)w[k] * (double)x[k];   /* exact in fp64 */
                acc += p;
                acc_abs += fabs(p);
            }
            Y[(size_t)n * (size_t)M + (size_t)m] = acc;
            S[(size_t)n * (size_t)M + (size_t)m] = acc_abs;
        }
        free(w);
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
