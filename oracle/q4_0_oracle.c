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

/*
 * binary32 -> binary16, round to nearest, ties to even, from the IEEE-754
 * fields: finite values too large for binary16 become infinity, values below
 * its smallest subnormal round to (signed) zero or to the smallest subnormal,
 * NaN stays NaN (quiet, sign kept).
 */
uint16_t oracle_float_to_half(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    int e = (int)((x >> 23) & 0xFF);          /* biased exponent of binary32 */
    uint32_t m = x & 0x7FFFFFu;               /* 23 fraction bits */
    if (e == 255)                              /* inf or NaN */
        return (uint16_t)(sign | 0x7C00u | (m ? 0x200u : 0u));
    /* value = 1.m * 2^(e-127) for e > 0, 0.m * 2^-126 for e == 0 */
    int he = e - 127 + 15;                     /* binary16 biased exponent if normal */
    if (he >= 31)
        return (uint16_t)(sign | 0x7C00u);     /* overflow */
    uint32_t mant;                             /* significand with the implicit bit, 24 bits */
    int shift;                                 /* right shift down to the 10-bit binary16 fraction */
    if (he >= 1) {
        mant = m | 0x800000u;
        shift = 13;
    } else {
        if (e == 0)
            return sign;                       /* binary32 subnormals are far below binary16's range */
        mant = m | 0x800000u;
        shift = 14 - he;                       /* binary16 subnormal: fraction = value / 2^-24 */
        if (shift > 24)
            return sign;                       /* rounds to zero: below half the smallest subnormal */
        he = 0;
    }
    uint32_t kept = mant >> shift;
    uint32_t rest = mant & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (kept & 1u)))
        kept += 1u;                            /* may carry into the exponent: still correct */
    if (he >= 1)
        return (uint16_t)(sign | (uint16_t)((((uint32_t)he << 10) + (kept - 0x400u))));
    return (uint16_t)(sign | (uint16_t)kept);  /* kept == 0x400 means the smallest normal */
}

/*
 * Quantise one block of 32 weights to Q4_0, following the block-quantisation
 * formula q(w) = clip(round(w / s) + z, q_min, q_max), w_hat = s * (q - z)
 * ("Architecture and module overview", weight-loading section) with z = 8,
 * q in [0, 15].  The pages leave the choice of s open; the reading used here:
 *   m = the weight of largest magnitude, sign kept (the first on ties),
 *   s = m / -8 rounded to binary16 (the stored d), so that m maps to q = 0,
 *   q = clip(rint(w / d) + 8, 0, 15) with the quotient taken in fp32 and the
 *   rounding to nearest even; an all-zero block stores d = +0 and q = 8 for
 *   all, and a quotient that is NaN also gives 8.
 */
static void quantize_block(const float *w, uint8_t *blk)
{
    float amax = 0.0f, m = 0.0f;
    for (int j = 0; j < QK; ++j) {
        float a = fabsf(w[j]);
        if (a > amax) {
            amax = a;
            m = w[j];
        }
    }
    uint16_t d_bits = amax > 0.0f ? oracle_float_to_half(m / -8.0f) : 0;   /* all-zero block: d = +0 */
    float d = (float)oracle_half_to_double(d_bits);
    int q[QK];
    for (int j = 0; j < QK; ++j) {
        if (d == 0.0f) {
            q[j] = 8;
            continue;
        }
        float t = rintf(w[j] / d) + 8.0f;
        if (t != t)
            q[j] = 8;
        else if (t < 0.0f)
            q[j] = 0;
        else if (t > 15.0f)
            q[j] = 15;
        else
            q[j] = (int)t;
    }
    blk[0] = (uint8_t)(d_bits & 0xFF);         /* little-endian binary16 */
    blk[1] = (uint8_t)(d_bits >> 8);
    for (int j = 0; j < 16; ++j)               /* low nibble: element j, high nibble: element j + 16 */
        blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

void oracle_quantize_q4_0(const float *W, int64_t M, int64_t K, uint8_t *out)
{
    int64_t nb = K / QK;
    for (int64_t r = 0; r < M; ++r)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block(W + r * K + b * QK, out + (r * nb + b) * BLOCK_BYTES);
}

/*
 * MUL_MAT_ID (expert-routed MUL_MAT; "GGUF loading, mmap and tensor
 * placement", step six, the MUL_MAT_ID probe: w ne = [K, M, n_expert], b ne =
 * [K, n_ids, tokens], ids ne = [n_ids, tokens]):
 *   Y[t][s][m] = sum_k w_e[m][k] * X[t][s][k],  e = ids[t][s]
 * W holds n_expert matrices of M rows one after the other; X is [T][S][K];
 * ids is [T][S]; Y and the tolerance scale S_abs are [T][S][M] (fp64, k
 * ascending, as in oracle_mul_mat_q4_0).  An id outside [0, n_expert) leaves
 * its Y and S_abs rows NaN.
 */
void oracle_mul_mat_id_q4_0(const uint8_t *W, int64_t n_expert, int64_t M, int64_t K,
                            const float *X, int64_t S, const int32_t *ids, int64_t T,
                            double *Y, double *S_abs, int nthreads)
{
    size_t expert_bytes = (size_t)M * (size_t)(K / QK) * BLOCK_BYTES;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t s = 0; s < S; ++s) {
            int32_t e = ids[t * S + s];
            double *y = Y + (size_t)(t * S + s) * (size_t)M;
            double *sa = S_abs + (size_t)(t * S + s) * (size_t)M;
            if (e < 0 || e >= n_expert) {
                for (int64_t m = 0; m < M; ++m)
                    y[m] = sa[m] = NAN;
                continue;
            }
            oracle_mul_mat_q4_0(W + (size_t)e * expert_bytes, M, K, X + (size_t)(t * S + s) * (size_t)K, 1,
                                y, sa, nthreads);
        }
}

/* A little-endian binary16 field as fp32 (exact). */
static float le_half_at(const uint8_t *p)
{
    return (float)oracle_half_to_double((uint16_t)(p[0] | (p[1] << 8)));
}

/*
 * The other legacy formats ("Architecture and module overview", the
 * quantisation-format section: 32 weights per block sharing one scale; Q4_1
 * additionally stores a min offset; Q8_0 is the 8-bit member).  The pages do
 * not print their structs; the readings (stated in the header) are:
 *   Q4_1: fp16 d, fp16 m, uint8_t qs[16]  (20 bytes); w = d*q + m, q = 0..15,
 *         low nibble of qs[j] = element j, high nibble = element j+16.
 *   Q8_0: fp16 d, int8_t qs[32]           (34 bytes); w = d*q, q = -128..127,
 *         qs[j] = element j.
 * Both fp16 fields are little-endian.  In fp32: d*q is exact (at most 11 x 8
 * significant bits); Q4_1 then adds m with one rounding.
 */
static int type_block_bytes(int type)
{
    switch (type) {
    case ORACLE_TYPE_Q4_0: return 18;
    case ORACLE_TYPE_Q4_1: return 20;
    case ORACLE_TYPE_Q8_0: return 34;
    case ORACLE_TYPE_Q4_K: return 144;
    case ORACLE_TYPE_Q5_0: return 22;
    case ORACLE_TYPE_Q5_1: return 24;
    default: return 0;
    }
}

/* Weights per block: 32 for the legacy formats, 256 for the k-quant. */
static int type_block_weights(int type)
{
    return type == ORACLE_TYPE_Q4_K ? 256 : QK;
}

size_t oracle_type_nbytes(int type, int64_t M, int64_t K)
{
    int64_t bw = type_block_weights(type);
    if (K % bw)
        return 0;
    return (size_t)M * (size_t)(K / bw) * (size_t)type_block_bytes(type);
}

/*
 * Q4_K's sixteen 6-bit fields (the reading in the header): sc[j] and m[j] of
 * sub-blocks j = 0..7 from the 12 bytes b[] that follow d and dmin.
 */
static void q4_k_fields(const uint8_t *b, int sc[8], int m[8])
{
    for (int j = 0; j < 4; ++j) {
        sc[j] = b[j] & 0x3F;
        m[j] = b[4 + j] & 0x3F;
        sc[4 + j] = (b[8 + j] & 0x0F) | ((b[j] >> 6) << 4);
        m[4 + j] = (b[8 + j] >> 4) | ((b[4 + j] >> 6) << 4);
    }
}

/*
 * One Q5_0 / Q5_1 block -> 32 fp32 weights (the reading in the header): the
 * 5-bit code of element e is its nibble plus 16 times bit e of qh.
 */
static void dequant_q5_block(int type, const uint8_t *blk, float *w)
{
    float d = le_half_at(blk);
    int off = type == ORACLE_TYPE_Q5_1 ? 4 : 2;             /* qh follows d (and m) */
    uint32_t qh = (uint32_t)blk[off] | ((uint32_t)blk[off + 1] << 8) |
                  ((uint32_t)blk[off + 2] << 16) | ((uint32_t)blk[off + 3] << 24);
    const uint8_t *qs = blk + off + 4;
    for (int e = 0; e < QK; ++e) {
        int nib = e < 16 ? (qs[e] & 0x0F) : (qs[e - 16] >> 4);
        int q = nib | (int)(((qh >> e) & 1u) << 4);
        if (type == ORACLE_TYPE_Q5_0) {
            w[e] = d * (float)(q - 16);
        } else {
            float m = le_half_at(blk + 2);
            float dq = d * (float)q;
            w[e] = dq + m;
        }
    }
}

/* One Q4_K super-block -> 256 fp32 weights, w = d*sc_j*q - dmin*m_j. */
static void dequant_q4_k_block(const uint8_t *blk, float *w)
{
    float d = le_half_at(blk);
    float dmin = le_half_at(blk + 2);
    int sc[8], m[8];
    q4_k_fields(blk + 4, sc, m);
    const uint8_t *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        int jl = 2 * c, jh = 2 * c + 1;                 /* sub-blocks of the low and high nibbles */
        float dl = d * (float)sc[jl], ml = dmin * (float)m[jl];
        float dh = d * (float)sc[jh], mh = dmin * (float)m[jh];
        for (int l = 0; l < 32; ++l) {
            int q_lo = qs[32 * c + l] & 0x0F;
            int q_hi = qs[32 * c + l] >> 4;
            w[64 * c + l] = dl * (float)q_lo - ml;
            w[64 * c + 32 + l] = dh * (float)q_hi - mh;
        }
    }
}

static float le_half(const uint8_t *p)
{
    return le_half_at(p);
}

static void dequant_row_typed(int type, const uint8_t *row, int64_t K, float *w)
{
    int64_t nb = K / QK;
    int bb = type_block_bytes(type);
    if (type == ORACLE_TYPE_Q4_0) {
        dequant_row(row, K, w);
        return;
    }
    if (type == ORACLE_TYPE_Q4_K) {
        for (int64_t b = 0; b < K / 256; ++b)
            dequant_q4_k_block(row + b * bb, w + b * 256);
        return;
    }
    if (type == ORACLE_TYPE_Q5_0 || type == ORACLE_TYPE_Q5_1) {
        for (int64_t b = 0; b < nb; ++b)
            dequant_q5_block(type, row + b * bb, w + b * QK);
        return;
    }
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = row + b * bb;
        float *wb = w + b * QK;
        float d = le_half(blk);
        if (type == ORACLE_TYPE_Q4_1) {
            float m = le_half(blk + 2);
            const uint8_t *qs = blk + 4;
            for (int j = 0; j < 16; ++j) {
                float lo = d * (float)(qs[j] & 0x0F);
                float hi = d * (float)(qs[j] >> 4);
                wb[j] = lo + m;
                wb[j + 16] = hi + m;
            }
        } else {  /* Q8_0 */
            const uint8_t *qs = blk + 2;
            for (int j = 0; j < QK; ++j) {
                int q = qs[j] < 128 ? (int)qs[j] : (int)qs[j] - 256;   /* two's complement */
                wb[j] = d * (float)q;
            }
        }
    }
}

void oracle_dequant_typed(int type, const uint8_t *W, int64_t M, int64_t K, float *out)
{
    if (K % type_block_weights(type))
        return;
    size_t row_bytes = (size_t)(K / type_block_weights(type)) * (size_t)type_block_bytes(type);
    for (int64_t m = 0; m < M; ++m)
        dequant_row_typed(type, W + (size_t)m * row_bytes, K, out + (size_t)m * (size_t)K);
}

void oracle_validate_typed(int type, const uint8_t *W, int64_t M, int64_t K, uint64_t *count, uint64_t *first)
{
    int bb = type_block_bytes(type);
    *count = 0;
    *first = UINT64_MAX;
    if (K % type_block_weights(type))
        return;
    uint64_t nblocks = (uint64_t)M * (uint64_t)(K / type_block_weights(type));
    for (uint64_t b = 0; b < nblocks; ++b) {
        const uint8_t *blk = W + b * (uint64_t)bb;
        int bad = !isfinite(oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8))));
        if (type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q4_K || type == ORACLE_TYPE_Q5_1)   /* m, or dmin */
            bad |= !isfinite(oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8))));
        if (bad) {
            if (*count == 0)
                *first = b;
            ++*count;
        }
    }
}

void oracle_mul_mat_typed(int type, const uint8_t *W, int64_t M, int64_t K, const float *X, int64_t N,
                          double *Y, double *S, int nthreads)
{
    if (K % type_block_weights(type))
        return;
    size_t row_bytes = (size_t)(K / type_block_weights(type)) * (size_t)type_block_bytes(type);
    if (nthreads < 1)
        nthreads = 1;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 4)
#endif
    for (int64_t m = 0; m < M; ++m) {
        float *w = (float *)malloc((size_t)(K > 0 ? K : 1) * sizeof(float));
        dequant_row_typed(type, W + (size_t)m * row_bytes, K, w);
        for (int64_t n = 0; n < N; ++n) {
            const float *x = X + (size_t)n * (size_t)K;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)w[k] * (double)x[k];
                acc += p;
                acc_abs += fabs(p);
            }
            Y[(size_t)n * (size_t)M + (size_t)m] = acc;
            S[(size_t)n * (size_t)M + (size_t)m] = acc_abs;
        }
        free(w);
    }
}
