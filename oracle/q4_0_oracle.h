/*
 * CPU oracle for Q4_0 dequantisation and MUL_MAT -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code.  It shares nothing with the CUDA library: no headers, no
 * helpers, no tables.
 *
 * What it computes, and where that is defined:
 *  - block_q4_0 is an fp16 scale d followed by uint8_t qs[16] holding 32
 *    four-bit codes, two per byte ("Binding GGUF weights to the compute
 *    graph", section 2.3, the block_q4_0 struct).  A block is 18 bytes; a row of K weights is K/32
 *    blocks, so a quantised tensor takes M*K/32*18 bytes, not M*K*bits/8
 *    (same section, the ggml_nbytes note).
 *  - Each code q maps back to w = s*(q - z) ("Architecture and module
 *    overview", weight-loading section, the block-quantisation formula); for
 *    Q4_0, s = d and z = 8, the low nibble of qs[j] is element j and the high
 *    nibble is element j+16 (the fixed Q4_0 convention of the method).
 *  - MUL_MAT takes the quantised weight W with ne = [K, M] and activations b
 *    with ne = [K, N], and dequantises inside the operator ("GGUF loading,
 *    mmap and tensor placement", step six, the MUL_MAT probe; section 2.3
 *    above).  The result Y has ne = [M, N]: Y[n][m] = sum_k w[m][k]*x[n][k].
 *
 * Precision: the scale is decoded exactly from its IEEE-754 binary16 fields;
 * w = d*(q-8) is formed in fp32 (exact: 11 significant bits times at most
 * 4 bits); products and sums of MUL_MAT are taken in fp64 in plain k order.
 *
 *  - The quantiser follows the block-quantisation formula q(w) = clip(
 *    round(w/s) + z, q_min, q_max) of the same section; how s is chosen is
 *    not fixed by the pages (the reading is stated at quantize_block).
 *
 * Every function here is pinned by the CPU tests (hand-derived block
 * fixtures, all 65536 binary16 patterns against numpy, one-hot columns,
 * exact special cases, brute force against a dense fp64 matmul; for the
 * quantiser: binary16 rounding against numpy, exact round trips, the nearest
 * level by brute force and the error model).
 */
#ifndef Q4_0_ORACLE_H
#define Q4_0_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of a Q4_0 matrix of M rows and K columns (K a multiple of 32). */
size_t oracle_q4_0_nbytes(int64_t M, int64_t K);

/* Exact value of an IEEE-754 binary16 bit pattern (subnormals, inf, NaN). */
double oracle_half_to_double(uint16_t h);

/* n patterns -> n fp32 values (binary16 values are all exact in fp32). */
void oracle_half_to_float_n(const uint16_t *h, size_t n, float *out);

/* Dequantise M rows of K/32 blocks each into out[M][K] (fp32). */
void oracle_dequant_q4_0(const uint8_t *W, int64_t M, int64_t K, float *out);

/*
 * MUL_MAT against Q4_0 weights:
 *   Y[n][m] = sum_k w[m][k] * X[n][k]       (fp64, k ascending)
 *   S[n][m] = sum_k |w[m][k] * X[n][k]|     (fp64; the tolerance scale)
 * W: M rows of K/32 blocks; X: [N][K] fp32; Y, S: [N][M] fp64.
 * nthreads > 1 splits the rows m over OpenMP threads; each output is still
 * one sequential sum, so the results do not depend on nthreads.
 */
void oracle_mul_mat_q4_0(const uint8_t *W, int64_t M, int64_t K,
                         const float *X, int64_t N,
                         double *Y, double *S, int nthreads);

/* binary32 -> binary16 bit pattern, round to nearest even (IEEE-754). */
uint16_t oracle_float_to_half(float f);

/*
 * fp32 weights W[M][K] -> M rows of K/32 Q4_0 blocks (the quantiser, the step
 * before MUL_MAT): per block, d = binary16(m / -8) with m the weight of largest
 * magnitude, q = clip(rint(w / d) + 8, 0, 15) in fp32 (see the .c file).
 */
void oracle_quantize_q4_0(const float *W, int64_t M, int64_t K, uint8_t *out);

/*
 * MUL_MAT_ID: Y[t][s][m] = sum_k w_e[m][k] * X[t][s][k] with e = ids[t][s]
 * (expert-routed; W = n_expert matrices of M rows each, X [T][S][K], ids
 * [T][S], Y and S_abs [T][S][M] in fp64).  Ids outside [0, n_expert) give
 * NaN rows.
 */
void oracle_mul_mat_id_q4_0(const uint8_t *W, int64_t n_expert, int64_t M, int64_t K,
                            const float *X, int64_t S, const int32_t *ids, int64_t T,
                            double *Y, double *S_abs, int nthreads);

/*
 * The other legacy formats of the quantisation-format section of
 * "Architecture and module overview" (32 weights per block, one scale; Q4_1
 * also a min offset; Q8_0 eight bits).  The pages do not print their structs;
 * the reading: Q4_1 = fp16 d, fp16 m, qs[16] (20 bytes), w = d*q + m with q =
 * 0..15 in the Q4_0 nibble order; Q8_0 = fp16 d, int8 qs[32] (34 bytes), w =
 * d*q.  ORACLE_TYPE_Q4_0 is the Q4_0 functions above.
 */
enum { ORACLE_TYPE_Q4_0 = 0, ORACLE_TYPE_Q4_1 = 1, ORACLE_TYPE_Q8_0 = 2, ORACLE_TYPE_Q4_K = 3,
       ORACLE_TYPE_Q5_0 = 4, ORACLE_TYPE_Q5_1 = 5 };
/*
 * Q5_0 and Q5_1, the 5-bit legacy formats named beside Q4_0 / Q4_1 in the
 * quantisation-format section (32 weights per block, one scale; the _1 form
 * also a min).  The pages print neither struct.  The reading, the layout
 * GGUF files carry:
 *   Q5_0: fp16 d, uint8_t qh[4], uint8_t qs[16]            (22 bytes), w = d*(q - 16)
 *   Q5_1: fp16 d, fp16 m, uint8_t qh[4], uint8_t qs[16]    (24 bytes), w = d*q + m
 * with the 5-bit code q of element e (0..31) = its nibble (low nibble of
 * qs[e] for e < 16, high nibble of qs[e-16] for e >= 16, as in Q4_0) plus 16
 * times bit e of the little-endian 32-bit word qh.  In fp32, d*(q-16) is exact
 * (11 x 5 significant bits); Q5_1's d*q is exact and m is added with one
 * rounding.
 */
/*
 * Q4_K, the 4-bit k-quant ("Architecture and module overview", the
 * quantisation-format section and the error-model paragraph of the
 * weight-loading section: k-quants group 256 weights per block and store the
 * block's scales and mins hierarchically inside it, an upper level in 6 bits
 * and a lower level in 4; "GGUF loading, mmap and tensor placement": a Q4_K
 * tensor takes ne[0]/256 x block-size bytes).  The pages print no struct.
 * The reading: the 6-bit level is a scale and a min per sub-block of 32
 * weights, the 4-bit level is the weight codes, and the bytes are laid out as
 * GGUF files carry them (the pages stress that the file's block layout is the
 * memory layout the kernels consume), a 144-byte super-block of 256 weights:
 *   bytes 0-1    fp16 d      (scale of the sub-block scales)
 *   bytes 2-3    fp16 dmin   (scale of the sub-block mins)
 *   bytes 4-15   sixteen 6-bit fields: sc_j and m_j of the 8 sub-blocks of
 *                32 weights (byte b = bytes[4 + b]):
 *                  b 0-3:  bits 0-5 = sc_b,     bits 6-7 = bits 4-5 of sc_{b+4}
 *                  b 4-7:  bits 0-5 = m_{b-4},  bits 6-7 = bits 4-5 of m_b
 *                  b 8-11: bits 0-3 = bits 0-3 of sc_{b-4}, bits 4-7 = bits 0-3 of m_{b-4}
 *   bytes 16-143 qs[128]: weight 64c + l (c = 0..3, l = 0..31) is the low
 *                nibble of qs[32c + l] (sub-block 2c); weight 64c + 32 + l is
 *                its high nibble (sub-block 2c + 1).
 * Weight i of sub-block j with code q: w = d*sc_j*q - dmin*m_j.  In fp32
 * d*sc_j (at most 17 significant bits) times q (4 bits) and dmin*m_j are
 * exact, so the fp32 weight is that value rounded once.  K must be a multiple
 * of 256 (the typed functions return 0 bytes / do nothing otherwise), and the
 * flat block index of validation counts super-blocks (row * K/256 + block).
 */
size_t oracle_type_nbytes(int type, int64_t M, int64_t K);
void oracle_dequant_typed(int type, const uint8_t *W, int64_t M, int64_t K, float *out);
void oracle_mul_mat_typed(int type, const uint8_t *W, int64_t M, int64_t K, const float *X, int64_t N,
                          double *Y, double *S, int nthreads);

/*
 * Row-data validation ("GGUF loading, mmap and tensor placement", the section
 * on --check-tensors and parallel validation: ggml_validate_row_data checks
 * each row's scale factors and integers; the reading: a block's fp16 scale
 * fields must be finite, and every 4-, 6- or 8-bit field is a valid integer).  Over the M x K weights in block format `type`: *count = the
 * number of blocks with a NaN or infinite scale (d; for Q4_1 and Q5_1 also m; for Q4_K also dmin),
 * *first = the smallest flat block index (row * K/32 + block; row * K/256 +
 * super-block for Q4_K) among them, or
 * UINT64_MAX when there is none.  A scale is tested by decoding it with
 * oracle_half_to_double and asking isfinite.
 */
void oracle_validate_typed(int type, const uint8_t *W, int64_t M, int64_t K, uint64_t *count, uint64_t *first);

/* Number of threads OpenMP would use by default (1 without OpenMP). */
int oracle_max_threads(void);

#ifdef __cplusplus
}
#endif

#endif
