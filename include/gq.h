/*
 * gq -- MUL_MAT against block-quantised Q4_0 weights on NVIDIA GB300 (sm_103a).
 *
 * The operation ("GGUF loading, mmap and tensor placement", step six, the
 * MUL_MAT probe; "ggml compute graph and memory allocator", the ggml_tensor
 * section on ne/nb):
 *   W  quantised weight, ggml ne = [K, M]: M rows, each K/32 block_q4_0.
 *   X  activations, F32, ne = [K, N]: N rows of K floats (K innermost).
 *   Y  result, F32, ne = [M, N]: Y[n][m] = sum_k w[m][k] * X[n][k].
 * block_q4_0 ("Binding GGUF weights to the compute graph", section 2.3): an
 * IEEE binary16 scale d (little-endian) followed by uint8_t qs[16]; 18 bytes
 * per 32 weights.  The low nibble of qs[j] is code q of element j, the high
 * nibble that of element j+16, and w = d*(q - 8) ("Architecture and module
 * overview", weight-loading section: w = s*(q - z)).  Dequantisation happens
 * inside the operator (section 2.3 above); W is never expanded in memory.
 *
 * Conventions for every entry point:
 *  - Pointers to tensors are DEVICE pointers owned by the caller; the library
 *    never frees or retains them.  Rows are contiguous: W row stride is
 *    K/32*18 bytes, X row stride K floats, Y row stride M floats.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *    enqueued asynchronously on it; the call returns after enqueueing.
 *  - The return value reports argument errors and launch errors found while
 *    enqueueing.  A device-side fault detected later (a bounded wait inside a
 *    kernel that gave up) is reported by gq_sync_status().
 *  - M or N equal to 0 is a no-op that returns GQ_OK; K equal to 0 (an empty
 *    sum) writes zeros to Y.
 *  - Non-finite scales or activations propagate as IEEE arithmetic does; they
 *    are not validated on the MUL_MAT path (gq_validate checks the scales).
 *  - No C++ exception crosses this interface.  Calls on different streams may
 *    run concurrently, and host threads may call in parallel, each on its own
 *    current device: the library sets its kernels' launch attributes once per
 *    (kernel, device) under a lock.  gq_last_error() is per thread.
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQ_OK = 0,
  GQ_ERR_NULL = -1,            /* a required pointer is NULL */
  GQ_ERR_SHAPE = -2,           /* negative size, K % 32 != 0, or a size overflows */
  GQ_ERR_ALIGN = -3,           /* pointer alignment the entry point requires is missing */
  GQ_ERR_CUDA = -4,            /* a CUDA runtime call or kernel launch failed */
  GQ_ERR_ALLOC = -5,           /* stream-ordered scratch allocation failed */
  GQ_ERR_DEVICE_TIMEOUT = -6,  /* a kernel's bounded wait gave up (see gq_sync_status) */
  GQ_ERR_UNSUPPORTED = -7,     /* current device is not compute capability 10.3 */
  GQ_ERR_BAD_INDEX = -8        /* an expert id outside [0, n_expert) reached gq_mul_mat_id_q4_0
                                  (reported by gq_sync_status) */
} gq_status;

/* Block formats of the typed entry points ("Architecture and module
 * overview", quantisation-format section: the legacy formats, 32 weights per
 * block with one scale; Q4_1 also stores a min offset; Q8_0 has 8-bit codes;
 * the k-quants, 256 weights per block with scales and mins stored
 * hierarchically inside it, an upper level in 6 bits and a lower one in 4).
 * The pages print only the Q4_0 struct; the layouts taken for the others:
 *   GQ_TYPE_Q4_0  fp16 d, uint8_t qs[16]          18 bytes  w = d*(q - 8)
 *   GQ_TYPE_Q4_1  fp16 d, fp16 m, uint8_t qs[16]  20 bytes  w = d*q + m
 *   GQ_TYPE_Q8_0  fp16 d, int8_t qs[32]           34 bytes  w = d*q
 *   GQ_TYPE_Q5_0  fp16 d, uint8_t qh[4], uint8_t qs[16]          22 bytes  w = d*(q - 16)
 *   GQ_TYPE_Q5_1  fp16 d, fp16 m, uint8_t qh[4], uint8_t qs[16]  24 bytes  w = d*q + m
 *   GQ_TYPE_Q4_K  fp16 d, fp16 dmin, uint8_t scales[12], uint8_t qs[128]
 *                 144 bytes per 256 weights (the GGUF super-block)
 *                 w = d*sc_j*q - dmin*m_j for sub-block j = 0..7 of 32 weights
 * (fp16 little-endian; legacy 4-bit codes: low nibble of qs[j] = element j,
 * high nibble = element j+16; Q8_0: qs[j] = element j; Q5_0 / Q5_1: the 5-bit
 * q of element e is its nibble in the Q4_0 order plus 16 times bit e of qh
 * read as a little-endian 32-bit word.  Q4_K: weight 64c + l
 * (l < 32) is the low nibble of qs[32c + l] in sub-block 2c, weight 64c+32+l
 * its high nibble in sub-block 2c+1; the 6-bit sc_j, m_j: for j < 4 bits 0-5
 * of scales[j] and scales[j+4]; for j >= 4 bits 0-3 from the low and high
 * nibble of scales[j+4] and bits 4-5 from the top two bits of scales[j-4]
 * and scales[j].)  Rows of Q4_K need K % 256 == 0. */
typedef enum {
  GQ_TYPE_Q4_0 = 0,
  GQ_TYPE_Q4_1 = 1,
  GQ_TYPE_Q8_0 = 2,
  GQ_TYPE_Q4_K = 3,
  GQ_TYPE_Q5_0 = 4,
  GQ_TYPE_Q5_1 = 5
} gq_type;

/* Bytes of a Q4_0 matrix of M rows and K columns: M*(K/32)*18
 * ("Binding GGUF weights to the compute graph", section 2.3, ggml_nbytes note).
 * Returns 0 for K % 32 != 0 or negative sizes. */
size_t gq_q4_0_nbytes(int64_t M, int64_t K);

/* Dequantise W (M x K, Q4_0) into out[M][K] fp32.  Bit-exact: every output is
 * the fp32 value d*(q-8), including the sign of zero.  No alignment needed
 * (16-byte aligned W and out take the vectorised kernel). */
gq_status gq_dequant_q4_0(const void *W, int64_t M, int64_t K, float *out, void *stream);

/* Quantise fp32 weights W[M][K] into M rows of K/32 Q4_0 blocks (18 bytes
 * each) at `out` (M*K/32*18 bytes): the step before MUL_MAT.  Follows the
 * block-quantisation formula q(w) = clip(round(w/s) + z, q_min, q_max),
 * w_hat = s*(q - z) ("Architecture and module overview", weight-loading
 * section) with z = 8, q in [0, 15].  The pages do not fix s; this library
 * takes, per block, m = the weight of largest magnitude (sign kept, the first
 * on ties), d = binary16(m / -8) rounded to nearest even (so m gets code 0;
 * an all-zero block stores d = +0), and q = clip(rint(w / d) + 8, 0, 15) with
 * the quotient an IEEE fp32 division (q = 8 when d == 0 or the quotient is
 * NaN).  Every element that is not clipped is within d/2 of its weight.
 * Device pointers; W 4-byte aligned (16 bytes takes the vector path); errors:
 * K % 32 != 0 or negative sizes -> GQ_ERR_SHAPE, NULL -> GQ_ERR_NULL. */
gq_status gq_quantize_q4_0(const float *W, int64_t M, int64_t K, void *out, void *stream);

/* Bytes of an M x K matrix in block format `type`: M*(K/32)*block bytes
 * (Q4_K: M*(K/256)*144); 0 for K not a multiple of the block's weights,
 * negative sizes or an unknown type. */
size_t gq_type_nbytes(gq_type type, int64_t M, int64_t K);

/* Dequantise W (M x K in block format `type`) into out[M][K] fp32, bit-exact:
 * d*q is exact in fp32 and Q4_1 adds m with one rounding (round to nearest
 * even); Q4_K's d*sc_j*q and dmin*m_j are exact in fp32 and their difference
 * is rounded once.  GQ_TYPE_Q4_0 is gq_dequant_q4_0.  Any alignment (16-byte
 * aligned W and out take vector loads and stores); errors as gq_dequant_q4_0
 * (Q4_K: K % 256 != 0 is GQ_ERR_SHAPE), plus GQ_ERR_SHAPE for an unknown type. */
gq_status gq_dequant(gq_type type, const void *W, int64_t M, int64_t K, float *out, void *stream);

/* Row-data validation ("GGUF loading, mmap and tensor placement", the
 * section on --check-tensors: ggml_validate_row_data checks each row's scale
 * factors and integers): scan W (M x K in block format `type`, rows
 * contiguous) for blocks whose fp16 scale fields are NaN or infinite -- d in
 * every format, m in Q4_1, dmin in Q4_K; codes and 6-bit fields are always
 * valid.  result: device pointer to two uint64 values, written on `stream`:
 * result[0] = the number of such blocks, result[1] = the smallest flat block
 * index (row * K/32 + block; for Q4_K row * K/256 + super-block) among them,
 * or UINT64_MAX when there is none.  Asynchronous: read result
 * after the stream.  Any alignment of W; result 8-byte aligned.  M or K == 0:
 * result (0, UINT64_MAX).  Errors: GQ_ERR_SHAPE (negative size, K % 32 != 0,
 * unknown type, Q4_K with K % 256 != 0), GQ_ERR_NULL (result NULL, or W NULL with M*K > 0),
 * GQ_ERR_ALIGN (result not 8-byte aligned). */
gq_status gq_validate(gq_type type, const void *W, int64_t M, int64_t K, uint64_t *result, void *stream);

/* gq_validate for Q4_0 weights. */
gq_status gq_validate_q4_0(const void *W, int64_t M, int64_t K, uint64_t *result, void *stream);

/* MUL_MAT with W in block format `type`: Y[N][M] = X[N][K] * W^T, fp32 in and
 * out.  GQ_TYPE_Q4_0 is gq_mul_mat_q4_0.  Q4_1, Q8_0 and Q4_K (whose K must be
 * a multiple of 256: GQ_ERR_SHAPE otherwise), with K % 256 == 0
 * and W, X, Y 16-byte aligned: N >= GQ_OPT_PREFILL_MIN_N converts X to bf16
 * and runs the tcgen05 kernel with this block format (N*K*2 bytes of
 * stream-ordered scratch, plus k-split scratch as in gq_mul_mat_q4_0); a
 * smaller N below 16 streams W through the decode kernel on this block format
 * (fp16 x, exact integer codes, fp32 block scales and accumulation; Q4_K:
 * per 32-weight sub-block the scale d*sc_j and the min dmin*m_j in fp32; the
 * tensor-core path rounds each fp32 weight to bf16).  Other
 * shapes: a warp per weight row decodes the blocks to fp32 in registers
 * and accumulates in fp32 (any alignment, K % 32 == 0); GQ_OPT_FORCE_GENERIC
 * forces it.  M, N == 0 no-op, K == 0 zeros.  Accuracy as gq_mul_mat_q4_0. */
gq_status gq_mul_mat(gq_type type, const void *W, int64_t M, int64_t K, const float *X, int64_t N, float *Y,
                     void *stream);

/* Y[N][M] = X[N][K] * W^T with W in Q4_0, fp32 in and out (see header).
 * Dispatch by N: N < 16 streams W through the decode kernel (fp16 x; where a
 * token's largest |x| in a warp's chunk of K (256 to a few thousand elements)
 * reaches 2^15 or stays below 2^-10 that chunk is staged times the exact power
 * of two that brings it into [2^14, 2^15), so that the token's largest values
 * keep fp16's 11 significant bits at any finite magnitude; exact integer
 * codes, fp32 block scales and accumulation); N >= 16 converts X to
 * bf16 once and runs the tcgen05 tensor-core kernel on bf16 tiles of the
 * dequantised W with fp32 accumulation (GQ_OPT_PREFILL_MIN_N moves the
 * threshold).  Fast paths need K % 256 == 0 and W, X, Y 16-byte aligned; other
 * shapes take a slower generic kernel.  The tensor-core path allocates N*K*2
 * bytes of stream-ordered scratch for bf16 X, plus, when it splits tiles
 * along k (GQ_OPT_PREFILL_STREAMK), 128 KiB per split piece and 8 bytes per
 * split tile for partial sums, from a pool the library keeps per device; it
 * frees them on the same stream.  Accuracy: |y - y_ref| <= 1e-3*sum_k|w_k x_k|
 * + 1e-5 on the synthetic workloads (random-sign data). */
gq_status gq_mul_mat_q4_0(const void *W, int64_t M, int64_t K, const float *X, int64_t N, float *Y,
                          void *stream);

/* MUL_MAT_ID: the expert-routed MUL_MAT of mixture-of-experts layers
 * ("GGUF loading, mmap and tensor placement", step six, the MUL_MAT_ID probe:
 * w ne = [K, M, n_expert], b ne = [K, n_ids, T], ids ne = [n_ids, T] of I32).
 *   W    n_expert Q4_0 matrices of M rows, one after the other (expert e's row
 *        m is row e*M + m; n_expert*M*K/32*18 bytes).
 *   X    F32 [T][n_ids][K]: the activation row of each (token t, slot s).
 *   ids  I32 [T][n_ids], device memory: the expert of each (t, s).
 *   Y    F32 [T][n_ids][M]: Y[t][s][m] = sum_k w_e[m][k] * X[t][s][k],
 *        e = ids[t][s].
 * The pairs are sorted by expert on the device (a stable counting sort, no
 * host synchronisation), so each expert's weights stream once for all its
 * tokens: with fewer than 16 tokens per used expert on average the decode
 * kernel runs one group of tokens per expert, otherwise the gathered tokens
 * go to the tcgen05 tensor-core kernel as bf16 (GQ_OPT_MOE_PATH forces either).
 * Accuracy as gq_mul_mat_q4_0.  Scratch (stream-ordered, library pool): the
 * routing tables, about (2*n_expert + 4*T*n_ids) * 4 bytes, plus T*n_ids*K*2
 * bytes of bf16 rows on the tensor-core path.
 *  - An id outside [0, n_expert) sets that Y row to NaN and makes the next
 *    gq_sync_status() return GQ_ERR_BAD_INDEX; the other rows are computed.
 *  - Fast paths need K % 256 == 0, W, X, Y 16-byte aligned, ids 4-byte
 *    aligned, n_expert <= 16384 and n_expert*M < 2^31; other shapes take a
 *    slower generic kernel.
 *  - T or n_ids or M equal to 0 is a no-op; K == 0 writes zeros (NaN for bad
 *    ids).  n_expert must be >= 1 (GQ_ERR_SHAPE). */
gq_status gq_mul_mat_id_q4_0(const void *W, int64_t n_expert, int64_t M, int64_t K, const float *X,
                             int64_t n_ids, const int32_t *ids, int64_t T, float *Y, void *stream);

/* The repack of Q4_0 weights for the fast kernels (the GPU analogue of the
 * library's repacked layouts).  ggml rows may have a padded stride (nb[1],
 * "ggml compute graph and memory allocator", the ggml_tensor section) and K
 * need only be a multiple of 32; the TMA kernels want rows of a multiple of
 * 256 weights.  gq_prepare_q4_0 copies each row of W (row_stride bytes apart;
 * 0 = packed, K/32*18) into `out`, rows of ceil(K/256)*144 bytes, and fills
 * each row up with zero blocks (d = +0, every code 8).  The blocks are copied
 * unchanged: the prepared matrix holds the same weights.  out needs
 * gq_prepared_q4_0_nbytes(M, K) bytes, 16-byte aligned; W any alignment.
 * Errors: K % 32 != 0, negative sizes, row_stride shorter than a row or a
 * prepared row above 2^31 bytes -> GQ_ERR_SHAPE; NULL -> GQ_ERR_NULL; out
 * unaligned -> GQ_ERR_ALIGN. */
size_t gq_prepared_q4_0_nbytes(int64_t M, int64_t K);
gq_status gq_prepare_q4_0(const void *W, int64_t M, int64_t K, int64_t row_stride, void *out, void *stream);

/* MUL_MAT on prepared weights (gq_prepare_q4_0): the result of
 * gq_mul_mat_q4_0 on the original W, through the fast kernels for any K % 32
 * == 0 (the decode kernel below the tensor-core threshold, else X -> bf16 and
 * the tcgen05 kernel; the zero blocks meet zero x).  K < 256 always takes the
 * decode kernel, 64 tokens per launch: with so few terms the bf16 rounding of
 * the tensor-core path does not average below the tolerance.  Wp, X, Y
 * 16-byte aligned; scratch as gq_mul_mat_q4_0. */
gq_status gq_mul_mat_q4_0_prepared(const void *Wp, int64_t M, int64_t K, const float *X, int64_t N, float *Y,
                                   void *stream);

/* MUL_MAT with activations the caller already holds in bf16: X_bf16[N][K]
 * (raw bfloat16 bits).  Runs the tensor-core kernel for every N >= 1.  Its
 * only allocation is the stream-ordered partial-sum scratch of split tiles
 * (see gq_mul_mat_q4_0); if that allocation fails it runs one CTA per tile
 * instead.  Needs K % 256 == 0, W and X_bf16 16-byte aligned.  Honours
 * GQ_OPT_X_STATIC for X_bf16 (the call then streams W and runs its MMAs while
 * the kernels ahead of it finish). */
gq_status gq_mul_mat_q4_0_bf16x(const void *W, int64_t M, int64_t K, const uint16_t *X_bf16, int64_t N,
                                float *Y, void *stream);

/* Same result as the tensor-core path of gq_mul_mat_q4_0 (bf16 activations,
 * tensor-core kernel), for any N >= 1, but with no device allocation: the
 * bf16 copy of X goes to a fixed 12 MiB array inside the library instead of
 * cudaMallocAsync scratch, and the tensor-core kernel runs one CTA per tile
 * (no stream-K partial sums).  The pages have no counterpart; it exists for
 * callers that cannot let a library allocate device memory (memory pools that
 * own the whole device, fixed arenas, allocation-free hot loops).
 *  - Needs K % 256 == 0 and N*K <= 6291456 (GQ_ERR_SHAPE otherwise), W 16-byte
 *    aligned, X and Y 4-byte aligned.
 *  - The 12 MiB array is reserved on each device where the library's kernels
 *    are first loaded and stays until that device's context is destroyed.
 *    The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  A device reset after it is not supported.
 *  - All calls share the array: calls whose GPU work overlaps race on it. */
gq_status gq_mul_mat_q4_0_noalloc(const void *W, int64_t M, int64_t K, const float *X, int64_t N, float *Y,
                                  void *stream);

/* y[i] = bf16(x[i]), round to nearest even (NaN stays NaN), for n elements. */
gq_status gq_f32_to_bf16(const float *x, uint16_t *y, int64_t n, void *stream);

/* Synchronise `stream`, then read and clear the device error word.  Returns
 * GQ_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up since the last
 * call, else GQ_ERR_BAD_INDEX if gq_mul_mat_id_q4_0 met an expert id out of
 * range, GQ_ERR_CUDA if the synchronisation failed, else GQ_OK. */
gq_status gq_sync_status(void *stream);

/* Tuning / test options (process-wide). */
typedef enum {
  GQ_OPT_PREFILL_MIN_N = 0,  /* N at which mul_mat switches to the tensor-core path (default 16) */
  GQ_OPT_FORCE_GENERIC = 1,  /* 1: every mul_mat takes the generic kernel (test aid) */
  GQ_OPT_WAIT_LIMIT_NS = 2,  /* bound on any in-kernel wait, nanoseconds (default 2e9) */
  GQ_OPT_WEIGHTS_STATIC = 3, /* 1: promise that no kernel launched right before a mul_mat on the same
                                stream writes its W, so the decode kernel (and the first chunks of the
                                tensor-core kernel) may start streaming W while that kernel finishes
                                (weight-stationary inference); default 0 */
  GQ_OPT_DECODE_VARIANT = 4, /* tuning: tile/warp layout of the N <= 32 decode kernel, 0..4 (default 0);
                                every variant computes the same result */
  GQ_OPT_PDL = 5,            /* 1 (default): launch kernels with programmatic dependent launch, so a
                                kernel may start while the previous one on the stream drains; every
                                write of Y waits for that previous kernel, and so does every read of X
                                unless GQ_OPT_X_STATIC promises otherwise */
  GQ_OPT_PREFILL_TILE_N = 6, /* tuning: token-tile width of the 1-CTA tensor-core kernel, 0 = by shape
                                (default), 128 or 256; a non-zero value also selects the 1-CTA kernel */
  GQ_OPT_PREFILL_PAIR = 7,   /* 1: N > 128 runs the 2-SM kernel (CTA pairs, 256 x 256 tiles);
                                0 (default): the 1-CTA kernel */
  GQ_OPT_PREFILL_STREAMK = 8, /* k-splitting of tiles in the tensor-core kernel: 1 (default) = when the
                                last wave of tiles would leave SMs idle, its tiles are split along k
                                over the idle SMs and the pieces summed in k order (the result does
                                not depend on timing); 0 = whole tiles only; n >= 2 = every tile
                                in n pieces (test aid) */
  GQ_OPT_PREFILL_SLOTS = 9,   /* test aid: run the tensor-core kernel as if the GPU had this many SMs
                                (CTA pairs: pairs); 0 (default) = the real count */
  GQ_OPT_DECODE_EARLY_STAGES = 10, /* with GQ_OPT_WEIGHTS_STATIC: how many ring stages of W the decode
                                kernel streams before the previous kernel finishes (1..64, capped by the
                                ring, default 2); later stages wait until x is staged */
  GQ_OPT_X_STATIC = 11,       /* 1: promise that X was completely written before the most recent call
                                on this stream made without the promise (e.g. several projections of
                                one activation: the first call without it, the others with it; or
                                activations copied in before a run of calls).  The decode kernel (N
                                below the tensor-core threshold) and gq_mul_mat_q4_0_bf16x then read X
                                and compute while the kernels ahead of them on the stream finish; Y
                                (and the tensor-core kernel's k-split scratch) are written only after
                                them.  A call without the promise reads X only after every kernel
                                ahead of it has finished, and lets later launches start only then, so
                                it orders everything after it.  Default 0 */
  GQ_OPT_MOE_PATH = 12,       /* gq_mul_mat_id_q4_0 kernel: 0 (default) by tokens per used expert,
                                1 decode kernel, 2 tensor-core kernel (fast-path shapes only) */
  GQ_OPT_TEST_DROP_ARRIVE = 13 /* test aid for the timeout path, 0 (default) off: 1 = the decode kernel's
                                W producer in CTA 0 never issues its second ring stage, 2 = the
                                tensor-core kernel's W producer in CTA 0 never issues its second raw
                                chunk.  The stage's consumers then wait out GQ_OPT_WAIT_LIMIT_NS, the
                                kernel drains what it issued, releases tensor memory and returns, and
                                gq_sync_status() reports GQ_ERR_DEVICE_TIMEOUT.  Nothing faults. */
} gq_option;
gq_status gq_set_option(gq_option opt, int64_t value);
int64_t gq_get_option(gq_option opt);

/* Human-readable text of the last error on this thread ("" if none). */
const char *gq_last_error(void);
const char *gq_status_string(gq_status s);

/* Library version: major*10000 + minor*100 + patch. */
int gq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H */
