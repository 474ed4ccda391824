// K2: decode / small-N MUL_MAT against Q4_0 (and Q4_1 / Q8_0) weights, plus
// the generic fallback kernel.
//
// Y[n][m] = sum_k w[m][k] * X[n][k],  w = d*(q-8)  ("Binding GGUF weights to
// the compute graph", section 2.3: blocks are dequantised inside MUL_MAT;
// "GGUF loading, mmap and tensor placement", step six: W ne=[K,M], b ne=[K,N]).
//
// Design (decode is HBM-bound: 0.5625 bytes of W per weight, N <= 64 tokens):
//  * A producer warp streams W with 2-D TMA boxes of 16 rows x 144 bytes (256
//    weights, 8 blocks per row) into a ring of shared-memory stages; each
//    stage holds KW such boxes, one per consumer warp (split-K inside the CTA).
//  * Consumer warps run mma.sync m16n8k16 (fp16 in, fp32 accumulate) with the
//    16 W rows as the A operand and up to 8 tokens per n8 tile as B.  A holds
//    codes straight from one LOP3 per pair: the fp16 bit pattern 0x6400 | q is
//    exactly 1024 + q (low nibbles) and 0x6400 | (q << 4) is 1024 + 16q (high
//    nibbles, met by x/16 in B).  The exact bias this adds, 1032*x + 1152*(x/16)
//    summed over the block, is precomputed per block and token and enters as
//    the MMA's C input with a minus sign, so each block's MMA pair yields
//    sum (q-8)*x directly.  The block scale d is then applied in fp32 to that
//    partial, so W is never rounded; only x is (fp16, relative <= 2^-11;
//    a token whose largest |x| in a warp's blocks reaches 2^15 or stays below
//    2^-10 is staged times an exact power of two and the warp's partial sums
//    are multiplied back).
//  * The four bytes of codes a lane needs are read straight from the raw
//    18-byte blocks: two blocks (36 bytes) form nine aligned 32-bit words, and
//    one PRMT rebuilds the word that straddles the scale of the even block.
//    Which 8 codes a lane owns therefore depends on the block's parity; the
//    x fragments staged in shared memory follow the same permutation of k
//    (a contraction does not care how k is ordered, only that A and B agree).
//  * The k-warps' partial sums of a 16-row tile are reduced through shared
//    memory; CTAs loop over tiles persistently.
//  * Launched with programmatic dependent launch: the grid may start while
//    the previous kernel on the stream drains; X is read and Y written only
//    after griddepcontrol.wait.  With `early_w` set, the producer also starts
//    streaming W before that wait (valid when the previous kernel does not
//    write W, as in weight-stationary inference); with `x_static` X is read
//    and the MMAs run before it too, and only the warp writing Y waits.
//  * The same kernel serves Q4_1 and Q8_0 blocks (F: 20- and 34-byte blocks,
//    their own code extraction and bias), Q4_K super-blocks (one 144-byte
//    super-block per box row; each 32-weight sub-block is a staging block of
//    its own with its scale d*sc_j and min dmin*m_j, its codes the low
//    (even sub-block) or high (odd) nibbles of 32 code bytes) and MUL_MAT_ID (MOE: groups of
//    routed tokens of one expert; a single token's slots read their expert
//    ids directly).
#include <algorithm>
#include <type_traits>
#include <cuda_fp16.h>

#include "gq_internal.h"
#include "gq_ptx.cuh"
#include "gq_q4k.cuh"

namespace gq {
namespace {

constexpr int kSubK = 256;         // weights per row per TMA box
constexpr int kSubBytesRow = 144;  // 8 blocks x 18 bytes (Q4_0)

// Bytes of one row of a TMA box (256 weights): Q4_0 144, Q4_1 160, Q8_0 272,
// Q4_K 144 (one super-block), Q5_0 176, Q5_1 192.
template <int F>
constexpr int sub_bytes_row() {
  return F == GQ_TYPE_Q4_1   ? 160
         : F == GQ_TYPE_Q8_0 ? 272
         : F == GQ_TYPE_Q5_0 ? 176
         : F == GQ_TYPE_Q5_1 ? 192
                             : kSubBytesRow;
}

// NT: n8 token tiles (N <= 8*NT); MT: m16 row tiles per warp (tile = 16*MT
// rows); KW: consumer warps, each taking one 256-k box of every stage; F: the
// block format (Q4_0, or Q4_1 whose min offset needs a second per-block table
// of x sums).
template <int NT, int MT, int KW, int STAGES, int F = GQ_TYPE_Q4_0>
struct DecodeCfg {
  static constexpr int kBM = 16 * MT;
  static constexpr int kRowBytes = sub_bytes_row<F>();
  static constexpr int kElem = kRowBytes > 256 ? 2 : 1;  // TMA element bytes (a box is at most 256 wide)
  // Q4_1, Q4_K and Q5_1 also keep per-block x sums for their min offsets
  static constexpr int kTables = (F == GQ_TYPE_Q4_1 || F == GQ_TYPE_Q4_K || F == GQ_TYPE_Q5_1) ? 2 : 1;
  static constexpr int kSubBytes = kBM * kRowBytes;
  static constexpr int kThreads = 32 * (KW + 1);
  static constexpr int kStageK = kSubK * KW;
  static constexpr int kStageBytes = kSubBytes * KW;
  static constexpr int kRingBytes = kStageBytes * STAGES;
  static constexpr int kSlots = STAGES + 1;  // tile accumulators in flight (see the reduction below)
  // one partial per k-warp: [KW][kBM][N] floats per slot
  __host__ __device__ static size_t slot_floats(int N) { return static_cast<size_t>(KW) * kBM * N; }
  // x fragments (2*KX*N bytes) + bias table (KX/32 blocks x N tokens, N rounded up to even)
  __host__ __device__ static size_t xs_bytes(int N, int KX) { return static_cast<size_t>(2) * KX * N; }
  __host__ __device__ static int cs_stride(int N) { return N + (N & 1); }
  __host__ __device__ static size_t cs_bytes(int N, int KX) {
    return static_cast<size_t>(KX / 32) * cs_stride(N) * sizeof(float);
  }
  // + per consumer warp and token the power-of-two factor its x was staged with
  static size_t smem_bytes(int N, int KX) {
    return kRingBytes + xs_bytes(N, KX) + kTables * cs_bytes(N, KX) +
           (kSlots * slot_floats(N) + kSlots + static_cast<size_t>(KW) * N) * sizeof(float) + (2 * STAGES + 1) * 8 +
           16 + 128;
  }
};

// x is staged as fp16 (x for the low nibbles, x/16 for the high ones).  A
// warp's chunk of a token whose largest |x| is m >= 2^15 would overflow fp16,
// and one whose m is below 2^-10 would leave the normal fp16 range (m/16 <
// 2^-14, where fp16 keeps fewer than 11 significant bits); such a chunk is
// staged as x * 2^e with the power of two that brings m into [2^14, 2^15)
// (clamped so that 2^e and 2^-e are normal fp32 numbers).  Any other chunk,
// and one whose m is 0 or non-finite (which then propagates as it would
// unscaled), keeps the factor 1.
constexpr float kXScaleFrom = 32768.f;          // 2^15
constexpr float kXScaleBelow = 0.0009765625f;   // 2^-10
__device__ __forceinline__ float x_scale(float m) {
  if (!(m >= kXScaleFrom || (m > 0.f && m < kXScaleBelow)) || !isfinite(m)) return 1.f;
  const int E = ((__float_as_int(m) >> 23) & 0xFF) - 127;  // m in [2^E, 2^(E+1)) (subnormal m: E = -127)
  const int e = max(-126, min(126, 14 - E));
  return __int_as_float((e + 127) << 23);                   // m * 2^e in [2^14, 2^15)
}
// 1/f for f a normal power of two, exactly (the exponent reflected about 0).
__device__ __forceinline__ float pow2_inverse(float f) { return __int_as_float((254 << 23) - __float_as_int(f)); }

// Bytes of the two 16-bit halves -> fp32 scale.
__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(w >> 16)));
}

// Word of 8 codes (bytes c0..c3) -> four f16x2 registers of biased codes:
// lo02 = (1024+q) of c0, c2 low nibbles, lo13 = c1, c3 low nibbles,
// hi02 / hi13 = (1024+16q) of the high nibbles.  One LOP3 each, all exact.
__device__ __forceinline__ void codes_to_f16(uint32_t v, uint32_t& lo02, uint32_t& lo13, uint32_t& hi02,
                                             uint32_t& hi13) {
  const uint32_t kMagic = 0x64006400u;  // fp16 1024 in both halves
  const uint32_t v8 = v >> 8;
  lo02 = lop3_and_or(v, 0x000F000Fu, kMagic);
  lo13 = lop3_and_or(v8, 0x000F000Fu, kMagic);
  hi02 = lop3_and_or(v, 0x00F000F0u, kMagic);
  hi13 = lop3_and_or(v8, 0x00F000F0u, kMagic);
}

// Stage x for one (block, token): four lane-slot fragments and the negated bias.
// Slot t of an even block holds code bytes c = {4t+2, 4t+3, 4t+4, 4t+5} (t < 3)
// or {0, 1, 14, 15} (t = 3); of an odd block c = {4t, .., 4t+3}.  The slot is
// [x[c0], x[c2], x[c1], x[c3]] (fp16) and [x[16+c0], x[16+c2], x[16+c1],
// x[16+c3]] / 16 (fp16), matching the A fragments built from those bytes.
template <int PARITY>
__device__ __forceinline__ float stage_block(const float (&x)[32], uint4* dst) {
  float bias = 0.f;
  __half xh[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    xh[j] = __float2half_rn(x[j]);
    xh[16 + j] = __float2half_rn(x[16 + j] * 0.0625f);
    bias = fmaf(1032.f, __half2float(xh[j]), bias);
    bias = fmaf(1152.f, __half2float(xh[16 + j]), bias);
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    int c0, c1, c2, c3;
    if (PARITY) {
      c0 = 4 * t; c1 = 4 * t + 1; c2 = 4 * t + 2; c3 = 4 * t + 3;
    } else if (t < 3) {
      c0 = 4 * t + 2; c1 = 4 * t + 3; c2 = 4 * t + 4; c3 = 4 * t + 5;
    } else {
      c0 = 0; c1 = 1; c2 = 14; c3 = 15;
    }
    __half2 h;
    uint4 pk;
    h = __halves2half2(xh[c0], xh[c2]); pk.x = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[c1], xh[c3]); pk.y = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c0], xh[16 + c2]); pk.z = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c1], xh[16 + c3]); pk.w = *reinterpret_cast<uint32_t*>(&h);
    dst[t] = pk;
  }
  return -bias;
}

// Q4_1 x staging: the natural k order (a lane owns code bytes 4t .. 4t+3 of
// every block, like an odd Q4_0 block), codes biased by 1024 with no zero
// point (A = 1024 + q for low nibbles, 1024 + 16q against x/16 for high
// ones), so the bias is 1024 * (sum of the fp16 x and x/16 values).  Also the
// block's sum of x as the MMA sees it (fp16 x, 16 * fp16(x/16)), which the
// min offset multiplies.
__device__ __forceinline__ float stage_block_q41(const float (&x)[32], uint4* dst, float* sx) {
  float bias = 0.f, sum = 0.f;
  __half xh[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    xh[j] = __float2half_rn(x[j]);
    xh[16 + j] = __float2half_rn(x[16 + j] * 0.0625f);
    bias += __half2float(xh[j]) + __half2float(xh[16 + j]);
    sum = fmaf(16.f, __half2float(xh[16 + j]), sum + __half2float(xh[j]));
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int c0 = 4 * t, c1 = 4 * t + 1, c2 = 4 * t + 2, c3 = 4 * t + 3;
    __half2 h;
    uint4 pk;
    h = __halves2half2(xh[c0], xh[c2]); pk.x = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[c1], xh[c3]); pk.y = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c0], xh[16 + c2]); pk.z = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c1], xh[16 + c3]); pk.w = *reinterpret_cast<uint32_t*>(&h);
    dst[t] = pk;
  }
  *sx = sum;
  return -1024.f * bias;
}

// Q4_K x staging of one 32-weight sub-block (natural k order, like Q4_1).  Its
// codes are the low nibbles (even sub-block: A = 1024 + q against fp16 x) or
// the high nibbles (odd: A = 1024 + 16q against fp16 x/16) of 32 code bytes,
// bytes 0-15 feeding the first MMA (fragment halves x, y) and bytes 16-31 the
// second (z, w).  The bias is 1024 * (sum of the staged values); the x sum the
// sub-block's min multiplies is the staged sum (times 16 when odd).
__device__ __forceinline__ float stage_block_q4k(const float (&x)[32], uint4* dst, float* sx, int odd) {
  const float f = odd ? 0.0625f : 1.f;
  float staged = 0.f;
  __half xh[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    xh[j] = __float2half_rn(x[j] * f);
    staged += __half2float(xh[j]);
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int c0 = 4 * t, c1 = 4 * t + 1, c2 = 4 * t + 2, c3 = 4 * t + 3;
    __half2 h;
    uint4 pk;
    h = __halves2half2(xh[c0], xh[c2]); pk.x = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[c1], xh[c3]); pk.y = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c0], xh[16 + c2]); pk.z = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c1], xh[16 + c3]); pk.w = *reinterpret_cast<uint32_t*>(&h);
    dst[t] = pk;
  }
  *sx = odd ? 16.f * staged : staged;
  return -1024.f * staged;
}

// Q5_0 / Q5_1 x staging: the natural k order (a lane owns code bytes 4t ..
// 4t+3, as for Q4_1) with 5-bit codes: A = 1024 + q against fp16 x (low
// nibbles) and 1024 + 16q against fp16 x/16 (high nibbles).  Q5_0's zero point
// 16 joins the bias: 1040 * sum(x) + 1280 * sum(x/16); Q5_1 keeps 1024 times
// the staged sums and, for its min, the x sum as the MMA sees it.
template <int F>
__device__ __forceinline__ float stage_block_q5(const float (&x)[32], uint4* dst, float* sx) {
  float lo = 0.f, hi = 0.f;
  __half xh[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    xh[j] = __float2half_rn(x[j]);
    xh[16 + j] = __float2half_rn(x[16 + j] * 0.0625f);
    lo += __half2float(xh[j]);
    hi += __half2float(xh[16 + j]);
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int c0 = 4 * t, c1 = 4 * t + 1, c2 = 4 * t + 2, c3 = 4 * t + 3;
    __half2 h;
    uint4 pk;
    h = __halves2half2(xh[c0], xh[c2]); pk.x = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[c1], xh[c3]); pk.y = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c0], xh[16 + c2]); pk.z = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + c1], xh[16 + c3]); pk.w = *reinterpret_cast<uint32_t*>(&h);
    dst[t] = pk;
  }
  if constexpr (F == GQ_TYPE_Q5_1) {
    *sx = fmaf(16.f, hi, lo);
    return -1024.f * (lo + hi);
  } else {
    return -(1040.f * lo + 1280.f * hi);
  }
}

// Bits 0-3 of b to bit 0 of bytes 0-3 (the four products b_i * 2^(7j) land on
// distinct bits, so the multiply carries nothing into the mask).
__device__ __forceinline__ uint32_t spread4(uint32_t b) { return (b * 0x00204081u) & 0x01010101u; }

// A code word of a Q5 block (bytes c0..c3 = elements 4t..4t+3 low, 16+4t..
// high) with the block's high-bit word qh -> the four f16x2 A registers of
// biased 5-bit codes: lo02 / lo13 = 1024 + q of (c0, c2) / (c1, c3) low
// nibbles, hi02 / hi13 = 1024 + 16q of the high ones.
__device__ __forceinline__ void q5_codes_to_f16(uint32_t v, uint32_t qh, int t, uint32_t& lo02, uint32_t& lo13,
                                                uint32_t& hi02, uint32_t& hi13) {
  const uint32_t kMagic = 0x64006400u;
  const uint32_t q5lo = (v & 0x0F0F0F0Fu) | (spread4((qh >> (4 * t)) & 0xFu) << 4);
  const uint32_t q5hi = ((v >> 4) & 0x0F0F0F0Fu) | (spread4((qh >> (16 + 4 * t)) & 0xFu) << 4);
  lo02 = lop3_and_or(q5lo, 0x001F001Fu, kMagic);
  lo13 = lop3_and_or(q5lo >> 8, 0x001F001Fu, kMagic);
  hi02 = lop3_and_or(q5hi << 4, 0x01F001F0u, kMagic);
  hi13 = lop3_and_or(q5hi >> 4, 0x01F001F0u, kMagic);
}

// Half of the biased codes of a word of 4 code bytes (c0..c3): the low
// nibbles as fp16 1024 + q, or the high nibbles as 1024 + 16q, in the pairs
// (c0, c2) and (c1, c3).
__device__ __forceinline__ void codes_half_f16(uint32_t v, int hi, uint32_t& r02, uint32_t& r13) {
  const uint32_t kMagic = 0x64006400u;
  const uint32_t mask = hi ? 0x00F000F0u : 0x000F000Fu;
  r02 = lop3_and_or(v, mask, kMagic);
  r13 = lop3_and_or(v >> 8, mask, kMagic);
}

// Q8_0 x staging: a lane owns elements 4t .. 4t+3 of each half of a block
// (k 2t, 2t+1 <- 4t, 4t+1 and k 2t+8, 2t+9 <- 4t+2, 4t+3 in the MMA); the codes
// enter as fp16 1024 + (c ^ 0x80) = 1152 + q, so the bias is 1152 * sum(x).
__device__ __forceinline__ float stage_block_q80(const float (&x)[32], uint4* dst) {
  float bias = 0.f;
  __half xh[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    xh[j] = __float2half_rn(x[j]);
    bias += __half2float(xh[j]);
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    __half2 h;
    uint4 pk;
    h = __halves2half2(xh[4 * t], xh[4 * t + 1]); pk.x = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[4 * t + 2], xh[4 * t + 3]); pk.y = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + 4 * t], xh[16 + 4 * t + 1]); pk.z = *reinterpret_cast<uint32_t*>(&h);
    h = __halves2half2(xh[16 + 4 * t + 2], xh[16 + 4 * t + 3]); pk.w = *reinterpret_cast<uint32_t*>(&h);
    dst[t] = pk;
  }
  return -1152.f * bias;
}

// Four int8 codes (one word) -> two f16x2 registers of 1024 + (c ^ 0x80):
// (c0, c1) and (c2, c3).
__device__ __forceinline__ void q8_to_f16(uint32_t v, uint32_t& r01, uint32_t& r23) {
  const uint32_t u = v ^ 0x80808080u;
  r01 = prmt(u, 0x64646464u, 0x4140u);
  r23 = prmt(u, 0x64646464u, 0x4342u);
}

// Two CTAs per SM only where the ring leaves room for a second one and x is
// one token tile (more tokens' x fragments fill the rest of shared memory);
// otherwise let the kernel use the registers of a single CTA.
template <int NT, int MT, int KW, int STAGES, int F = GQ_TYPE_Q4_0>
constexpr int decode_min_blocks() {
  return (NT == 1 && STAGES * KW * 16 * MT * sub_bytes_row<F>() <= 80 * 1024) ? 2 : 1;
}

// Stage x for one (block, token) entry in the block format's fragment order:
// the fragments, the negated bias (cs[n]) and, for Q4_1 / Q4_K, the x sum (sx[n]);
// the padding column of an odd token count is zeroed with the last token.
template <int F>
__device__ __forceinline__ void stage_entry(const float (&xv)[32], uint4* dst, float* cs, float* sx, int n, int Nt,
                                            int parity) {
  if constexpr (F == GQ_TYPE_Q4_1) {
    cs[n] = stage_block_q41(xv, dst, &sx[n]);
    if ((Nt & 1) && n == Nt - 1) sx[Nt] = 0.f;
  } else if constexpr (F == GQ_TYPE_Q4_K) {
    cs[n] = stage_block_q4k(xv, dst, &sx[n], parity);  // parity: odd sub-block of its super-block
    if ((Nt & 1) && n == Nt - 1) sx[Nt] = 0.f;
  } else if constexpr (F == GQ_TYPE_Q5_0 || F == GQ_TYPE_Q5_1) {
    cs[n] = stage_block_q5<F>(xv, dst, &sx[n]);
    if (F == GQ_TYPE_Q5_1 && (Nt & 1) && n == Nt - 1) sx[Nt] = 0.f;
  } else if constexpr (F == GQ_TYPE_Q8_0) {
    cs[n] = stage_block_q80(xv, dst);
  } else {
    cs[n] = parity ? stage_block<1>(xv, dst) : stage_block<0>(xv, dst);
  }
  if ((Nt & 1) && n == Nt - 1) cs[Nt] = 0.f;
}

// The x staging's rare path (out of line): per token, the largest |x| over
// this warp's blocks of the chunk, its factor wsc[n] (x_scale), and the
// chunk's entries staged again as x * wsc[n].  Blocks past K were zeroed by
// the first pass.  perm: the token -> x row map of a routed MUL_MAT_ID group
// (or nullptr: row row0 + n).
template <int F, int kStageK>
__device__ __noinline__ void stage_x_scaled(const float* __restrict__ X, int K, const int* perm, int row0, int kc0,
                                            int kend,
                                            int nst, int N, int Nt, int kw, int lane, uint4* xs, float* cs,
                                            float* sxs, int csn, float* wsc) {
  constexpr int kBoxBlocks = kSubK / kQK;
  auto xrow = [&](int n) -> size_t {
    return perm ? static_cast<size_t>(__ldg(perm + n)) : static_cast<size_t>(row0 + n);
  };
  for (int n = lane; n < Nt; n += 32) {
    float m = 0.f;
    for (int st = 0; st < nst; ++st)
      for (int i = 0; i < kBoxBlocks; ++i) {
        const int bl = st * (kStageK / kQK) + kw * kBoxBlocks + i;
        if (kc0 + bl * kQK >= kend) continue;
        const float4* xr = reinterpret_cast<const float4*>(X + xrow(n) * K + static_cast<size_t>(kc0 + bl * kQK));
        for (int j = 0; j < 8; ++j) {
          const float4 v = __ldg(xr + j);
          m = fmaxf(fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
        }
      }
    wsc[n] = x_scale(m);
  }
  __syncwarp();
  const int nent = nst * kBoxBlocks * Nt;
  for (int e = lane; e < nent; e += 32) {
    const int st = e / (kBoxBlocks * Nt), rem = e % (kBoxBlocks * Nt);
    const int bl = st * (kStageK / kQK) + kw * kBoxBlocks + rem / Nt;
    const int n = rem % Nt;
    if (kc0 + bl * kQK >= kend) continue;
    const float f = wsc[n];
    float xv[32];
    const float4* xr = reinterpret_cast<const float4*>(X + xrow(n) * K + static_cast<size_t>(kc0 + bl * kQK));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = __ldg(xr + i);
      xv[4 * i] = v.x * f; xv[4 * i + 1] = v.y * f; xv[4 * i + 2] = v.z * f; xv[4 * i + 3] = v.w * f;
    }
    stage_entry<F>(xv, xs + (bl * N + n) * 4, cs + bl * csn, sxs + bl * csn, n, Nt, (kc0 / kQK + bl) & 1);
  }
  __syncwarp();
}

// MOE: MUL_MAT_ID over the decode groups of rt (expert e, up to N tokens
// each; with ONE, one token).  N is then the group capacity, which fixes the
// shared-memory layout;
// a group's own token count Nt <= N sets the work.  W rows of expert e start
// at e * M; x and Y rows are the pairs perm[first + n].  The CTAs are shared
// out evenly among the groups (each CTA taking every cpg-th tile of its
// group), or, with more groups than CTAs, CTA b runs groups b, b + grid, ...
template <int NT, int MT, int KW, int STAGES, bool ONE, bool MOE = false, int F = GQ_TYPE_Q4_0>
__global__ void __launch_bounds__(32 * (KW + 1), (decode_min_blocks<NT, MT, KW, STAGES, F>()))
    k_decode_q4_0(const __grid_constant__ CUtensorMap tmW, const float* __restrict__ X, int N, int M, int K,
                  int KX, float* __restrict__ Y, uint64_t limit_ns, uint32_t* err, int early_stages,
                  int x_static, const MoeRoute rt, int drop) {
  static_assert(F == GQ_TYPE_Q4_0 || !MOE, "the other block formats run the plain MUL_MAT layout");
  using Cfg = DecodeCfg<NT, MT, KW, STAGES, F>;
  constexpr int kBM = Cfg::kBM;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* ring = smem;
  uint4* xs = reinterpret_cast<uint4*>(smem + Cfg::kRingBytes);
  float* cs = reinterpret_cast<float*>(smem + Cfg::kRingBytes + Cfg::xs_bytes(N, KX));
  float* sxs = cs + Cfg::cs_bytes(N, KX) / sizeof(float);  // Q4_1: per-block x sums, laid out like cs
  float* acc_slots = cs + Cfg::kTables * Cfg::cs_bytes(N, KX) / sizeof(float);  // [kSlots][KW][kBM][N]
  const int csn = Cfg::cs_stride(N);
  const int slot_floats = static_cast<int>(Cfg::slot_floats(N));
  int* slot_count = reinterpret_cast<int*>(acc_slots + Cfg::kSlots * slot_floats);
  float* xsc = reinterpret_cast<float*>(slot_count + Cfg::kSlots);  // [KW][N]: x staged as x * xsc
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(xsc + KW * N) + 7) & ~uintptr_t(7));
  uint64_t* x_ready = bars + 2 * STAGES;  // every consumer warp has staged the first chunk of x
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (M + kBM - 1) / kBM;
  const int nchunks = (K + KX - 1) / KX;
  const int stages_per_chunk = KX / Cfg::kStageK;
  // Groups of this CTA: gk = 0 .. ngrp-1 is group g_first + gk * g_step, and
  // within it tiles t_first, t_first + t_step, ...
  int ngrp = 1, g_first = 0, g_step = 1, t_first = static_cast<int>(blockIdx.x), t_step = static_cast<int>(gridDim.x);
  // Group g: its expert (direct groups -- single-token launches only: pair g
  // alone, its id read here; an id outside [0, ne) marks the group bad).
  const bool direct = MOE && ONE && rt.ids != nullptr;
  auto grp_expert = [&](int g) -> int { return direct ? __ldg(rt.ids + g) : rt.groups[3 * g]; };
  auto grp_bad = [&](int e) -> bool { return direct && (e < 0 || e >= rt.ne); };
  if (MOE) {
    pdl_wait();  // the routing tables (or the ids) come from the kernel before
    const int ng = direct ? rt.np : rt.meta[1], grid = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    if (ng <= grid) {
      const int cpg = ng > 0 ? grid / ng : 1;
      g_first = b / cpg;
      ngrp = g_first < ng ? 1 : 0;
      t_first = b % cpg;
      t_step = cpg;
    } else {
      g_first = b;
      g_step = grid;
      ngrp = (ng - b + grid - 1) / grid;
      t_first = 0;
      t_step = 1;
    }
  }

  if (threadIdx.x < Cfg::kSlots) slot_count[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);            // full: producer's expect_tx arrive + tx bytes
      mbar_init(smem_u32(&bars[STAGES + s]), KW);  // empty: one arrive per consumer warp
    }
    mbar_init(smem_u32(x_ready), KW);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The next kernel on the stream may launch once every CTA has signalled.
  // A kernel that reads X only after the kernel before it (no x_static, or
  // MUL_MAT_ID, which waited above) signals after that wait, so that a later
  // x-static launch cannot start before the kernels ahead of this one are
  // done; an x-static kernel signals at once.
  if (MOE || x_static) pdl_launch_dependents();
  __syncthreads();

  if (warp == KW) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop and one elected lane issues: a converged
    // warp issues TMA faster than a lone lane of a diverged one.
    {
      const bool issuer = elect_one();
      if (issuer) tma_prefetch_desc(&tmW);
      // With early_stages > 0 the first stages of W stream before the previous
      // kernel finishes; the rest waits until x is staged, so that the x loads
      // right after the dependency do not queue behind a ring full of W.
      if (!early_stages) pdl_wait();
      bool x_waited = early_stages == 0;
      uint32_t q = 0;
      bool ok = true;
      for (int gk = 0; gk < ngrp && ok; ++gk)
      for (int c = 0; c < nchunks && ok; ++c) {
        const int ge = MOE ? grp_expert(g_first + gk * g_step) : 0;
        if (MOE && grp_bad(ge)) continue;  // the consumers skip it too
        const int wrow0 = ge * M;
        const int kc0 = c * KX;
        const int kend = min(K, kc0 + KX);
        const int nst = min(stages_per_chunk, (kend - kc0 + Cfg::kStageK - 1) / Cfg::kStageK);
        for (int tile = t_first; tile < ntiles && ok; tile += t_step) {
          for (int st = 0; st < nst; ++st, ++q) {
            const int slot = q % STAGES;
            const uint32_t ph = (q / STAGES) & 1;
            if (!x_waited && q >= static_cast<uint32_t>(early_stages)) {
              x_waited = true;
              if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(x_ready), 0, limit_ns, abort_flag, err))) {
                ok = false;
                break;
              }
            }
            if (!__all_sync(0xFFFFFFFFu,
                            mbar_wait_bounded(smem_u32(&bars[STAGES + slot]), ph ^ 1, limit_ns, abort_flag, err))) {
              ok = false;
              break;
            }
            // test hook: stage 1 of CTA 0 is never issued, so its consumers'
            // bounded wait runs out (GQ_OPT_TEST_DROP_ARRIVE)
            if (drop && blockIdx.x == 0 && q == 1) continue;
            const int k0 = kc0 + st * Cfg::kStageK;
            const int nvalid = min(KW, (kend - k0 + kSubK - 1) / kSubK);
            const uint32_t full = smem_u32(&bars[slot]);
            if (issuer) {
              mbar_arrive_expect_tx(full, nvalid * Cfg::kSubBytes);
              for (int j = 0; j < nvalid; ++j) {
                const int xb = ((k0 + j * kSubK) / kSubK) * (Cfg::kRowBytes / Cfg::kElem);  // element column
                tma_load_2d(smem_u32(ring + slot * Cfg::kStageBytes + j * Cfg::kSubBytes), &tmW, xb,
                            wrow0 + tile * kBM, full);
              }
            }
            __syncwarp();
          }
        }
      }
      if (!ok && issuer) {
        // Let copies already issued land before the CTA can exit.
        for (uint32_t i = 0; i < STAGES && i < q; ++i) {
          const uint32_t qq = q - 1 - i;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(&bars[qq % STAGES]), (qq / STAGES) & 1) &&
                 globaltimer_ns() - t0 < limit_ns) {
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int kw = warp;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t sel = (t == 3) ? 0x5432u : 0x7654u;  // even-block word: U, or Z.hi | U.lo for t == 3
  uint32_t q = 0;
  int tile_iter = 0;
  bool live = true;  // false once a bounded wait gave up; the loops still run to keep barriers matched
  // X may come from the previous kernel (unless the caller promised it does
  // not: x_static); Y may still be read by it, so Y is written after the wait.
  if (!x_static) {
    pdl_wait();
    if (!MOE) pdl_launch_dependents();
  }

  for (int gk = 0; gk < ngrp; ++gk)
  for (int c = 0; c < nchunks; ++c) {
    // Tokens of this group: Nt (<= N, the layout's width); token n's x and Y
    // row is xrow(n).
    int Nt = N, first = 0;
    if (MOE) {
      const int g = g_first + gk * g_step;
      if (direct) {
        first = g;
        Nt = 1;
        if (grp_bad(grp_expert(g))) {
          // A bad id: this CTA's rows of the pair's Y row become NaN.
          if (c == 0 && kw == 0) {
            for (int tile = t_first; tile < ntiles; tile += t_step)
              for (int r = lane; r < kBM; r += 32)
                if (tile * kBM + r < M) Y[static_cast<size_t>(g) * M + tile * kBM + r] = __int_as_float(0x7FC00000);
            if (lane == 0) atomicOr(err, DEVERR_BAD_ID);
          }
          continue;
        }
      } else {
        const int* grp = rt.groups + 3 * g;
        first = grp[1];
        Nt = grp[2];
      }
    }
    auto xrow = [&](int n) -> size_t {
      return MOE ? (direct ? static_cast<size_t>(first + n) : static_cast<size_t>(__ldg(rt.perm + first + n))) : n;
    };
    const int kc0 = c * KX;
    const int kend = min(K, kc0 + KX);
    const int nst = min(stages_per_chunk, (kend - kc0 + Cfg::kStageK - 1) / Cfg::kStageK);
    const int nbl = nst * Cfg::kStageK / kQK;  // local blocks covered by this chunk's stages

    // Stage this chunk of x: per (block, token) four fp16 lane-slot fragments
    // (k permuted like the codes) and the negated bias of the biased codes.
    // Each warp stages only the blocks of its own k boxes (box kw of every
    // stage), which only it reads: no CTA-wide barrier, so a warp starts on
    // its W as soon as its own x has arrived.
    // fp16 holds |x| < 65520 with 11 significant bits from 2^-14 on.  A token
    // whose largest |x| in this warp's blocks reaches 2^15, or stays below
    // 2^-10, is staged again as x * 2^e (exact; x_scale), and the warp's
    // partial sums for it are multiplied by 2^-e (exact); every other token
    // keeps the factor 1.  A lane notes the largest |x| it staged and whether
    // some block it staged was small but not all zero.
    __syncwarp();  // this warp's previous chunk of fragments is no longer read
    constexpr int kBoxBlocks = kSubK / kQK;  // 8
    const int nent = nst * kBoxBlocks * Nt;  // (stage, block of the box, token) entries of this warp
    float lmax = 0.f;                        // largest |x| this lane staged
    bool lsmall = false;                     // some staged block's largest |x| is in (0, 2^-10)
    for (int e = lane; e < nent; e += 32) {
      const int st = e / (kBoxBlocks * Nt), rem = e % (kBoxBlocks * Nt);
      const int bl = st * (Cfg::kStageK / kQK) + kw * kBoxBlocks + rem / Nt;  // block within the chunk
      const int n = rem % Nt;
      if (kc0 + bl * kQK >= kend) {
        // Past K inside the last 256-k box (rows padded to a multiple of 256
        // weights with zero blocks): zero x, so that the zero blocks add
        // exact zeros rather than whatever the slot held before.
        uint4* dst = xs + (bl * N + n) * 4;
        dst[0] = dst[1] = dst[2] = dst[3] = make_uint4(0u, 0u, 0u, 0u);
        cs[bl * csn + n] = 0.f;
        if ((Nt & 1) && n == Nt - 1) cs[bl * csn + Nt] = 0.f;
        if (Cfg::kTables == 2) {
          sxs[bl * csn + n] = 0.f;
          if ((Nt & 1) && n == Nt - 1) sxs[bl * csn + Nt] = 0.f;
        }
        continue;
      }
      float xv[32];
      const float4* xr =
          reinterpret_cast<const float4*>(X + xrow(n) * K + static_cast<size_t>(kc0 + bl * kQK));
      float em = 0.f;  // this block's largest |x|
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(xr + i);
        xv[4 * i] = v.x; xv[4 * i + 1] = v.y; xv[4 * i + 2] = v.z; xv[4 * i + 3] = v.w;
        em = fmaxf(fmaxf(em, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
      }
      lmax = fmaxf(lmax, em);
      lsmall |= em > 0.f && em < kXScaleBelow;
      stage_entry<F>(xv, xs + (bl * N + n) * 4, cs + bl * csn, sxs + bl * csn, n, Nt, (kc0 / kQK + bl) & 1);
    }
    const bool xwide = __any_sync(0xFFFFFFFFu, lmax >= kXScaleFrom || lsmall);
    if (xwide)
      stage_x_scaled<F, Cfg::kStageK>(X, K, (MOE && !direct) ? rt.perm + first : nullptr, MOE ? first : 0, kc0,
                                      kend, nst, N, Nt, kw, lane, xs, cs, sxs, csn, xsc + kw * N);
    __syncwarp();
    if (gk == 0 && c == 0 && lane == 0) mbar_arrive(smem_u32(x_ready));

    // The tiles of this chunk.  WIDE: this warp staged some token scaled by
    // xsc (rare), so its partial sums are taken back by 1 / xsc at the
    // hand-off; a separate copy of the loop, so that the usual one is not
    // touched by it.
    auto run_tiles = [&](auto wide_tag) {
    constexpr bool WIDE = decltype(wide_tag)::value;
    for (int tile = t_first; tile < ntiles; tile += t_step, ++tile_iter) {
      float acc[MT][NT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;

      for (int st = 0; st < nst; ++st, ++q) {
        const int slot = q % STAGES;
        if (live) live = mbar_wait_bounded(smem_u32(&bars[slot]), (q / STAGES) & 1, limit_ns, abort_flag, err);
        const int k0 = kc0 + st * Cfg::kStageK + kw * kSubK;
        if (live && k0 < kend) {
          const uint8_t* sub = ring + slot * Cfg::kStageBytes + kw * Cfg::kSubBytes + g * Cfg::kRowBytes;
          const int bl0 = (k0 - kc0) / kQK;
          const uint4* xsp = xs + (bl0 * N + g) * 4 + t;     // + block * 4N + nt * 32
          const float* csp = cs + bl0 * csn + 2 * t;         // + block * csn + nt * 8
          const uint4* xs1 = xs + bl0 * 4 + t;               // N = 1: token 0, slot t
          const float* cs1 = cs + bl0 * csn;                 // N = 1: token 0's bias
          const float* sxp = sxs + bl0 * csn + 2 * t;        // Q4_1 / Q4_K: x sums, like csp
          const float* sx1 = sxs + bl0 * csn;                // Q4_1 / Q4_K, N = 1
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            uint32_t wd[MT][2][2];  // [m-tile][row g / g+8][even / odd block] code words
            [[maybe_unused]] uint32_t wh[MT][2][2];  // Q8_0: the code word of the block's second half
            float dd[MT][2][2];     // scales
            float mm[MT][2][2];     // Q4_1 / Q4_K min offsets
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const uint8_t* rb = sub + (mt * 16 + 8 * r) * Cfg::kRowBytes;
                if constexpr (F == GQ_TYPE_Q5_0) {
                  // 22-byte blocks: the pair 2p, 2p+1 starts 4-byte aligned (44p).
                  // Even block: d in the low half of word 0, qh in bytes 2-5,
                  // code word t in bytes 6+4t..9+4t (straddling words); odd
                  // block (byte 22): d in the high half of word 5, qh word 6,
                  // code word t = word 7 + t.
                  const uint32_t* w = reinterpret_cast<const uint32_t*>(rb + 44 * p);
                  const uint32_t w0 = w[0];
                  wd[mt][r][0] = prmt(w[1 + t], w[2 + t], 0x5432u);
                  wh[mt][r][0] = prmt(w0, w[1], 0x5432u);
                  wd[mt][r][1] = w[7 + t];
                  wh[mt][r][1] = w[6];
                  dd[mt][r][0] = half_lo(w0);
                  dd[mt][r][1] = half_hi(w[5]);
                  mm[mt][r][0] = mm[mt][r][1] = 0.f;
                } else if constexpr (F == GQ_TYPE_Q5_1) {
                  // 24-byte blocks, all fields word-aligned: d | m << 16, qh, 4 code words.
                  const uint32_t* w = reinterpret_cast<const uint32_t*>(rb + 48 * p);
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const uint32_t H = w[6 * e];
                    wh[mt][r][e] = w[6 * e + 1];
                    wd[mt][r][e] = w[6 * e + 2 + t];
                    dd[mt][r][e] = half_lo(H);
                    mm[mt][r][e] = half_hi(H);
                  }
                } else if constexpr (F == GQ_TYPE_Q4_K) {
                  // One 144-byte super-block per box row: sub-blocks 2p (low
                  // nibbles) and 2p+1 (high nibbles) of code bytes 32p .. 32p+31;
                  // a lane takes code words t and t + 4 of them.  w = d*sc*q -
                  // dmin*m: scale d*sc (exact in fp32), min offset -dmin*m.
                  const uint32_t* hw = reinterpret_cast<const uint32_t*>(rb);
                  const uint32_t H = hw[0], F0 = hw[1], F1 = hw[2], F2 = hw[3];
                  wd[mt][r][0] = wd[mt][r][1] = hw[4 + 8 * p + t];
                  wh[mt][r][0] = wh[mt][r][1] = hw[8 + 8 * p + t];
                  const float d = half_lo(H), dmin = half_hi(H);
                  uint32_t sc0, m0, sc1, m1;
                  if (p == 0) {
                    q4k_scale_min<0>(F0, F1, F2, sc0, m0);
                    q4k_scale_min<1>(F0, F1, F2, sc1, m1);
                  } else if (p == 1) {
                    q4k_scale_min<2>(F0, F1, F2, sc0, m0);
                    q4k_scale_min<3>(F0, F1, F2, sc1, m1);
                  } else if (p == 2) {
                    q4k_scale_min<4>(F0, F1, F2, sc0, m0);
                    q4k_scale_min<5>(F0, F1, F2, sc1, m1);
                  } else {
                    q4k_scale_min<6>(F0, F1, F2, sc0, m0);
                    q4k_scale_min<7>(F0, F1, F2, sc1, m1);
                  }
                  dd[mt][r][0] = d * static_cast<float>(sc0);
                  dd[mt][r][1] = d * static_cast<float>(sc1);
                  mm[mt][r][0] = -(dmin * static_cast<float>(m0));
                  mm[mt][r][1] = -(dmin * static_cast<float>(m1));
                } else if constexpr (F == GQ_TYPE_Q4_1) {
                  // 20-byte blocks: word 0 = d | m << 16, words 1..4 the codes
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const uint8_t* bb = rb + 20 * (2 * p + e);
                    const uint32_t H = *reinterpret_cast<const uint32_t*>(bb);
                    wd[mt][r][e] = *reinterpret_cast<const uint32_t*>(bb + 4 + 4 * t);
                    dd[mt][r][e] = half_lo(H);
                    mm[mt][r][e] = half_hi(H);
                  }
                } else if constexpr (F == GQ_TYPE_Q8_0) {
                  // 34-byte blocks: the pair 2p, 2p+1 starts 4-byte aligned (68p).
                  // Even block: d in the low half of word 0, code word k is the
                  // high half of word k and the low half of word k+1.  Odd block
                  // (byte 34): d in the high half of word 8, code word k is word
                  // 9 + k.  A lane takes code words t and t + 4 of each block.
                  const uint32_t* w = reinterpret_cast<const uint32_t*>(rb + 68 * p);
                  const uint32_t w0 = w[0], w8 = w[8];
                  wd[mt][r][0] = prmt(w[t], w[t + 1], 0x5432u);
                  wh[mt][r][0] = prmt(w[t + 4], w[t + 5], 0x5432u);
                  wd[mt][r][1] = w[9 + t];
                  wh[mt][r][1] = w[13 + t];
                  dd[mt][r][0] = half_lo(w0);
                  dd[mt][r][1] = half_hi(w8);
                  mm[mt][r][0] = mm[mt][r][1] = 0.f;
                } else {
                  rb += 36 * p;
                  const uint32_t Z = *reinterpret_cast<const uint32_t*>(rb);
                  const uint32_t U = *reinterpret_cast<const uint32_t*>(rb + 4 + 4 * t);
                  const uint32_t W4 = *reinterpret_cast<const uint32_t*>(rb + 16);
                  const uint32_t Y1 = *reinterpret_cast<const uint32_t*>(rb + 20 + 4 * t);
                  wd[mt][r][0] = prmt(Z, U, sel);
                  wd[mt][r][1] = Y1;
                  dd[mt][r][0] = half_lo(Z);
                  dd[mt][r][1] = half_hi(W4);
                  mm[mt][r][0] = mm[mt][r][1] = 0.f;
                }
              }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int b = 2 * p + e;
              uint4 xf[NT];
              float2 nb[NT];
              float2 sxv[NT];  // Q4_1 / Q4_K: the columns' x sums of this block
              if (ONE) {
                // N = 1: every lane takes token 0's fragment (columns 1..7 then
                // repeat column 0 and are never stored) and its bias.
                xf[0] = xs1[b * 4];
                const float bias = cs1[b * 2];  // stride of the bias table for N = 1
                nb[0] = make_float2(bias, 0.f);
                sxv[0] = make_float2(Cfg::kTables == 2 ? sx1[b * 2] : 0.f, 0.f);
              } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  xf[nt] = (nt * 8 + g < Nt) ? xsp[b * 4 * N + nt * 32] : make_uint4(0u, 0u, 0u, 0u);
                  nb[nt] = (nt * 8 + 2 * t < Nt) ? *reinterpret_cast<const float2*>(csp + b * csn + nt * 8)
                                                 : make_float2(0.f, 0.f);
                  sxv[nt] = (Cfg::kTables == 2 && nt * 8 + 2 * t < Nt)
                                ? *reinterpret_cast<const float2*>(sxp + b * csn + nt * 8)
                                : make_float2(0.f, 0.f);
                }
              }
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                uint32_t a_lo[4], a_hi[4];
                if constexpr (F == GQ_TYPE_Q5_0 || F == GQ_TYPE_Q5_1) {
                  q5_codes_to_f16(wd[mt][0][e], wh[mt][0][e], t, a_lo[0], a_lo[2], a_hi[0], a_hi[2]);
                  q5_codes_to_f16(wd[mt][1][e], wh[mt][1][e], t, a_lo[1], a_lo[3], a_hi[1], a_hi[3]);
                } else if constexpr (F == GQ_TYPE_Q4_K) {
                  // sub-block 2p + e: code bytes 0-15 (word wd) then 16-31 (word wh)
                  codes_half_f16(wd[mt][0][e], e, a_lo[0], a_lo[2]);
                  codes_half_f16(wd[mt][1][e], e, a_lo[1], a_lo[3]);
                  codes_half_f16(wh[mt][0][e], e, a_hi[0], a_hi[2]);
                  codes_half_f16(wh[mt][1][e], e, a_hi[1], a_hi[3]);
                } else if constexpr (F == GQ_TYPE_Q8_0) {
                  q8_to_f16(wd[mt][0][e], a_lo[0], a_lo[2]);
                  q8_to_f16(wd[mt][1][e], a_lo[1], a_lo[3]);
                  q8_to_f16(wh[mt][0][e], a_hi[0], a_hi[2]);
                  q8_to_f16(wh[mt][1][e], a_hi[1], a_hi[3]);
                } else {
                  codes_to_f16(wd[mt][0][e], a_lo[0], a_lo[2], a_hi[0], a_hi[2]);
                  codes_to_f16(wd[mt][1][e], a_lo[1], a_lo[3], a_hi[1], a_hi[3]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  float tsum[4];
                  const float init[4] = {nb[nt].x, nb[nt].y, nb[nt].x, nb[nt].y};
                  mma_m16n8k16_f16(tsum, a_lo, xf[nt].x, xf[nt].y, init);
                  mma_m16n8k16_f16(tsum, a_hi, xf[nt].z, xf[nt].w, tsum);
                  if constexpr (Cfg::kTables == 2) {
                    // sum (d q + m) x = d * sum(q x) + m * sum(x)
                    acc[mt][nt][0] = fmaf(mm[mt][0][e], sxv[nt].x, fmaf(dd[mt][0][e], tsum[0], acc[mt][nt][0]));
                    acc[mt][nt][2] = fmaf(mm[mt][1][e], sxv[nt].x, fmaf(dd[mt][1][e], tsum[2], acc[mt][nt][2]));
                    if (!ONE) {
                      acc[mt][nt][1] = fmaf(mm[mt][0][e], sxv[nt].y, fmaf(dd[mt][0][e], tsum[1], acc[mt][nt][1]));
                      acc[mt][nt][3] = fmaf(mm[mt][1][e], sxv[nt].y, fmaf(dd[mt][1][e], tsum[3], acc[mt][nt][3]));
                    }
                  } else {
                    acc[mt][nt][0] = fmaf(dd[mt][0][e], tsum[0], acc[mt][nt][0]);
                    acc[mt][nt][2] = fmaf(dd[mt][1][e], tsum[2], acc[mt][nt][2]);
                    if (!ONE) {  // with N = 1 only column 0 (c0, c2) is ever stored
                      acc[mt][nt][1] = fmaf(dd[mt][0][e], tsum[1], acc[mt][nt][1]);
                      acc[mt][nt][3] = fmaf(dd[mt][1][e], tsum[3], acc[mt][nt][3]);
                    }
                  }
                }
              }
            }
          }
        }
        __syncwarp();
        if (live && lane == 0) mbar_arrive(smem_u32(&bars[STAGES + slot]));
      }

      // Hand this warp's partial sums to the tile's shared slot; the last of
      // the KW warps to arrive adds the KW partials in a fixed order (so the
      // result does not depend on timing), writes Y and releases the slot.  A
      // warp cannot run more than STAGES tiles ahead of the slowest one (it
      // needs the stages that warp still has to release), so kSlots =
      // STAGES + 1 slots are never reused while still in use.
      const int aslot = tile_iter % Cfg::kSlots;
      float* as = acc_slots + aslot * slot_floats;
      float* mine = as + kw * kBM * Nt;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = nt * 8 + 2 * t + (i & 1);
            if (n < Nt)
              mine[n * kBM + mt * 16 + g + 8 * (i >> 1)] =
                  WIDE ? acc[mt][nt][i] * pow2_inverse(xsc[kw * N + n]) : acc[mt][nt][i];
          }
      __syncwarp();
      int prev = 0;
      if (lane == 0) {
        __threadfence_block();
        prev = atomicAdd(&slot_count[aslot], 1);
      }
      prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
      if (prev == KW - 1) {
        if (x_static) pdl_wait();
        __threadfence_block();
        // Partials are [warp][token][row]: lanes walk rows, so the shared
        // reads are conflict-free and the Y stores coalesce along m.  After
        // the first x chunk, Y already holds the earlier chunks' sums: load
        // all of them before any store (independent loads, one latency).
        constexpr int kPer = (kBM * 8 * NT + 31) / 32;  // outputs per lane at most
        float yold[kPer];
        if (c > 0) {
#pragma unroll
          for (int j = 0; j < kPer; ++j) {
            const int idx = lane + 32 * j;
            const int n = idx / kBM, row = tile * kBM + idx % kBM;
            yold[j] = (idx < kBM * Nt && live && row < M) ? Y[xrow(n) * M + row] : 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int idx = lane + 32 * j;
          if (idx >= kBM * Nt) break;
          const int n = idx / kBM, r = idx % kBM;
          const int row = tile * kBM + r;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < KW; ++w) v += *reinterpret_cast<volatile float*>(&as[(w * Nt + n) * kBM + r]);
          if (live && row < M) Y[xrow(n) * M + row] = (c == 0) ? v : (yold[j] + v);
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          slot_count[aslot] = 0;
        }
      }
    }
    };
    if (xwide)
      run_tiles(std::true_type{});
    else
      run_tiles(std::false_type{});
  }
}

int g_early_stages = 2;  // W stages a launch may stream before the dependency (capped by the ring)
int decode_early_stages() { return g_early_stages; }
int g_x_static = 0;      // the caller promises X is not written by the kernel right before
int decode_x_static() { return g_x_static; }

template <int NT, int MT, int KW, int STAGES, bool ONE = false, bool MOE = false, int F = GQ_TYPE_Q4_0>
cudaError_t launch_cfg(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int N, int M, int K, float* Y,
                       uint64_t limit_ns, int xs_budget, int early_w, int pdl, cudaStream_t s,
                       const MoeRoute& rt = MoeRoute{}, int64_t max_groups = 0) {
  // MUL_MAT_ID needs the routing before it knows which weights to stream
  const int early_stages = (early_w && !MOE) ? std::max(1, std::min(STAGES, decode_early_stages())) : 0;
  using Cfg = DecodeCfg<NT, MT, KW, STAGES, F>;
  // Every box lands in a ring slot of kBM rows x kRowBytes: a tensor map
  // encoded with another box would overrun the slots, so it is refused.
  if (box.rows != static_cast<uint32_t>(Cfg::kBM) || box.row_bytes != static_cast<uint32_t>(Cfg::kRowBytes))
    return cudaErrorInvalidValue;
  // x chunk: a multiple of the stage width, as long as the budget allows
  int KX = (xs_budget / (2 * N)) / Cfg::kStageK * Cfg::kStageK;
  if (KX < Cfg::kStageK) KX = Cfg::kStageK;
  const int Kpad = (K + Cfg::kStageK - 1) / Cfg::kStageK * Cfg::kStageK;
  if (KX > Kpad) KX = Kpad;
  const size_t smem = Cfg::smem_bytes(N, KX);
  auto kern = k_decode_q4_0<NT, MT, KW, STAGES, ONE, MOE, F>;
  cudaError_t e = kernel_smem(reinterpret_cast<const void*>(kern), smem, true);
  if (e != cudaSuccess) return e;
  int occ_cache = 1;
  e = kernel_occupancy(reinterpret_cast<const void*>(kern), Cfg::kThreads, smem, &occ_cache);
  if (e != cudaSuccess) return e;
  const int ntiles = (M + Cfg::kBM - 1) / Cfg::kBM;
  // Small CTAs (two fit on an SM) run one per SM, so that the next launch's
  // CTA can share the SM and overlap this one.
  const int per_sm = (KW <= 4) ? 1 : occ_cache;
  const int64_t work = MOE ? ntiles * max_groups : ntiles;
  const int grid = static_cast<int>(std::min<int64_t>(work, static_cast<int64_t>(device_info().sm_count) * per_sm));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, *tmW, X, N, M, K, KX, Y, limit_ns, device_error_word(), early_stages,
                            MOE ? 0 : decode_x_static(), rt, test_drop() == 1 ? 1 : 0);
}

// -------------------------------------------------------------------------
// Generic fallback: any K % 32 == 0, any alignment, any N.  One warp per row;
// W bytes are re-read per token (from cache).  Used for shapes the fast paths
// do not take (K % 256 != 0, unaligned pointers).
__global__ void k_generic_q4_0(const uint8_t* __restrict__ W, int64_t M, int64_t K, const float* __restrict__ X,
                               int64_t N, float* __restrict__ Y) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / kQK;
  const int64_t row_bytes = nb * kBlockBytes;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t m = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint8_t* row = W + m * row_bytes;
    for (int64_t n = 0; n < N; ++n) {
      const float* x = X + n * K;
      float acc = 0.f;
      for (int64_t b = lane; b < nb; b += 32) {
        const uint8_t* blk = row + b * kBlockBytes;
        const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(blk[0] | (blk[1] << 8))));
        float part = 0.f;
        for (int j = 0; j < 16; ++j) {
          const uint32_t byte = blk[2 + j];
          part = fmaf(static_cast<float>(static_cast<int>(byte & 0xF) - 8), x[b * kQK + j], part);
          part = fmaf(static_cast<float>(static_cast<int>(byte >> 4) - 8), x[b * kQK + j + 16], part);
        }
        acc = fmaf(d, part, acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (lane == 0) Y[n * M + m] = acc;
    }
  }
}

}  // namespace

// Decode configuration by N: (NT, MT, KW, STAGES).  The variant index can be
// overridden for tuning (GQ_OPT_DECODE_VARIANT); 0 = default.
int decode_rows_per_tile(int64_t N, int variant) {
  if (N == 1) return variant == 1 ? 16 : (variant == 2 ? 64 : 32);
  if (N <= 8) return (variant == 2) ? 16 : 32;
  if (N <= 16) return (variant == 1 || variant == 4) ? 16 : 32;
  if (N <= 32) return variant == 2 ? 32 : 16;
  return 16;
}

void decode_w_box(int64_t N, int variant, uint32_t* box_x_bytes, uint32_t* box_rows) {
  *box_x_bytes = kSubBytesRow;
  *box_rows = static_cast<uint32_t>(decode_rows_per_tile(N, variant));
}

void set_decode_early_stages(int n) { g_early_stages = n; }
void set_decode_x_static(int on) { g_x_static = on ? 1 : 0; }
int get_decode_x_static() { return g_x_static; }
int get_decode_early_stages() { return g_early_stages; }

cudaError_t launch_decode(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int64_t N, int64_t M, int64_t K, float* Y,
                          uint64_t wait_limit_ns, int early_w, int variant, int pdl, cudaStream_t s) {
  const int n = static_cast<int>(N), m = static_cast<int>(M), k = static_cast<int>(K);
  if (N == 1) {
    if (variant == 1) return launch_cfg<1, 1, 16, 4, true>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    if (variant == 2) return launch_cfg<1, 4, 8, 2, true>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    if (variant == 3) return launch_cfg<1, 2, 8, 2, true>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    if (variant == 4) return launch_cfg<1, 2, 4, 3, true>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    // By default, when consecutive launches may overlap (X and W not written by
    // the previous kernel), the small 4-warp CTA lets the next launch's CTA
    // share the SM.  Measured over the 7B-like layer sequence this beats the
    // 8-warp CTA by ~19 % even for 11008-row matrices (2.3 tiles per SM), which
    // alone run faster on the 8-warp CTA; from 4 tiles per SM on (e.g. the
    // 32000-row output projection) the 8-warp CTA stays.
    if (variant == 0 && early_w && decode_x_static() && (m + 31) / 32 <= 4 * device_info().sm_count)
      return launch_cfg<1, 2, 4, 3, true>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    return launch_cfg<1, 2, 8, 3, true>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
  }
  if (N <= 8) {
    if (variant == 2) return launch_cfg<1, 1, 8, 4>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    // The co-resident 4-warp CTA, as for N = 1, where it measured faster when
    // repeated: up to 4 tokens and one 32-row tile per SM (4096 x 4096: 2
    // tokens 4.95 -> 3.82 us, 4 tokens 6.23 -> 4.86 us); with 8 tokens, or
    // 11008 rows and 2 tokens, the 8-warp CTA was faster.
    if (variant == 0 && N <= 4 && early_w && decode_x_static() && (m + 31) / 32 <= device_info().sm_count)
      return launch_cfg<1, 2, 4, 3>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    return launch_cfg<1, 2, 8, 3>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
  }
  if (N <= 16) {
    if (variant == 1) return launch_cfg<2, 1, 8, 3>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    if (variant == 2) return launch_cfg<2, 2, 4, 3>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
    if (variant == 3) return launch_cfg<2, 2, 4, 2>(tmW, box, X, n, m, k, Y, wait_limit_ns, 128 << 10, early_w, pdl, s);
    if (variant == 4) return launch_cfg<2, 1, 4, 4>(tmW, box, X, n, m, k, Y, wait_limit_ns, 128 << 10, early_w, pdl, s);
    return launch_cfg<2, 2, 8, 2>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
  }
  if (N <= 32) {
    if (variant == 1) return launch_cfg<4, 1, 4, 4>(tmW, box, X, n, m, k, Y, wait_limit_ns, 128 << 10, early_w, pdl, s);
    if (variant == 2) return launch_cfg<4, 2, 4, 2>(tmW, box, X, n, m, k, Y, wait_limit_ns, 128 << 10, early_w, pdl, s);
    if (variant == 3) return launch_cfg<4, 1, 8, 2>(tmW, box, X, n, m, k, Y, wait_limit_ns, 128 << 10, early_w, pdl, s);
    return launch_cfg<4, 1, 4, 4>(tmW, box, X, n, m, k, Y, wait_limit_ns, 96 << 10, early_w, pdl, s);
  }
  // N = 33..64: two k-warps, so that a stage's x (2 * 512 * N bytes) and the
  // partial sums fit in shared memory next to the ring
  return launch_cfg<8, 1, 2, 4>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
}

// MUL_MAT_ID group capacity: one token for a single-token batch (its slots
// pick distinct experts, so every group holds one token and the N = 1 kernel
// runs), else room for twice the mean tokens per used expert (an expert with
// more tokens than that runs as several groups).
int decode_moe_cap(int64_t P, int64_t E, int64_t T) {
  if (T == 1) return 1;
  const int64_t used = std::max<int64_t>(1, std::min(E, P));
  const int64_t want = 2 * ((P + used - 1) / used);
  return want <= 8 ? 8 : want <= 16 ? 16 : want <= 32 ? 32 : 64;
}

void decode_moe_w_box(int cap, uint32_t* box_x_bytes, uint32_t* box_rows) {
  *box_x_bytes = kSubBytesRow;
  *box_rows = cap <= 16 ? 32u : 16u;
}

cudaError_t launch_decode_moe(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int cap, int64_t E, int64_t M, int64_t K,
                              int64_t P, const MoeRoute& rt, float* Y, uint64_t wait_limit_ns, int pdl,
                              cudaStream_t s) {
  const int m = static_cast<int>(M), k = static_cast<int>(K);
  const int64_t max_groups = std::min(E, P) + P / cap + 1;
  if (cap == 1)
    return launch_cfg<1, 2, 8, 3, true, true>(tmW, box, X, 1, m, k, Y, wait_limit_ns, 64 << 10, 0, pdl, s, rt, max_groups);
  if (cap == 8)
    return launch_cfg<1, 2, 8, 3, false, true>(tmW, box, X, 8, m, k, Y, wait_limit_ns, 64 << 10, 0, pdl, s, rt, max_groups);
  if (cap == 16)
    return launch_cfg<2, 2, 8, 2, false, true>(tmW, box, X, 16, m, k, Y, wait_limit_ns, 64 << 10, 0, pdl, s, rt, max_groups);
  if (cap == 32)
    return launch_cfg<4, 1, 4, 4, false, true>(tmW, box, X, 32, m, k, Y, wait_limit_ns, 96 << 10, 0, pdl, s, rt, max_groups);
  return launch_cfg<8, 1, 2, 4, false, true>(tmW, box, X, 64, m, k, Y, wait_limit_ns, 64 << 10, 0, pdl, s, rt, max_groups);
}

// Q4_1 / Q8_0 at N = 1: the decode kernel with 20- or 34-byte blocks (32-row
// tiles, 160- or 272-byte box rows); the 4-warp co-resident CTA under the same
// promises as Q4_0.
// Q8_0's stages are 1.9x Q4_0's: one stage fewer, so that the ring fits (the
// 8-warp CTA) and two 4-warp CTAs still share an SM.
template <int F>
cudaError_t launch_decode_fmt(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int64_t M, int64_t K, float* Y,
                              uint64_t wait_limit_ns, int early_w, int pdl, cudaStream_t s) {
  constexpr int kSt = F == GQ_TYPE_Q8_0 ? 2 : 3;
  const int m = static_cast<int>(M), k = static_cast<int>(K);
  if (early_w && decode_x_static() && (m + 31) / 32 <= 4 * device_info().sm_count)
    return launch_cfg<1, 2, 4, kSt, true, false, F>(tmW, box, X, 1, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
  return launch_cfg<1, 2, 8, kSt, true, false, F>(tmW, box, X, 1, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
}

// 2..15 tokens: 32-row tiles and two stages (the larger blocks' rings and the
// x fragments of up to 16 tokens must fit in shared memory beside each other).
template <int F>
cudaError_t launch_decode_fmt_n(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int64_t N, int64_t M, int64_t K, float* Y,
                                uint64_t wait_limit_ns, int early_w, int pdl, cudaStream_t s) {
  constexpr int kKw = F == GQ_TYPE_Q8_0 ? 4 : 8;
  const int n = static_cast<int>(N), m = static_cast<int>(M), k = static_cast<int>(K);
  if (N <= 8)
    return launch_cfg<1, 2, kKw, 2, false, false, F>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
  return launch_cfg<2, 2, kKw, 2, false, false, F>(tmW, box, X, n, m, k, Y, wait_limit_ns, 64 << 10, early_w, pdl, s);
}

cudaError_t launch_decode_legacy(int type, const CUtensorMap* tmW, const DecodeBox& box, const float* X, int64_t N, int64_t M, int64_t K,
                                 float* Y, uint64_t wait_limit_ns, int early_w, int pdl, cudaStream_t s) {
  if (type == GQ_TYPE_Q4_K)
    return N == 1 ? launch_decode_fmt<GQ_TYPE_Q4_K>(tmW, box, X, M, K, Y, wait_limit_ns, early_w, pdl, s)
                  : launch_decode_fmt_n<GQ_TYPE_Q4_K>(tmW, box, X, N, M, K, Y, wait_limit_ns, early_w, pdl, s);
  if (type == GQ_TYPE_Q5_0)
    return N == 1 ? launch_decode_fmt<GQ_TYPE_Q5_0>(tmW, box, X, M, K, Y, wait_limit_ns, early_w, pdl, s)
                  : launch_decode_fmt_n<GQ_TYPE_Q5_0>(tmW, box, X, N, M, K, Y, wait_limit_ns, early_w, pdl, s);
  if (type == GQ_TYPE_Q5_1)
    return N == 1 ? launch_decode_fmt<GQ_TYPE_Q5_1>(tmW, box, X, M, K, Y, wait_limit_ns, early_w, pdl, s)
                  : launch_decode_fmt_n<GQ_TYPE_Q5_1>(tmW, box, X, N, M, K, Y, wait_limit_ns, early_w, pdl, s);
  if (type == GQ_TYPE_Q8_0)
    return N == 1 ? launch_decode_fmt<GQ_TYPE_Q8_0>(tmW, box, X, M, K, Y, wait_limit_ns, early_w, pdl, s)
                  : launch_decode_fmt_n<GQ_TYPE_Q8_0>(tmW, box, X, N, M, K, Y, wait_limit_ns, early_w, pdl, s);
  return N == 1 ? launch_decode_fmt<GQ_TYPE_Q4_1>(tmW, box, X, M, K, Y, wait_limit_ns, early_w, pdl, s)
                : launch_decode_fmt_n<GQ_TYPE_Q4_1>(tmW, box, X, N, M, K, Y, wait_limit_ns, early_w, pdl, s);
}

cudaError_t launch_generic(const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                           cudaStream_t s) {
  const int64_t blocks = (M + 7) / 8;
  const int grid = static_cast<int>(std::min<int64_t>(blocks, static_cast<int64_t>(device_info().sm_count) * 16));
  k_generic_q4_0<<<grid, 256, 0, s>>>(W, M, K, X, N, Y);
  return cudaGetLastError();
}

}  // namespace gq
