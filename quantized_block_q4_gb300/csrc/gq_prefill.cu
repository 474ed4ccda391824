// K0: fp32 -> bf16 conversion of the activations, and K3: the prefill
// MUL_MAT against Q4_0 weights on tcgen05 tensor cores.
//
// K3 computes Y[n][m] = sum_k w[m][k] * x[n][k] for a 128-row x BN-token tile
// per CTA ("GGUF loading, mmap and tensor placement", step six: the MUL_MAT
// probe with a 512-token batch; "Binding GGUF weights to the compute graph",
// section 2.3: the kernel reads the blocks and dequantises them itself).
// Roles (608 threads):
//   warp 0  TMA producer of raw W rows (128 x 144 bytes = 256 weights each)
//           into a shared-memory ring; it runs ahead of the x producer by
//           up to the ring depth (12 steps of 64 k), which hides HBM latency.
//   warp 18 TMA producer of bf16 x tiles (BN x 64, 128-byte swizzle).
//   warp 1  allocates 512 TMEM columns: the fp32 accumulator (BN columns) and
//           a ring of A stages (32 columns = 64 bf16 k each).  One thread
//           issues tcgen05.mma with A read from tensor memory and B (x) from
//           shared memory (M=128, N=BN, K=16, bf16 x bf16 -> fp32) and
//           commits to the rings' "empty" barriers.
//   warps 2-17 dequantise in four groups of four warps: group g takes the
//           64-k step g of every 256-k chunk; a thread owns one W row of the
//           tile, i.e. one TMEM lane, and stores RN_bf16(d*(q-8)) for the
//           step's 64 weights into its lane with one tcgen05.st.  Then they
//           read the accumulator with tcgen05.ld (warp w reads TMEM lanes
//           32*(w%4)..; group g takes a quarter of the columns) and store
//           fp32 Y, consecutive lanes writing consecutive m.
// Work split: a CTA runs a contiguous range of (tile, 256-k chunk) units,
// possibly several tiles (stream-K, PrefillWork below); the rings and the
// accumulator hand-off carry over from one tile to the next.
// Dequantisation to bf16 with a single rounding, in bf16x2 arithmetic: the
// fp16 scale is split exactly as d = d_hi + d_lo (both bf16; d_lo holds the
// last 3 bits), q - 8 is formed exactly as (128 + q) - 136 from the bit
// pattern 0x4300 | q, q'*d_lo is exact in bf16, and one fused
// fma.rn.bf16x2(q', d_hi, q'*d_lo) rounds d*(q-8) once.
// Every wait is bounded; a timeout sets the device error word, the roles
// drain what they issued, TMEM is released and the CTA exits.
// Launched with programmatic dependent launch (K0 too): the next launch's
// CTAs take each SM as this one's CTA there leaves, and every role waits for
// the kernel before ahead of its first global access (W may stream a few
// chunks early when the caller promises the weights are not being written).
#include <algorithm>
#include <atomic>
#include <random>
#include <cuda_bf16.h>

#include "gq_internal.h"
#include "gq_ptx.cuh"
#include "gq_q4k.cuh"

namespace gq {
namespace {

// 8 elements per thread per step: two float4 loads, one 16-byte store.  Under
// programmatic dependent launch it waits for the kernel before (which may
// have written x, or may still read y) before touching memory.
__global__ void k_f32_to_bf16(const float* __restrict__ x, uint16_t* __restrict__ y, int64_t n) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) == 0;
  if (vec) {
    const int64_t n8 = n / 8;
    for (int64_t i = i0; i < n8; i += stride) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(x) + 2 * i);
      const float4 b = __ldg(reinterpret_cast<const float4*>(x) + 2 * i + 1);
      __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
      uint4 o;
      o.x = *reinterpret_cast<uint32_t*>(&p0);
      o.y = *reinterpret_cast<uint32_t*>(&p1);
      o.z = *reinterpret_cast<uint32_t*>(&p2);
      o.w = *reinterpret_cast<uint32_t*>(&p3);
      reinterpret_cast<uint4*>(y)[i] = o;
    }
    for (int64_t i = n8 * 8 + i0; i < n; i += stride) {
      __nv_bfloat16 h = __float2bfloat16_rn(x[i]);
      y[i] = *reinterpret_cast<uint16_t*>(&h);
    }
  } else {
    for (int64_t i = i0; i < n; i += stride) {
      __nv_bfloat16 h = __float2bfloat16_rn(x[i]);
      y[i] = *reinterpret_cast<uint16_t*>(&h);
    }
  }
}

}  // namespace

cudaError_t launch_f32_to_bf16(const float* x, uint16_t* y, int64_t n, cudaStream_t s, int pdl) {
  const int64_t work = (n + 7) / 8;
  const int grid =
      static_cast<int>(std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(device_info().sm_count) * 8));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_f32_to_bf16, x, y, n);
}

namespace {

// F: block format of W (GQ_TYPE_*).  Q4_0 blocks are 18 bytes, Q4_1 20,
// Q8_0 34; a raw stage holds 8 blocks (256 k) of each of the 128 rows.  A Q4_K
// super-block is itself 256 k in 144 bytes (18 bytes per 32 weights).
template <int F>
constexpr int fmt_block_bytes() {
  return (F == GQ_TYPE_Q4_0 || F == GQ_TYPE_Q4_K) ? 18
         : F == GQ_TYPE_Q4_1                      ? 20
         : F == GQ_TYPE_Q5_0                      ? 22
         : F == GQ_TYPE_Q5_1                      ? 24
                                                  : 34;
}

template <int BN, bool PAIR, int F = GQ_TYPE_Q4_0>
struct PrefillCfg {
  static constexpr int kBM = 128;       // W rows per CTA (a CTA pair covers 256)
  static constexpr int kBK = 64;        // k per MMA stage: one 128-byte row of bf16
  static constexpr int kRawK = 256;     // k per raw W stage (one work unit)
  static constexpr int kBlk = fmt_block_bytes<F>();
  static constexpr int kRawRow = 8 * kBlk;   // bytes of 8 blocks: 144, 160 or 272
  // The TMA box is at most 256 elements wide: Q8_0's 272-byte rows are read
  // as 136 16-bit elements.
  static constexpr int kRawElem = kRawRow > 256 ? 2 : 1;
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int kXRows = BN / kCtas;            // x rows (tokens) this CTA loads per stage
  static constexpr int kACols = kBK / 2;               // TMEM columns per A stage
  // One ring of S stages, each an A tile in TMEM (64 k of the 128 rows) and
  // an x tile in shared memory; the accumulator takes the first BN columns.
  // The larger raw stages of Q4_1 / Q8_0 leave room for fewer x stages.
  static constexpr int RS = F == GQ_TYPE_Q8_0 ? 2 : 3;
  static constexpr int S = PAIR ? 8 : (BN == 256 ? (kRawRow == 144 ? 5 : 4) : 8);
  static_assert(BN + S * kACols <= 512, "TMEM holds the accumulator and the A stages");
  // Step c of the ring goes to stage c mod S and is written by dequant group
  // c mod 4, which waits on the stage's "empty" barrier by phase parity.  With
  // S >= 4 that group's own previous step (c - 4) already needed the MMA of
  // step c - 4 - S, and MMAs complete in order, so the barrier is at most one
  // phase behind and the parity is unambiguous.  With fewer stages than
  // groups it can be two phases behind: the wait passes early and the group
  // overwrites an A stage that an MMA still reads.
  static_assert(S >= 4, "an A/x stage ring shorter than the four dequant groups lets a parity wait pass early");
  static constexpr int kTmemCols = 512;
  static constexpr int kRawBytes = kBM * kRawRow;  // 18432 for Q4_0
  // 16-byte words a dequantising thread loads to cover its two blocks (Q4_K:
  // the super-block's 16-byte header and the 32 code bytes of its step; Q5_0:
  // 44 bytes from an offset of up to 12 into the first word)
  static constexpr int kWinWords = F == GQ_TYPE_Q8_0 ? 5 : (F == GQ_TYPE_Q5_0 ? 4 : 3);
  static constexpr int kBBytes = kXRows * 128;
  static constexpr int kOffB = 0;
  static constexpr int kOffRaw = kOffB + S * kBBytes;
  static constexpr int kOffBar = kOffRaw + RS * kRawBytes;
  static constexpr int kNBar = 2 * RS + 2 * S + 2;
  static constexpr int kOffTmem = kOffBar + kNBar * 8;
  static constexpr int kOffAbort = kOffTmem + 8;
  static constexpr int kOffFlag = kOffAbort + 8;       // two words: "this CTA reduces the tile"
  static constexpr int kSmem = kOffFlag + 8 + 1024;   // + slack to align the base to 1024
  static constexpr int kDeqWarps = 16;  // warps 2..17, 4 groups of 4: one 64-k step of each 256-k chunk per group
  static constexpr int kXWarp = 2 + kDeqWarps;  // warp 0 loads W, warp 1 issues MMAs, the last warp loads x
  static constexpr int kThreads = 32 * (3 + kDeqWarps);
  static constexpr int kSlotFloats = BN * kBM;         // one CTA's partial tile, [column][row]
  static_assert(kSmem <= 216 * 1024, "shared memory budget (the Q4_0 BN = 256 ring uses 215 KB)");
};

// Work schedule of a launch over G work ranges (one CTA, or one CTA pair,
// each; G <= the SMs or pairs, so every range runs at once):
//   * tiles [R, T) are whole tiles, dealt round-robin: range g runs tiles
//     R + g, R + g + G, ... (persistent: the rings and the accumulator
//     hand-off carry over from one tile to the next);
//   * tiles [0, R) are each split into s pieces along k (256-k chunks
//     [p*nr/s, (p+1)*nr/s)); piece p of tile t is the first segment of range
//     t*s + p.  The pieces' partial sums meet in a workspace and the range that
//     finds all the others published adds them, in k order.
// R = 0 is the plain one-tile-per-CTA split when T <= G.
struct PrefillWork {
  int64_t T;      // output tiles; tile t = (row block t / ntn, token block t % ntn)
  int64_t G;      // work ranges
  int nr;         // 256-k chunks per tile, K / 256
  int ntn;        // token tiles per row block
  int R, s;       // split tiles and pieces per split tile
  float* ws;      // one partial-tile slot per piece and CTA (nullptr when R == 0)
  unsigned long long* count;  // per split tile and CTA of a pair: (epoch << 8) | pieces published
  unsigned long long epoch;   // this launch's tag (< 2^56): a counter with another tag reads as 0
  int early_w;    // W is not written by the kernels before: its first chunks may stream before the PDL wait
  int x_static;   // X is not written by the kernels that may still run: only Y (and scratch) wait for the kernel before
  int drop;       // test hook (GQ_OPT_TEST_DROP_ARRIVE): raw chunk 1 of CTA 0 is never issued
};

// Arrival counters need no zeroing between launches: a counter whose tag is
// not this launch's epoch counts as zero pieces.
__device__ __forceinline__ int pieces_published(unsigned long long v, unsigned long long epoch) {
  return (v >> 8) == epoch ? static_cast<int>(v & 0xFF) : 0;
}

// Count one more published piece; returns how many were published before it
// (-1 if the update kept failing, which only heavy contention could cause).
__device__ __forceinline__ int publish_piece(unsigned long long* count, unsigned long long epoch) {
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(count);
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const int before = pieces_published(cur, epoch);
    const unsigned long long want = (epoch << 8) | static_cast<unsigned long long>(before + 1);
    const unsigned long long seen = atomicCAS(count, cur, want);
    if (seen == cur) return before;
    cur = seen;
  }
  return -1;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

struct Seg {
  int64_t t;   // tile
  int r0, r1;  // chunk range [r0, r1) of the tile
};

__device__ __forceinline__ int seg_count(int g, const PrefillWork& wk) {
  const int64_t full = wk.T - wk.R;
  const int64_t nfull = full > g ? (full - g + wk.G - 1) / wk.G : 0;
  return (g < static_cast<int64_t>(wk.R) * wk.s ? 1 : 0) + static_cast<int>(nfull);
}

__device__ __forceinline__ Seg seg_of(int g, int i, const PrefillWork& wk) {
  Seg sg;
  if (g < static_cast<int64_t>(wk.R) * wk.s) {
    if (i == 0) {
      const int p = g % wk.s;
      sg.t = g / wk.s;
      sg.r0 = p * wk.nr / wk.s;
      sg.r1 = (p + 1) * wk.nr / wk.s;
      return sg;
    }
    --i;
  }
  sg.t = wk.R + g + static_cast<int64_t>(i) * wk.G;
  sg.r0 = 0;
  sg.r1 = wk.nr;
  return sg;
}

// MUL_MAT_ID work item w (items run in (expert, 128-row tile, BN-token tile)
// order, so the token tiles of one weight tile run side by side and share it
// in L2): the expert is the last e with item_start[e] <= w.
struct MoeItem {
  int wrow;    // first W row among all experts' rows (TMA y)
  int mrow0;   // first output row within the expert
  int xrow;    // first gathered x row (sorted position) of the tile
  int nvalid;  // tokens in the tile (1..BN)
};

__device__ __forceinline__ MoeItem moe_item(int w, const MoeRoute& rt, int E, int Mexp, int bn) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(rt.item_start + mid) <= w) lo = mid; else hi = mid - 1;
  }
  const int local = w - __ldg(rt.item_start + lo);
  const int first = __ldg(rt.off + lo), cnt = __ldg(rt.off + lo + 1) - first;
  const int ntn = (cnt + bn - 1) / bn;
  const int im = local / ntn, j = local - im * ntn;
  MoeItem it;
  it.mrow0 = im * 128;
  it.wrow = lo * Mexp + it.mrow0;
  it.xrow = first + j * bn;
  it.nvalid = min(bn, cnt - j * bn);
  return it;
}

__device__ __forceinline__ uint32_t scale_pair(uint32_t qp, uint32_t dhi2, uint32_t dlo2) {
  return bfma2_u32(qp, dhi2, bmul2_u32(qp, dlo2));
}

// Four consecutive code bytes c0..c3 -> bf16x2 pairs of RN(d*(q-8)):
// lo01 = (c0.lo, c1.lo), lo23 = (c2.lo, c3.lo), hi01 = (c0.hi, c1.hi), hi23 = (c2.hi, c3.hi).
__device__ __forceinline__ void word_to_bf16(uint32_t q, uint32_t dhi2, uint32_t dlo2, uint32_t& lo01,
                                             uint32_t& lo23, uint32_t& hi01, uint32_t& hi23) {
  const uint32_t kMagic = 0x43004300u;  // bf16 128 in both halves
  const uint32_t kSub = 0x43084308u;    // bf16 136
  const uint32_t p = prmt(q, 0u, 0x3120u);  // bytes c0 c2 c1 c3
  lo01 = scale_pair(bsub2_u32(lop3_and_or(p, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
  lo23 = scale_pair(bsub2_u32(lop3_and_or(p >> 8, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
  hi01 = scale_pair(bsub2_u32(lop3_and_or(p >> 4, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
  hi23 = scale_pair(bsub2_u32(lop3_and_or(p >> 12, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
}

// Exact split of an fp16 scale into bf16 d_hi + d_lo, each broadcast to both halves.
__device__ __forceinline__ void split_scale(uint32_t d_bits, uint32_t& dhi2, uint32_t& dlo2) {
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(d_bits)));
  const __nv_bfloat16 hi = __float2bfloat16_rn(d);
  const __nv_bfloat16 lo = __float2bfloat16_rn(d - __bfloat162float(hi));  // exact: at most 3 bits remain
  const uint32_t h = *reinterpret_cast<const uint16_t*>(&hi), l = *reinterpret_cast<const uint16_t*>(&lo);
  dhi2 = h | (h << 16);
  dlo2 = l | (l << 16);
}

// One block's 16 code bytes (4 words, k-consecutive) -> 16 bf16x2 words
// holding k = 0..31 of the block in order (o[i] = k 2i, 2i+1).
__device__ __forceinline__ void block_words(const uint32_t (&q)[4], uint32_t d_bits, uint32_t* o) {
  uint32_t dhi2, dlo2;
  split_scale(d_bits, dhi2, dlo2);
  // low nibbles of bytes 0..15 are k 0..15, high nibbles are k 16..31
  word_to_bf16(q[0], dhi2, dlo2, o[0], o[1], o[8], o[9]);
  word_to_bf16(q[1], dhi2, dlo2, o[2], o[3], o[10], o[11]);
  word_to_bf16(q[2], dhi2, dlo2, o[4], o[5], o[12], o[13]);
  word_to_bf16(q[3], dhi2, dlo2, o[6], o[7], o[14], o[15]);
}

// Byte j (a constant) of q as an exact fp32 integer: one byte permute builds
// the float 2^23 + byte, one subtraction removes 2^23.
template <int J>
__device__ __forceinline__ float byte_f(uint32_t q) {
  return __uint_as_float(prmt(q, 0x4B000000u, 0x7650u | J)) - 8388608.0f;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Q4_1 and Q8_0 steps: elements as fp32 (d*q exact; Q4_1 then adds m with
// one rounding), rounded once more to bf16 in pairs (element 2i in the low
// half of o[i], as for Q4_0).

// One Q4_1 block: h = d | m << 16, c[4] = the 16 code bytes.
__device__ __forceinline__ void q41_block(uint32_t h, const uint32_t (&c)[4], uint32_t* o) {
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(h & 0xFFFF)));
  const float m = __half2float(__ushort_as_half(static_cast<uint16_t>(h >> 16)));
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float lo[4], hi[4];
    const uint32_t ql = c[w] & 0x0F0F0F0Fu, qhi = (c[w] >> 4) & 0x0F0F0F0Fu;
    // d*q is exact, so one fused multiply-add rounds d*q + m once
    lo[0] = __fmaf_rn(d, byte_f<0>(ql), m); hi[0] = __fmaf_rn(d, byte_f<0>(qhi), m);
    lo[1] = __fmaf_rn(d, byte_f<1>(ql), m); hi[1] = __fmaf_rn(d, byte_f<1>(qhi), m);
    lo[2] = __fmaf_rn(d, byte_f<2>(ql), m); hi[2] = __fmaf_rn(d, byte_f<2>(qhi), m);
    lo[3] = __fmaf_rn(d, byte_f<3>(ql), m); hi[3] = __fmaf_rn(d, byte_f<3>(qhi), m);
    o[2 * w] = pack_bf16(lo[0], lo[1]);
    o[2 * w + 1] = pack_bf16(lo[2], lo[3]);
    o[8 + 2 * w] = pack_bf16(hi[0], hi[1]);
    o[8 + 2 * w + 1] = pack_bf16(hi[2], hi[3]);
  }
}

// One Q8_0 block: d bits, c[8] = the 32 code bytes (two's complement; c ^
// 0x80 is the code + 128).
__device__ __forceinline__ void q80_block(uint32_t d_bits, const uint32_t (&c)[8], uint32_t* o) {
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(d_bits)));
  const float off = -128.0f * d;  // exact
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t u = c[w] ^ 0x80808080u;  // code + 128 in each byte
    float e[4];
    // d*(u - 128) = d*u - 128d, every term exact: one fused multiply-add
    e[0] = __fmaf_rn(d, byte_f<0>(u), off);
    e[1] = __fmaf_rn(d, byte_f<1>(u), off);
    e[2] = __fmaf_rn(d, byte_f<2>(u), off);
    e[3] = __fmaf_rn(d, byte_f<3>(u), off);
    o[2 * w] = pack_bf16(e[0], e[1]);
    o[2 * w + 1] = pack_bf16(e[2], e[3]);
  }
}

// Q4_K step G of a super-block row: sub-blocks 2G (the low nibbles of code
// bytes 32G .. 32G+31, k 0..31 of the step) and 2G+1 (their high nibbles, k
// 32..63).  v[0..3]: the header (d | dmin << 16 and the field words F0, F1,
// F2); v[4..11]: the 32 code bytes.  Elements in fp32 (d*sc*q exact, the min
// subtracted with one rounding), then rounded to bf16 in pairs.
template <int G>
__device__ __forceinline__ void q4k_step_words(const uint32_t* v, uint32_t* o) {
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(v[0] & 0xFFFF)));
  const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(v[0] >> 16)));
  uint32_t sc0, m0, sc1, m1;
  q4k_scale_min<2 * G>(v[1], v[2], v[3], sc0, m0);
  q4k_scale_min<2 * G + 1>(v[1], v[2], v[3], sc1, m1);
  const float d0 = d * static_cast<float>(sc0), mn0 = dmin * static_cast<float>(m0);
  const float d1 = d * static_cast<float>(sc1), mn1 = dmin * static_cast<float>(m1);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t c = v[4 + w];  // code bytes 4w .. 4w+3
    const uint32_t ql = c & 0x0F0F0F0Fu, qhi = (c >> 4) & 0x0F0F0F0Fu;
    float lo[4], hi[4];
    lo[0] = __fmaf_rn(d0, byte_f<0>(ql), -mn0); hi[0] = __fmaf_rn(d1, byte_f<0>(qhi), -mn1);
    lo[1] = __fmaf_rn(d0, byte_f<1>(ql), -mn0); hi[1] = __fmaf_rn(d1, byte_f<1>(qhi), -mn1);
    lo[2] = __fmaf_rn(d0, byte_f<2>(ql), -mn0); hi[2] = __fmaf_rn(d1, byte_f<2>(qhi), -mn1);
    lo[3] = __fmaf_rn(d0, byte_f<3>(ql), -mn0); hi[3] = __fmaf_rn(d1, byte_f<3>(qhi), -mn1);
    o[2 * w] = pack_bf16(lo[0], lo[1]);
    o[2 * w + 1] = pack_bf16(lo[2], lo[3]);
    o[16 + 2 * w] = pack_bf16(hi[0], hi[1]);
    o[16 + 2 * w + 1] = pack_bf16(hi[2], hi[3]);
  }
}

// The 32-bit little-endian value at byte offset B (a constant) of the window v.
template <int B>
__device__ __forceinline__ uint32_t win_word(const uint32_t* v) {
  if constexpr (B % 4 == 0) return v[B / 4];
  else return __funnelshift_r(v[B / 4], v[B / 4 + 1], 8 * (B % 4));
}

// Bits 0-3 of b to bit 0 of bytes 0-3 (the four products b_i * 2^(7j) land
// on distinct bits, so the multiply carries nothing into the mask).
__device__ __forceinline__ uint32_t spread4(uint32_t b) { return (b * 0x00204081u) & 0x01010101u; }

// One Q5_0 / Q5_1 block at byte offset B of the window: 32 elements w =
// d*(q - 16) (exact in fp32: d*q and 16d are) or d*q + m (d*q exact, one
// rounding), rounded to bf16 in pairs (o[i] = elements 2i, 2i+1).  Per code
// word: four 5-bit codes (nibbles with their high bits at bit 4 of each byte),
// each byte made an fp32 2^23 + q by one byte permute.
template <int F, int B>
__device__ __forceinline__ void q5_block_words(const uint32_t* v, uint32_t* o) {
  constexpr int qo = F == GQ_TYPE_Q5_1 ? 4 : 2;  // high-bit word, then 16 code bytes
  const uint32_t h = win_word<B>(v);
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(h & 0xFFFF)));
  const float add = F == GQ_TYPE_Q5_1 ? __half2float(__ushort_as_half(static_cast<uint16_t>(h >> 16))) : -16.0f * d;
  const uint32_t qh = win_word<B + qo>(v);
  const uint32_t cw[4] = {win_word<B + qo + 4>(v), win_word<B + qo + 8>(v), win_word<B + qo + 12>(v),
                          win_word<B + qo + 16>(v)};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t c = cw[w];
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // low nibbles: elements 4w.., high nibbles: 16 + 4w..
      const uint32_t q = ((half ? c >> 4 : c) & 0x0F0F0F0Fu) | (spread4((qh >> (16 * half + 4 * w)) & 0xFu) << 4);
      const float e[4] = {__fmaf_rn(d, byte_f<0>(q), add), __fmaf_rn(d, byte_f<1>(q), add),
                          __fmaf_rn(d, byte_f<2>(q), add), __fmaf_rn(d, byte_f<3>(q), add)};
      o[8 * half + 2 * w] = pack_bf16(e[0], e[1]);
      o[8 * half + 2 * w + 1] = pack_bf16(e[2], e[3]);
    }
  }
}

// Group G's two blocks of a 256-k chunk row from the loaded window v (the
// 16-byte words from byte (2*G*block bytes) & ~15 of the row; for Q4_K the
// header and the step's code bytes).
template <int F, int G>
__device__ __forceinline__ void step_words_fmt(const uint32_t* v, uint32_t* o) {
  if constexpr (F == GQ_TYPE_Q4_K) {
    q4k_step_words<G>(v, o);
  } else if constexpr (F == GQ_TYPE_Q5_0 || F == GQ_TYPE_Q5_1) {
    constexpr int bb = F == GQ_TYPE_Q5_0 ? 22 : 24;
    constexpr int b0 = (2 * G * bb) % 16;  // the group's first block within the window
    q5_block_words<F, b0>(v, o);
    q5_block_words<F, b0 + bb>(v, o + 16);
  } else if constexpr (F == GQ_TYPE_Q4_1) {
    constexpr int w0 = (40 * G % 16) / 4;  // 0, 2, 0, 2
    const uint32_t c0[4] = {v[w0 + 1], v[w0 + 2], v[w0 + 3], v[w0 + 4]};
    const uint32_t c1[4] = {v[w0 + 6], v[w0 + 7], v[w0 + 8], v[w0 + 9]};
    q41_block(v[w0], c0, o);
    q41_block(v[w0 + 5], c1, o + 16);
  } else {
    // 68*G mod 16 = 4G: block 0 starts at word G, block 1 at byte 4G + 34
    uint32_t c0[8], c1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      c0[k] = prmt(v[G + k], v[G + k + 1], 0x5432u);  // bytes 4G + 2 + 4k ..
      c1[k] = v[G + 9 + k];                            // bytes 4G + 36 + 4k ..
    }
    q80_block(v[G] & 0xFFFFu, c0, o);
    q80_block(v[G + 8] >> 16, c1, o + 16);
  }
}

// Bounded wait on the last phase issued into each slot of a ring (drain path).
__device__ __forceinline__ void drain_ring(uint64_t* full, int slots, uint32_t issued, uint64_t limit_ns) {
  for (int s = 0; s < slots; ++s) {
    if (static_cast<uint32_t>(s) >= issued) break;
    const uint32_t last = ((issued - 1 - s) / slots) * slots + s;  // largest index < issued in slot s
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&full[s]), (last / slots) & 1) && globaltimer_ns() - t0 < limit_ns) {
    }
  }
}

// MOE: MUL_MAT_ID over routed pairs (1-CTA tiles only).  M is then the rows of
// one expert, N is unused, the work items come from rt (item i of the launch
// goes to CTA i % gridDim.x) and x rows are loaded in 64-row boxes, only as
// many as the tile's tokens need.
template <int BN, bool PAIR, bool MOE = false, int F = GQ_TYPE_Q4_0>
__global__ void __launch_bounds__(PrefillCfg<BN, PAIR, F>::kThreads, 1)
    k_prefill_q4_0(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int N, int M,
                   float* __restrict__ Y, const PrefillWork wk, uint64_t limit_ns, uint32_t* err,
                   const MoeRoute rt, int E) {
  static_assert(!(MOE && PAIR), "MUL_MAT_ID uses the 1-CTA kernel");
  static_assert(!(MOE && F != GQ_TYPE_Q4_0), "MUL_MAT_ID takes Q4_0 weights");
  using C = PrefillCfg<BN, PAIR, F>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + C::RS;
  uint64_t* full = raw_empty + C::RS;   // stage holds A (dequant arrivals) and x (TMA bytes)
  uint64_t* empty = full + C::S;        // stage's MMAs have completed
  uint64_t* acc_full = empty + C::S;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  volatile int* reduce_flag = reinterpret_cast<volatile int*>(smem + C::kOffFlag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A pair shares one range of work units; its leader (rank 0) issues the MMAs.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int gi = static_cast<int>(blockIdx.x / C::kCtas);
  // Programmatic dependent launch.  MUL_MAT_ID: the routing tables and the
  // gathered x come from the kernels before, so every role waits first.
  // MUL_MAT: each role waits for the kernel before (which may have written x
  // or W, or may still read Y or this launch's scratch) before its first
  // access to global memory, or its first bounded wait on a role that does;
  // with early_w only the first raw W chunks stream before that.
  if (MOE) pdl_wait();
  const int nseg = MOE ? (rt.meta[0] > gi ? (rt.meta[0] - gi + static_cast<int>(gridDim.x) - 1) /
                                                 static_cast<int>(gridDim.x)
                                           : 0)
                       : seg_count(gi, wk);
  const int nr = wk.nr;
  // Barriers the leader's MMA thread waits on receive the arrivals of both CTAs.
  auto leader_bar = [&](uint64_t* bar) -> uint32_t { return PAIR ? mapa_shared(smem_u32(bar), 0) : smem_u32(bar); };
  auto arrive_leader = [&](uint64_t* bar) {
    if (PAIR)
      mbar_arrive_remote(leader_bar(bar));
    else
      mbar_arrive(smem_u32(bar));
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RS; ++i) {
      mbar_init(smem_u32(&raw_full[i]), 1);
      mbar_init(smem_u32(&raw_empty[i]), C::kDeqWarps);
    }
    for (int i = 0; i < C::S; ++i) {
      // the 4 dequant warps of the owning group in each CTA, plus the leader's
      // x producer (expect_tx); every x half completes its bytes on it
      mbar_init(smem_u32(&full[i]), 4 * C::kCtas + 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), C::kDeqWarps * C::kCtas);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The next kernel may launch once every CTA has signalled: at once with
  // x_static, else after this CTA's x producer has waited for the kernel
  // before, so that a later x-static launch cannot start before the kernels
  // ahead of this one are done.
  if (!MOE && wk.x_static) pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ W producer
    // The whole warp runs the loop (waits, bookkeeping) and one elected lane
    // issues; a converged warp issues TMA and tcgen05 work faster than a lone
    // lane of a diverged one.
    {
      const bool issuer = elect_one();
      if (issuer) tma_prefetch_desc(&tmW);
      uint32_t nraw = 0;
      // static W under an x-static launch: nothing of this producer waits for the kernel before
      bool ok = true, waited = MOE || (wk.early_w && wk.x_static);
      for (int i = 0; i < nseg && ok; ++i) {
        Seg sg;
        int m0;
        if constexpr (MOE) {
          m0 = moe_item(gi + i * static_cast<int>(gridDim.x), rt, E, M, BN).wrow;
          sg.r0 = 0;
          sg.r1 = nr;
        } else {
          sg = seg_of(gi, i, wk);
          m0 = static_cast<int>(sg.t / wk.ntn) * (C::kBM * C::kCtas) + static_cast<int>(rank) * C::kBM;
        }
        for (int r = sg.r0; r < sg.r1; ++r) {
          if (!waited && (!wk.early_w || nraw >= static_cast<uint32_t>(C::RS))) {
            pdl_wait();
            waited = true;
          }
          const uint32_t slot = nraw % C::RS;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&raw_empty[slot]), ((nraw / C::RS) & 1) ^ 1,
                                                         limit_ns, abort_flag, err))) {
            ok = false;
            break;
          }
          if (wk.drop && blockIdx.x == 0 && nraw == 1) {  // test hook: the chunk's dequant warps wait it out
            ++nraw;
            continue;
          }
          if (issuer) {
            mbar_arrive_expect_tx(smem_u32(&raw_full[slot]), C::kRawBytes);
            tma_load_2d(sbase + C::kOffRaw + slot * C::kRawBytes, &tmW, r * (C::kRawRow / C::kRawElem), m0,
                        smem_u32(&raw_full[slot]));
          }
          __syncwarp();
          ++nraw;
        }
      }
      if (!ok && issuer) drain_ring(raw_full, C::RS, nraw, limit_ns);
    }
  } else if (warp == C::kXWarp) {
    // ------------------------------------------------------------ x producer
    {
      const bool issuer = elect_one();
      if (issuer) tma_prefetch_desc(&tmX);
      if (!MOE && !wk.x_static) {
        pdl_wait();
        pdl_launch_dependents();
      }
      uint32_t nb = 0;
      bool ok = true;
      for (int i = 0; i < nseg && ok; ++i) {
        Seg sg;
        int n0, nbox = 0;
        if constexpr (MOE) {
          const MoeItem it = moe_item(gi + i * static_cast<int>(gridDim.x), rt, E, M, BN);
          sg.r0 = 0;
          sg.r1 = nr;
          n0 = it.xrow;
          nbox = (it.nvalid + 63) / 64;  // 64-row boxes: rows past the tile's tokens are not loaded
        } else {
          sg = seg_of(gi, i, wk);
          n0 = static_cast<int>(sg.t % wk.ntn) * BN + static_cast<int>(rank) * C::kXRows;
        }
        for (int ks = 4 * sg.r0; ks < 4 * sg.r1; ++ks) {
          const uint32_t bs = nb % C::S;
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait_bounded(smem_u32(&empty[bs]), ((nb / C::S) & 1) ^ 1, limit_ns, abort_flag, err))) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + C::kOffB + bs * C::kBBytes;
          if (issuer) {
            if constexpr (MOE) {
              mbar_arrive_expect_tx(smem_u32(&full[bs]), nbox * 64 * 128);
              for (int b = 0; b < nbox; ++b)
                tma_load_2d(dst + b * 64 * 128, &tmX, ks * C::kBK, n0 + b * 64, smem_u32(&full[bs]));
            } else if (PAIR) {
              if (leader) mbar_arrive_expect_tx(smem_u32(&full[bs]), C::kCtas * C::kBBytes);
              tma_load_2d_pair(dst, &tmX, ks * C::kBK, n0, leader_bar(&full[bs]));
            } else {
              mbar_arrive_expect_tx(smem_u32(&full[bs]), C::kBBytes);
              tma_load_2d(dst, &tmX, ks * C::kBK, n0, smem_u32(&full[bs]));
            }
          }
          __syncwarp();
          ++nb;
        }
      }
      // (a pair's x copies complete on the leader's barriers: only the leader can drain them)
      if (!ok && leader && issuer) drain_ring(full, C::S, nb, limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the leader of a pair)
    // As for the W producer: the converged warp waits, one elected lane issues.
    if (leader) {
      const bool issuer = elect_one();
      if (!MOE && !wk.x_static) pdl_wait();
      uint32_t idesc = umma_idesc_bf16_f32(C::kBM * C::kCtas, BN);
      uint32_t c = 0, seg = 0;
      bool ok = true;
      for (int i = 0; i < nseg && ok; ++i) {
        Seg sg;
        if constexpr (MOE) {
          // only the tile's tokens, rounded up to the MMA's N granularity of 16
          const int nv = moe_item(gi + i * static_cast<int>(gridDim.x), rt, E, M, BN).nvalid;
          idesc = umma_idesc_bf16_f32(C::kBM, static_cast<uint32_t>((nv + 15) / 16 * 16));
          sg.r0 = 0;
          sg.r1 = nr;
        } else {
          sg = seg_of(gi, i, wk);
        }
        // the previous segment's epilogue must have read the accumulator
        if (seg > 0 && !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(acc_empty), (seg - 1) & 1, limit_ns,
                                                                  abort_flag, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 4 * sg.r0; ks < 4 * sg.r1; ++ks, ++c) {
          const uint32_t st = c % C::S;
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait_bounded(smem_u32(&full[st]), (c / C::S) & 1, limit_ns, abort_flag, err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + BN + st * C::kACols;
          const uint32_t b_addr = sbase + C::kOffB + st * C::kBBytes;
          if (issuer) {
#pragma unroll
            for (int kk = 0; kk < C::kBK / 16; ++kk) {
              const uint32_t acc = ks != 4 * sg.r0 || kk != 0;
              if (PAIR)
                umma_bf16_ts_pair(tmem_base, a_tmem + kk * 8, umma_desc_sw128(b_addr + kk * 32), idesc, acc);
              else
                umma_bf16_ts(tmem_base, a_tmem + kk * 8, umma_desc_sw128(b_addr + kk * 32), idesc, acc);
            }
            if (PAIR)
              umma_commit_pair(smem_u32(&empty[st]), 3);
            else
              umma_commit(smem_u32(&empty[st]));
          }
          __syncwarp();
        }
        // also on the error path: tracks every MMA issued so far
        if (issuer) {
          if (PAIR)
            umma_commit_pair(smem_u32(acc_full), 3);
          else
            umma_commit(smem_u32(acc_full));
        }
        __syncwarp();
        ++seg;
      }
      // Do not leave while MMAs issued by this thread may still run: the last
      // commit tracks all of them.
      if (seg > 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(acc_full), (seg - 1) & 1) && globaltimer_ns() - t0 < limit_ns) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue
    // With x_static nothing before the first epilogue touches global memory
    // that the kernel before may still use: Y and the k-split scratch wait there.
    if (!MOE && !wk.x_static) pdl_wait();
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int grp = (warp - 2) >> 2;     // 64-k step grp of every 256-k chunk; then columns grp/4 of the tile
    const int row = quad * 32 + lane;    // W row within this CTA's 128 == TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const bool e0 = warp == 2 && lane == 0;
    constexpr int kCbPerGrp = BN / 128;  // 32-column blocks of the accumulator per group
    const int cb0 = grp * kCbPerGrp, cb1 = cb0 + kCbPerGrp;
    // This group's two blocks of a raw row start at byte 2*grp*kBlk: read the
    // 16-byte words that cover them (for Q4_0 the 36 bytes start at word grp).
    // Q4_K: the row's 16-byte header, then the step's 32 code bytes at 16 + 32*grp.
    const int raw_off = F == GQ_TYPE_Q4_K ? row * C::kRawRow : row * C::kRawRow + (2 * C::kBlk * grp & ~15);
    bool live = true;
    uint32_t cr = 0, c = 0, seg = 0;
    for (int i = 0; i < nseg; ++i) {
      Seg sg;
      MoeItem it{};
      if constexpr (MOE) {
        it = moe_item(gi + i * static_cast<int>(gridDim.x), rt, E, M, BN);
        sg.r0 = 0;
        sg.r1 = nr;
      } else {
        sg = seg_of(gi, i, wk);
      }
      for (int r = sg.r0; r < sg.r1; ++r, ++cr, c += 4) {
        const uint32_t rslot = cr % C::RS;
        const uint32_t as = (c + grp) % C::S;
        if (live) live = mbar_wait_bounded(smem_u32(&raw_full[rslot]), (cr / C::RS) & 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        uint32_t v[4 * C::kWinWords];
        if (live) {
          const uint4* src = reinterpret_cast<const uint4*>(smem + C::kOffRaw + rslot * C::kRawBytes + raw_off);
          const int win0 = F == GQ_TYPE_Q4_K ? 0 : (2 * C::kBlk * grp & ~15);  // window start within the row
#pragma unroll
          for (int i = 0; i < C::kWinWords; ++i) {
            // Q4_K: word 0 is the header, words 1-2 the code bytes at 16 + 32*grp.
            // A word that would start past the row (Q5_0's last group needs 3 of
            // its 4) is not loaded: it holds no byte of the group's blocks.
            if (F != GQ_TYPE_Q4_K && win0 + 16 * i >= C::kRawRow) {
              v[4 * i] = v[4 * i + 1] = v[4 * i + 2] = v[4 * i + 3] = 0u;
              continue;
            }
            const uint4 x = src[(F == GQ_TYPE_Q4_K && i > 0) ? i + 2 * grp : i];
            v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
          }
        }
        __syncwarp();
        if (live && lane == 0) mbar_arrive(smem_u32(&raw_empty[rslot]));
        // Dequantise first, then wait for the A stage: only the store is left
        // between the stage becoming free and the MMA that reads it.
        uint32_t o[32];
        if constexpr (F != GQ_TYPE_Q4_0) {
          switch (grp) {  // warp-uniform
            case 0: step_words_fmt<F, 0>(v, o); break;
            case 1: step_words_fmt<F, 1>(v, o); break;
            case 2: step_words_fmt<F, 2>(v, o); break;
            default: step_words_fmt<F, 3>(v, o); break;
          }
        } else {
          uint32_t w[9];  // blocks 2*grp and 2*grp+1 of the row
#pragma unroll
          for (int i = 0; i < 9; ++i)
            w[i] = grp == 0 ? v[i] : grp == 1 ? v[i + 1] : grp == 2 ? v[i + 2] : v[i + 3];
          const uint32_t q0[4] = {prmt(w[0], w[1], 0x5432u), prmt(w[1], w[2], 0x5432u), prmt(w[2], w[3], 0x5432u),
                                  prmt(w[3], w[4], 0x5432u)};
          const uint32_t q1[4] = {w[5], w[6], w[7], w[8]};
          block_words(q0, w[0] & 0xFFFFu, o);
          block_words(q1, w[4] >> 16, o + 16);
        }
        if (live) live = mbar_wait_bounded(smem_u32(&empty[as]), (((c + grp) / C::S) & 1) ^ 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        if (live) {
          tmem_st_32x32b_x32(lane_addr + BN + as * C::kACols, o);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (live && lane == 0) arrive_leader(&full[as]);
      }

      // ---- epilogue of this segment: this group's quarter of the accumulator columns
      if (!MOE && wk.x_static && seg == 0) pdl_wait();
      if (live) live = mbar_wait_bounded(smem_u32(acc_full), seg & 1, limit_ns, abort_flag, err);
      live = __all_sync(0xFFFFFFFFu, live);
      tc_fence_after();
      if constexpr (MOE) {
        // Column n of the tile is sorted position it.xrow + n; its Y row is
        // the pair perm[it.xrow + n].  Lane j fetches the pair of column
        // 32*cb + j and the warp shares them.
        const int m = it.mrow0 + row;
        if (live) {
#pragma unroll 1
          for (int cb = cb0; cb < cb1 && cb * 32 < it.nvalid; ++cb) {
            uint32_t v32[32];
            tmem_ld_32x32b_x32(lane_addr + cb * 32, v32);
            const int nl = cb * 32 + lane;
            const int my_pair = nl < it.nvalid ? __ldg(rt.perm + it.xrow + nl) : 0;
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int pr = __shfl_sync(0xFFFFFFFFu, my_pair, jj);
              if (m < M && cb * 32 + jj < it.nvalid) Y[static_cast<size_t>(pr) * M + m] = __uint_as_float(v32[jj]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(acc_empty);
        ++seg;
        continue;
      }
      const int m = static_cast<int>(sg.t / wk.ntn) * (C::kBM * C::kCtas) + static_cast<int>(rank) * C::kBM + row;
      const int n0 = static_cast<int>(sg.t % wk.ntn) * BN;
      // Columns n0 + ncols .. n0 + BN - 1 are past N (their x rows were zero
      // fill): neither stored, published nor reduced.
      const int ncols = min(BN, N - n0);
      if (sg.r0 == 0 && sg.r1 == nr) {
        if (live) {
#pragma unroll 1
          for (int cb = cb0; cb < cb1 && cb * 32 < ncols; ++cb) {
            uint32_t v32[32];
            tmem_ld_32x32b_x32(lane_addr + cb * 32, v32);
            tmem_ld_wait();
            if (m < M) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int n = n0 + cb * 32 + jj;
                if (n < N) Y[static_cast<size_t>(n) * M + m] = __uint_as_float(v32[jj]);
              }
            }
          }
        }
      } else {
        // Part of a split tile.  The CTA that sees every other split published
        // reduces: partial sums are added in the order of their k ranges, so
        // the result does not depend on which CTA finishes last.  Each CTA of
        // a pair does this for its own 128 rows.
        const int64_t t = sg.t;
        const int ga = static_cast<int>(t) * wk.s, nsplit = wk.s;  // pieces: ranges ga .. ga + s - 1
        unsigned long long* count = wk.count + t * C::kCtas + rank;
        volatile int* flag = reduce_flag + (seg & 1);
        if (e0) *flag = live && pieces_published(ld_acquire_gpu_u64(count), wk.epoch) == nsplit - 1;
        named_bar_sync(1, 32 * C::kDeqWarps);
        int last = *flag;
        if (!last) {
          if (live) {  // publish this split's partial tile
            float* p = wk.ws + (static_cast<int64_t>(gi) * C::kCtas + rank) * C::kSlotFloats + row;
#pragma unroll 1
            for (int cb = cb0; cb < cb1 && cb * 32 < ncols; ++cb) {
              uint32_t v32[32];
              tmem_ld_32x32b_x32(lane_addr + cb * 32, v32);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) __stcg(p + (cb * 32 + jj) * C::kBM, __uint_as_float(v32[jj]));
            }
          }
          __threadfence();
          named_bar_sync(1, 32 * C::kDeqWarps);
          if (e0) {
            const int before = live ? publish_piece(count, wk.epoch) : -1;
            if (before < 0 && live) atomicOr(err, 1u);
            *flag = before == nsplit - 1;
          }
          named_bar_sync(1, 32 * C::kDeqWarps);
          last = *flag;
        }
        if (last && live) {
          __threadfence();
#pragma unroll 1
          for (int hb = 2 * cb0; hb < 2 * cb1 && hb * 16 < ncols; ++hb) {  // 16-column halves of this group's blocks
            float acc[16];
#pragma unroll 1
            for (int g = ga; g < ga + nsplit; ++g) {
              uint32_t q[16];  // split g's partial sums of these 16 columns
              if (g == gi) {
                tmem_ld_32x32b_x16(lane_addr + hb * 16, q);
                tmem_ld_wait();
              } else {
                const float* p =
                    wk.ws + (static_cast<int64_t>(g) * C::kCtas + rank) * C::kSlotFloats + hb * 16 * C::kBM + row;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) q[jj] = __float_as_uint(__ldcg(p + jj * C::kBM));
              }
              if (g == ga) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) acc[jj] = __uint_as_float(q[jj]);
              } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) acc[jj] += __uint_as_float(q[jj]);
              }
            }
            if (m < M) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                const int n = n0 + hb * 16 + jj;
                if (n < N) Y[static_cast<size_t>(n) * M + m] = acc[jj];
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(acc_empty);
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA frees TMEM or leaves while the pair's MMAs or arrivals may touch it
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

int64_t g_streamk = 1;  // 0: never split tiles; 1: split the last partial wave when it pays; n >= 2: split every tile in n
int64_t g_slots = 0;    // 0: work ranges up to the SM count (pairs: half); n > 0: at most n ranges (test aid)

// Launch tags for the arrival counters: unique per launch in this process; the
// start is random so that scratch memory left by another process's launches
// cannot carry a matching tag either.
std::atomic<unsigned long long> g_epoch{(static_cast<unsigned long long>(std::random_device{}()) << 24) + 1};

// Cost model of a launch, in hundredths of the time one CTA takes for a
// 256-k chunk of a 128 x 256 tile, fitted to this kernel's measured times on
// the GB300 (graphs of calls on weights streamed from DRAM, 4096 to 14336
// rows, K 4096 and 11008, N 512; each estimate within 2 %):
//   a chunk of a 128 x 128 tile                 97  (half the MMA work; the per-step cost stays)
//   a CTA's start and its last epilogue        570 (BN 256) / 430 (BN 128)
//   each further tile's epilogue               520 (BN 256) / 260 (BN 128)
//   a split tile's publish and reduce          830 + 150 per piece beyond two
struct PlanCost {
  int64_t chunk, start, epilogue;
};
constexpr PlanCost plan_cost(int bn) { return bn == 128 ? PlanCost{97, 430, 260} : PlanCost{100, 570, 520}; }
constexpr int64_t split_fixup_cost(int64_t s) { return 830 + 150 * (s - 2); }

// Schedule of T tiles of nr chunks on P ranges (PrefillWork): w = T / P whole
// tiles per range, and the rem = T % P left over either as one more whole
// tile for rem ranges or, when the cost model says it is faster, split
// s = P / rem ways along k.  Returns the estimated cost.
// overlap: the launch runs its main loop beside the launches before and after
// it on the stream (the x-static promise under programmatic dependent launch),
// and they take the SMs it leaves idle.  Its own span then matters less than
// the SM time it uses, which a split only adds to (the hand-off), so its
// tiles stay whole.
int64_t prefill_plan(int64_t T, int64_t nr, int64_t P, bool allow_split, int bn, PrefillWork* wk, bool overlap) {
  if (g_slots > 0) P = g_slots;
  P = std::max<int64_t>(P, 1);
  const PlanCost c = plan_cost(bn);
  wk->T = T;
  wk->R = 0;
  wk->s = 1;
  wk->G = std::min(T, P);
  const int64_t w = T / P, rem = T - w * P;
  const int64_t waves = w + (rem ? 1 : 0);
  const int64_t whole = waves * nr * c.chunk + c.start + (waves > 0 ? waves - 1 : 0) * c.epilogue;
  if (!allow_split || g_streamk == 0 || nr < 2) return whole;
  if (g_streamk >= 2) {  // every tile in pieces (test aid)
    wk->s = static_cast<int>(std::min(g_streamk, nr));
    wk->R = static_cast<int>(T);
    wk->G = T * wk->s;
    return whole;
  }
  if (rem == 0 || overlap) return whole;
  const int64_t s = std::min(P / rem, nr / 2);
  if (s < 2) return whole;
  const int64_t split =
      w * nr * c.chunk + (nr + s - 1) / s * c.chunk + c.start + w * c.epilogue + split_fixup_cost(s);
  if (split >= whole) return whole;
  wk->R = static_cast<int>(rem);
  wk->s = static_cast<int>(s);
  wk->G = std::max(std::min(T, P), rem * s);
  return split;
}

template <int BN, bool PAIR, int F = GQ_TYPE_Q4_0>
cudaError_t launch_prefill_cfg(const CUtensorMap* tmW, const CUtensorMap* tmX, int N, int M, int K, float* Y,
                               uint64_t limit_ns, bool allow_scratch, int early_w, int x_static, int pdl,
                               cudaStream_t s) {
  using C = PrefillCfg<BN, PAIR, F>;
  auto kern = k_prefill_q4_0<BN, PAIR, false, F>;
  {
    cudaError_t e = kernel_smem(reinterpret_cast<const void*>(kern), C::kSmem, false);
    if (e != cudaSuccess) return e;
  }
  const int64_t ntn = (N + BN - 1) / BN;
  const int64_t rows = C::kBM * C::kCtas;
  const int64_t T = ((M + rows - 1) / rows) * ntn;
  const int64_t nr = K / C::kRawK;
  PrefillWork wk{};
  wk.nr = static_cast<int>(nr);
  wk.ntn = static_cast<int>(ntn);
  wk.early_w = pdl && early_w;
  wk.x_static = pdl && x_static;
  wk.drop = test_drop() == 2 ? 1 : 0;
  prefill_plan(T, nr, device_info().sm_count / C::kCtas, allow_scratch, BN, &wk, wk.x_static != 0);
  void* scratch = nullptr;
  if (wk.R > 0) {  // split tiles: partial-tile slots and arrival counters
    const size_t ws_bytes =
        static_cast<size_t>(wk.R) * wk.s * C::kCtas * static_cast<size_t>(C::kSlotFloats) * sizeof(float);
    const size_t cnt_bytes = static_cast<size_t>(wk.R) * C::kCtas * sizeof(unsigned long long);
    if (scratch_alloc(&scratch, ws_bytes + cnt_bytes, s) == cudaSuccess) {
      wk.ws = static_cast<float*>(scratch);
      wk.count = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(scratch) + ws_bytes);
      wk.epoch = g_epoch.fetch_add(1) & ((1ull << 56) - 1);
    } else {  // no scratch: whole tiles only
      cudaGetLastError();
      if (scratch) scratch_free(scratch, s);
      scratch = nullptr;
      wk.R = 0;
      wk.s = 1;
      wk.G = std::min<int64_t>(T, std::max<int64_t>(1, g_slots > 0 ? g_slots : device_info().sm_count / C::kCtas));
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(wk.G * C::kCtas));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, *tmW, *tmX, N, M, Y, wk, limit_ns, device_error_word(), MoeRoute{}, 0);
  if (scratch) {
    cudaError_t f = scratch_free(scratch, s);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

int g_bn_override = 0;  // 0: choose by shape; 128 or 256: force the tile width (tuning)

// Tile width: 128 tokens up to N = 128; beyond, whichever of 128 and 256 the
// cost model above rates faster for this shape (e.g. 4096 x 4096 x 512: 64
// tiles of 256 tokens leave 88 of 152 SMs idle or split tiles, 128 tiles of
// 128 tokens do not).  Under overlap (see prefill_plan) the SMs a launch
// leaves idle go to its neighbours, and 256-token tiles take the least SM
// time (a 64-k step costs about as much at either width).
int prefill_bn(int64_t N, int64_t M, int64_t K, bool allow_split, bool overlap) {
  if (g_bn_override) return g_bn_override;
  if (N <= 128) return 128;
  if (overlap) return 256;
  const int64_t P = device_info().sm_count, rows = (M + 127) / 128, nr = K / 256;
  PrefillWork w128{}, w256{};
  const int64_t c128 = prefill_plan(rows * ((N + 127) / 128), nr, P, allow_split, 128, &w128, false);
  const int64_t c256 = prefill_plan(rows * ((N + 255) / 256), nr, P, allow_split, 256, &w256, false);
  return c128 < c256 ? 128 : 256;
}

// 0 (default): 1-CTA kernel with 128 x prefill_bn tiles; 1: 2-SM pair kernel (256 x 256 tiles).
int g_pair_mode = 0;
bool use_pair(int64_t N) { return g_pair_mode && g_bn_override == 0 && N > 128; }

}  // namespace

void set_prefill_bn_override(int bn) { g_bn_override = bn; }
int get_prefill_bn_override() { return g_bn_override; }

void prefill_boxes(int64_t N, int64_t M, int64_t K, bool allow_split, bool overlap, int type, uint32_t* w_box_x,
                   uint32_t* w_elem_bytes, uint32_t* w_box_rows, uint32_t* x_box_k, uint32_t* x_box_rows) {
  const uint32_t raw_row = static_cast<uint32_t>(type_row_bytes(type, 256));  // 256 k of a row
  *w_elem_bytes = raw_row > 256 ? 2u : 1u;
  *w_box_x = raw_row / *w_elem_bytes;
  *w_box_rows = 128;
  *x_box_k = 64;
  *x_box_rows = (type == GQ_TYPE_Q4_0 && use_pair(N)) ? 128u
                                                        : static_cast<uint32_t>(prefill_bn(N, M, K, allow_split, overlap));
}

void set_prefill_pair_mode(int on) { g_pair_mode = on ? 1 : 0; }
void set_prefill_streamk(int64_t v) { g_streamk = v; }
int64_t get_prefill_streamk() { return g_streamk; }
void set_prefill_slots(int64_t v) { g_slots = v; }
int64_t get_prefill_slots() { return g_slots; }
int get_prefill_pair_mode() { return g_pair_mode; }

cudaError_t launch_prefill_moe(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t E, int64_t M, int64_t K,
                               int64_t P, const MoeRoute& rt, float* Y, uint64_t wait_limit_ns, int pdl,
                               cudaStream_t s) {
  using C = PrefillCfg<kMoeBN, false>;
  auto kern = k_prefill_q4_0<kMoeBN, false, true>;
  {
    cudaError_t e = kernel_smem(reinterpret_cast<const void*>(kern), C::kSmem, false);
    if (e != cudaSuccess) return e;
  }
  // Work items: at most (row tiles) x (token tiles), where the token tiles of
  // all experts number at most P / BN + min(E, P).
  const int64_t n_mtiles = (M + C::kBM - 1) / C::kBM;
  const int64_t max_items = n_mtiles * ((P + kMoeBN - 1) / kMoeBN + std::min(E, P));
  int64_t G = device_info().sm_count;
  if (g_slots > 0) G = g_slots;
  G = std::max<int64_t>(1, std::min(G, max_items));
  PrefillWork wk{};
  wk.nr = static_cast<int>(K / C::kRawK);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, *tmW, *tmX, 0, static_cast<int>(M), Y, wk, wait_limit_ns,
                            device_error_word(), rt, static_cast<int>(E));
}

cudaError_t launch_prefill(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t N, int64_t M, int64_t K,
                           float* Y, uint64_t wait_limit_ns, bool allow_scratch, int early_w, int x_static, int pdl,
                           cudaStream_t s, int type) {
  const int n = static_cast<int>(N), m = static_cast<int>(M), k = static_cast<int>(K);
  const bool overlap = pdl && x_static;
  if (type == GQ_TYPE_Q4_1) {
    if (prefill_bn(N, M, K, allow_scratch, overlap) == 128)
      return launch_prefill_cfg<128, false, GQ_TYPE_Q4_1>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
    return launch_prefill_cfg<256, false, GQ_TYPE_Q4_1>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  }
  if (type == GQ_TYPE_Q8_0) {
    if (prefill_bn(N, M, K, allow_scratch, overlap) == 128)
      return launch_prefill_cfg<128, false, GQ_TYPE_Q8_0>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
    return launch_prefill_cfg<256, false, GQ_TYPE_Q8_0>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  }
  if (type == GQ_TYPE_Q5_0) {
    if (prefill_bn(N, M, K, allow_scratch, overlap) == 128)
      return launch_prefill_cfg<128, false, GQ_TYPE_Q5_0>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
    return launch_prefill_cfg<256, false, GQ_TYPE_Q5_0>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  }
  if (type == GQ_TYPE_Q5_1) {
    if (prefill_bn(N, M, K, allow_scratch, overlap) == 128)
      return launch_prefill_cfg<128, false, GQ_TYPE_Q5_1>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
    return launch_prefill_cfg<256, false, GQ_TYPE_Q5_1>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  }
  if (type == GQ_TYPE_Q4_K) {
    if (prefill_bn(N, M, K, allow_scratch, overlap) == 128)
      return launch_prefill_cfg<128, false, GQ_TYPE_Q4_K>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
    return launch_prefill_cfg<256, false, GQ_TYPE_Q4_K>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  }
  if (use_pair(N)) return launch_prefill_cfg<256, true>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  if (prefill_bn(N, M, K, allow_scratch, overlap) == 128) return launch_prefill_cfg<128, false>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
  return launch_prefill_cfg<256, false>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, early_w, x_static, pdl, s);
}

}  // namespace gq
