// KL: the other legacy block formats, Q4_1, Q8_0, Q5_0 and Q5_1:
// dequantisation (bit-exact) and MUL_MAT.
//
// "Architecture and module overview", quantisation-format section: the legacy
// formats keep one scale per block of 32 weights, Q4_1 additionally a min
// offset, Q8_0 eight bits per weight.  Layout read from that section and the
// Q4_0 struct of "Binding GGUF weights to the compute graph", section 2.3:
//   Q4_1: ggml_half d, ggml_half m, uint8_t qs[16]  (20 bytes), w = d*q + m,
//         q = 0..15, low nibble of qs[j] = element j, high nibble = j+16;
//   Q8_0: ggml_half d, int8_t qs[32]                (34 bytes), w = d*q.
//   Q5_0: ggml_half d, uint8_t qh[4], uint8_t qs[16]           (22 bytes), w = d*(q - 16),
//   Q5_1: ggml_half d, ggml_half m, uint8_t qh[4], uint8_t qs[16] (24 bytes), w = d*q + m,
//         the 5-bit q of element e = its Q4_0-order nibble + 16 * bit e of
//         the little-endian word qh.
// In fp32 d*q is exact (at most 11 x 8 significant bits); Q4_1 and Q5_1 add m
// with one rounding.  Both kernels evaluate exactly that, so dequantisation is
// bit-exact and MUL_MAT sees the same weights.
//
// MUL_MAT here is the decode-shaped kernel for these formats: one warp per
// weight row, eight lanes per block, four blocks per step (coalesced W and x
// loads), each lane keeping the W words of 8 steps in flight.  Per block part
// and token a lane forms sum(q x) over its four exact
// integer codes in fp32 and applies the scale, d*sum(q x) (+ m*sum(x) for
// Q4_1): the same value as sum((d q + m) x) up to rounding order.  Up to kTok tokens per pass; the lanes' partial sums meet by
// shuffles.  W is read from DRAM once per pass; more tokens than kTok re-read
// it from L2.
#include <algorithm>
#include <cuda_fp16.h>

#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {
namespace {

template <int T>
struct Fmt;
template <>
struct Fmt<GQ_TYPE_Q4_1> {
  static constexpr int kBytes = 20;
};
template <>
struct Fmt<GQ_TYPE_Q8_0> {
  static constexpr int kBytes = 34;
};
template <>
struct Fmt<GQ_TYPE_Q5_0> {
  static constexpr int kBytes = 22;
};
template <>
struct Fmt<GQ_TYPE_Q5_1> {
  static constexpr int kBytes = 24;
};

// Formats with a min offset m (the fp16 field after d) and 5-bit formats.
template <int T>
constexpr bool has_min() { return T == GQ_TYPE_Q4_1 || T == GQ_TYPE_Q5_1; }
template <int T>
constexpr bool five_bit() { return T == GQ_TYPE_Q5_0 || T == GQ_TYPE_Q5_1; }
// Byte offsets of Q5's high-bit word and codes within a block.
template <int T>
constexpr int q5_qh_off() { return T == GQ_TYPE_Q5_1 ? 4 : 2; }

__device__ __forceinline__ float half_at(const uint8_t* p) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(p[0] | (p[1] << 8))));
}

// The little-endian high-bit word of a Q5 block (byte loads: any alignment).
template <int T>
__device__ __forceinline__ uint32_t q5_high_bits(const uint8_t* blk) {
  const uint8_t* p = blk + q5_qh_off<T>();
  return p[0] | (p[1] << 8) | (p[2] << 16) | (static_cast<uint32_t>(p[3]) << 24);
}

// Element e (0..31) of a block held in shared or global memory.
template <int T>
__device__ __forceinline__ float weight(const uint8_t* blk, int e, float d, float m) {
  if constexpr (five_bit<T>()) {
    const uint32_t byte = blk[q5_qh_off<T>() + 4 + (e & 15)];
    const uint32_t q = (e < 16 ? (byte & 0xF) : (byte >> 4)) | (((q5_high_bits<T>(blk) >> e) & 1u) << 4);
    if constexpr (T == GQ_TYPE_Q5_0) return __fmul_rn(d, static_cast<float>(static_cast<int>(q) - 16));
    else return __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
  } else if constexpr (T == GQ_TYPE_Q4_1) {
    const uint32_t byte = blk[4 + (e & 15)];
    const uint32_t q = e < 16 ? (byte & 0xF) : (byte >> 4);
    return __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
  } else {
    (void)m;
    return __fmul_rn(d, static_cast<float>(static_cast<int8_t>(blk[2 + e])));
  }
}

constexpr int kDqThreads = 256;
constexpr int kDqTile = 256;  // blocks per tile: a multiple of 8, so 16-byte aligned tiles stay aligned

// Tiles of 256 blocks are staged in shared memory (16-byte loads when W is
// 16-byte aligned, else byte loads); each thread then writes float4 outputs,
// consecutive threads consecutive 16 bytes.
template <int T>
__global__ void __launch_bounds__(kDqThreads) k_dequant_legacy(const uint8_t* __restrict__ W, int64_t nblocks,
                                                               float* __restrict__ out, int vec_in, int vec_out) {
  constexpr int kB = Fmt<T>::kBytes;
  __shared__ __align__(16) uint8_t tile[kDqTile * kB];
  const int64_t ntiles = (nblocks + kDqTile - 1) / kDqTile;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t b0 = t * kDqTile;
    const int nb = static_cast<int>(nblocks - b0 < kDqTile ? nblocks - b0 : kDqTile);
    const int nbytes = nb * kB;
    const uint8_t* src = W + b0 * kB;
    __syncthreads();
    if (vec_in) {
      for (int c = threadIdx.x; c * 16 < nbytes; c += kDqThreads) {
        if (c * 16 + 16 <= nbytes)
          *reinterpret_cast<uint4*>(tile + c * 16) = __ldg(reinterpret_cast<const uint4*>(src + c * 16));
        else
          for (int i = c * 16; i < nbytes; ++i) tile[i] = src[i];
      }
    } else {
      for (int i = threadIdx.x; i < nbytes; i += kDqThreads) tile[i] = src[i];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < nb * 8; o += kDqThreads) {
      const int b = o >> 3, part = o & 7;
      const uint8_t* blk = tile + b * kB;
      const float d = half_at(blk);
      const float m = has_min<T>() ? half_at(blk + 2) : 0.f;
      float4 v;
      v.x = weight<T>(blk, 4 * part, d, m);
      v.y = weight<T>(blk, 4 * part + 1, d, m);
      v.z = weight<T>(blk, 4 * part + 2, d, m);
      v.w = weight<T>(blk, 4 * part + 3, d, m);
      float* dst = out + (b0 + b) * kQK + 4 * part;
      if (vec_out) {
        *reinterpret_cast<float4*>(dst) = v;
      } else {
        dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
      }
    }
  }
}

constexpr int kTok = 4;  // tokens per pass of the MUL_MAT kernel

// Integer codes to fp32 without the conversion unit: 0x4B000000 | u is the
// float 2^23 + u exactly (u < 2^23), so subtracting 2^23 leaves u.
__device__ __forceinline__ float u2f(uint32_t u) { return __int_as_float(0x4B000000 | u) - 8388608.0f; }

// The raw words a lane needs for elements 4p..4p+3 (p = 0..7) of a block:
// the scale word (d, and m for Q4_1) and the 4 code bytes.
// Q5 part p (elements 4p..4p+3): their 4 nibbles in bits 0-3 of each byte of
// the result, and their 4 high bits (bits 4p..4p+3 of qh) in bit 4 of each byte.
__device__ __forceinline__ uint32_t q5_part_codes(uint32_t codes, uint32_t qh, int p) {
  const uint32_t nib = ((p & 4) ? codes >> 4 : codes) & 0x0F0F0F0Fu;
  const uint32_t hb = (qh >> (4 * p)) & 0xFu;  // bit i: element 4p + i
  // bit i to bit 8i: the products hb_i * 2^(7j) land on distinct bits, so the
  // multiply carries nothing into the mask
  const uint32_t spread = (hb * 0x00204081u) & 0x01010101u;
  return nib | (spread << 4);
}

template <int T>
__device__ __forceinline__ void load_part(const uint8_t* __restrict__ blk, int p, uint32_t& h, uint32_t& v) {
  if constexpr (five_bit<T>()) {
    // 22- / 24-byte blocks of a 2-byte aligned row: 16-bit loads
    const uint16_t* w = reinterpret_cast<const uint16_t*>(blk);
    constexpr int qo = q5_qh_off<T>() / 2;  // qh at halfword qo, codes at qo + 2
    h = has_min<T>() ? (static_cast<uint32_t>(__ldg(w)) | (static_cast<uint32_t>(__ldg(w + 1)) << 16))
                     : static_cast<uint32_t>(__ldg(w));
    const uint32_t qh = static_cast<uint32_t>(__ldg(w + qo)) | (static_cast<uint32_t>(__ldg(w + qo + 1)) << 16);
    const int c = qo + 2 + 2 * (p & 3);
    const uint32_t codes = static_cast<uint32_t>(__ldg(w + c)) | (static_cast<uint32_t>(__ldg(w + c + 1)) << 16);
    v = q5_part_codes(codes, qh, p);
  } else if constexpr (T == GQ_TYPE_Q4_1) {
    // 20-byte blocks of a 4-byte aligned row: the scale word and one code word
    const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
    h = __ldg(w);
    v = __ldg(w + 1 + (p & 3)) >> ((p & 4) ? 4 : 0);  // parts 4..7: high nibbles
  } else {
    // 34-byte blocks are 2-byte aligned: the scale and two 16-bit code loads
    const uint16_t* w = reinterpret_cast<const uint16_t*>(blk);
    h = __ldg(w);
    v = static_cast<uint32_t>(__ldg(w + 1 + 2 * p)) | (static_cast<uint32_t>(__ldg(w + 2 + 2 * p)) << 16);
  }
}

// Codes as fp32 (exact small integers: Q4_1 0..15, Q8_0 -128..127; a Q8_0
// code c is (c ^ 0x80) - 128 with c ^ 0x80 in 0..255) and the scales.
template <int T>
__device__ __forceinline__ void decode_part(uint32_t h, uint32_t v, float (&q)[4], float& d, float& m) {
  d = __half2float(__ushort_as_half(static_cast<uint16_t>(h & 0xFFFF)));
  if constexpr (five_bit<T>()) {
    m = has_min<T>() ? __half2float(__ushort_as_half(static_cast<uint16_t>(h >> 16))) : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = u2f((v >> (8 * j)) & 0x1F) - (T == GQ_TYPE_Q5_0 ? 16.0f : 0.0f);
  } else if constexpr (T == GQ_TYPE_Q4_1) {
    m = __half2float(__ushort_as_half(static_cast<uint16_t>(h >> 16)));
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = u2f((v >> (8 * j)) & 0xF);
  } else {
    m = 0.f;
    v ^= 0x80808080u;
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = u2f((v >> (8 * j)) & 0xFF) - 128.0f;
  }
}

constexpr int kSteps = 8;  // steps of four blocks whose W words a lane loads before using them

// Eight lanes share a block (lane l takes elements 4*(l%8) .. +3 of block
// 4*step + l/8), so a warp's x loads of one step are 512 contiguous bytes and
// its W loads cover four consecutive blocks.  A lane first loads the W words
// of kSteps steps (the kernel is bound by DRAM latency otherwise), then
// computes them.
template <int T>
__global__ void __launch_bounds__(256) k_mul_mat_legacy(const uint8_t* __restrict__ W, int M, int K,
                                                        const float* __restrict__ X, int N, float* __restrict__ Y) {
  constexpr int kB = Fmt<T>::kBytes;
  const int lane = threadIdx.x & 31;
  const int part = lane & 7, sub = lane >> 3;
  const int nb = K / kQK;
  const int64_t row_bytes = static_cast<int64_t>(nb) * kB;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint8_t* row = W + m * row_bytes;
    for (int n0 = 0; n0 < N; n0 += kTok) {
      const int nt = N - n0 < kTok ? N - n0 : kTok;
      float acc[kTok] = {};
      for (int b0 = sub; b0 < nb; b0 += 4 * kSteps) {
        uint32_t h[kSteps], v[kSteps];
#pragma unroll
        for (int i = 0; i < kSteps; ++i) {
          h[i] = 0;
          v[i] = 0;
          if (b0 + 4 * i < nb) load_part<T>(row + static_cast<int64_t>(b0 + 4 * i) * kB, part, h[i], v[i]);
        }
        float q[kSteps][4], d[kSteps], mn[kSteps];
#pragma unroll
        for (int i = 0; i < kSteps; ++i) decode_part<T>(h[i], v[i], q[i], d[i], mn[i]);
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t < nt) {
            // this token's x for all kSteps steps first (independent loads), then the sums
            const float4* xr = reinterpret_cast<const float4*>(X + static_cast<int64_t>(n0 + t) * K) + part;
            float4 xv[kSteps];
#pragma unroll
            for (int i = 0; i < kSteps; ++i)
              xv[i] = (b0 + 4 * i < nb) ? __ldg(xr + (b0 + 4 * i) * (kQK / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            float a = acc[t];
#pragma unroll
            for (int i = 0; i < kSteps; ++i) {
              float qx = q[i][0] * xv[i].x;
              qx = fmaf(q[i][1], xv[i].y, qx);
              qx = fmaf(q[i][2], xv[i].z, qx);
              qx = fmaf(q[i][3], xv[i].w, qx);
              a = fmaf(d[i], qx, a);
              if (has_min<T>()) a = fmaf(mn[i], (xv[i].x + xv[i].y) + (xv[i].z + xv[i].w), a);
            }
            acc[t] = a;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        if (lane == 0 && t < nt) Y[static_cast<int64_t>(n0 + t) * M + m] = a;
      }
    }
  }
}

// The same computation with each warp's rows double-buffered in shared
// memory: one lane copies the next whole row with a bulk copy while the warp
// computes the current one, so every warp keeps a full row of W in flight.
// Needs W 16-byte aligned and rows a multiple of 16 bytes.
constexpr int kBulkMaxWarps = 8;

template <int T>
__global__ void __launch_bounds__(256) k_mul_mat_legacy_bulk(const uint8_t* __restrict__ W, int M, int K,
                                                             const float* __restrict__ X, int N,
                                                             float* __restrict__ Y, uint64_t limit_ns,
                                                             uint32_t* err) {
  constexpr int kB = Fmt<T>::kBytes;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kBulkMaxWarps][2];
  __shared__ volatile int abort_flag;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = lane & 7, sub = lane >> 3;
  const int nb = K / kQK;
  const uint32_t rb = static_cast<uint32_t>(nb * kB);  // row bytes, a multiple of 16
  uint8_t* buf[2] = {smem + (2 * warp) * rb, smem + (2 * warp + 1) * rb};
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    mbar_init(smem_u32(&bars[warp][0]), 1);
    mbar_init(smem_u32(&bars[warp][1]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int gw = blockIdx.x * (blockDim.x >> 5) + warp, nw = gridDim.x * (blockDim.x >> 5);
  if (gw < M && lane == 0) {
    mbar_arrive_expect_tx(smem_u32(&bars[warp][0]), rb);
    bulk_load(smem_u32(buf[0]), W + static_cast<int64_t>(gw) * rb, rb, smem_u32(&bars[warp][0]));
  }
  int issued = gw < M ? 1 : 0, i = 0;
  bool live = true;
  for (int m = gw; m < M && live; m += nw, ++i) {
    const int j = i & 1;
    if (m + nw < M && lane == 0) {  // the other buffer was last read before the previous __syncwarp
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(smem_u32(&bars[warp][j ^ 1]), rb);
      bulk_load(smem_u32(buf[j ^ 1]), W + static_cast<int64_t>(m + nw) * rb, rb, smem_u32(&bars[warp][j ^ 1]));
      ++issued;
    }
    live = mbar_wait_bounded(smem_u32(&bars[warp][j]), (i >> 1) & 1, limit_ns, &abort_flag, err);
    live = __all_sync(0xFFFFFFFFu, live);
    if (!live) break;
    const uint8_t* row = buf[j];
    for (int n0 = 0; n0 < N; n0 += kTok) {
      const int nt = N - n0 < kTok ? N - n0 : kTok;
      float acc[kTok] = {};
      for (int b0 = sub; b0 < nb; b0 += 4 * kSteps) {
        float q[kSteps][4], d[kSteps], mn[kSteps];
#pragma unroll
        for (int s2 = 0; s2 < kSteps; ++s2) {
          uint32_t h = 0, v = 0;
          const int b = b0 + 4 * s2;
          if (b < nb) {
            const uint8_t* blk = row + b * kB;
            if constexpr (five_bit<T>()) {
              const uint16_t* w16 = reinterpret_cast<const uint16_t*>(blk);
              constexpr int qo = q5_qh_off<T>() / 2;
              h = has_min<T>() ? (static_cast<uint32_t>(w16[0]) | (static_cast<uint32_t>(w16[1]) << 16)) : w16[0];
              const uint32_t qh = static_cast<uint32_t>(w16[qo]) | (static_cast<uint32_t>(w16[qo + 1]) << 16);
              const int c = qo + 2 + 2 * (part & 3);
              v = q5_part_codes(static_cast<uint32_t>(w16[c]) | (static_cast<uint32_t>(w16[c + 1]) << 16), qh, part);
            } else if constexpr (T == GQ_TYPE_Q4_1) {
              h = *reinterpret_cast<const uint32_t*>(blk);
              v = *reinterpret_cast<const uint32_t*>(blk + 4 + 4 * (part & 3)) >> ((part & 4) ? 4 : 0);
            } else {
              h = *reinterpret_cast<const uint16_t*>(blk);
              v = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(blk + 2 + 4 * part)) |
                  (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(blk + 4 + 4 * part)) << 16);
            }
          }
          decode_part<T>(h, v, q[s2], d[s2], mn[s2]);
        }
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t < nt) {
            const float4* xr = reinterpret_cast<const float4*>(X + static_cast<int64_t>(n0 + t) * K) + part;
            float4 xv[kSteps];
#pragma unroll
            for (int s2 = 0; s2 < kSteps; ++s2)
              xv[s2] = (b0 + 4 * s2 < nb) ? __ldg(xr + (b0 + 4 * s2) * (kQK / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            float a = acc[t];
#pragma unroll
            for (int s2 = 0; s2 < kSteps; ++s2) {
              float qx = q[s2][0] * xv[s2].x;
              qx = fmaf(q[s2][1], xv[s2].y, qx);
              qx = fmaf(q[s2][2], xv[s2].z, qx);
              qx = fmaf(q[s2][3], xv[s2].w, qx);
              a = fmaf(d[s2], qx, a);
              if (has_min<T>()) a = fmaf(mn[s2], (xv[s2].x + xv[s2].y) + (xv[s2].z + xv[s2].w), a);
            }
            acc[t] = a;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        if (lane == 0 && t < nt) Y[static_cast<int64_t>(n0 + t) * M + m] = a;
      }
    }
    __syncwarp();  // every lane is done with buf[j] before it is refilled
  }
  // Leave no copy in flight: wait (bounded) for the last phase of each buffer.
  if (lane == 0) {
    for (int k = issued - 1; k >= 0 && k >= issued - 2; --k) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&bars[warp][k & 1]), (k >> 1) & 1) && globaltimer_ns() - t0 < limit_ns) {
      }
    }
  }
}

// Any alignment: one warp per row, byte loads of W and scalar loads of x.
template <int T>
__global__ void k_mul_mat_legacy_bytes(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                       const float* __restrict__ X, int64_t N, float* __restrict__ Y) {
  constexpr int kB = Fmt<T>::kBytes;
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / kQK;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t m = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint8_t* row = W + m * nb * kB;
    for (int64_t n = 0; n < N; ++n) {
      const float* x = X + n * K;
      float acc = 0.f;
      for (int64_t b = lane; b < nb; b += 32) {
        const uint8_t* blk = row + b * kB;
        const float d = half_at(blk);
        const float mn = has_min<T>() ? half_at(blk + 2) : 0.f;
        for (int e = 0; e < kQK; ++e) acc = fmaf(weight<T>(blk, e, d, mn), x[b * kQK + e], acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (lane == 0) Y[n * M + m] = acc;
    }
  }
}

template <int T>
cudaError_t launch_dequant_t(const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s) {
  const int64_t ntiles = (nblocks + kDqTile - 1) / kDqTile;
  const int grid = static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(device_info().sm_count) * 8));
  const int vec_in = (reinterpret_cast<uintptr_t>(W) & 15) == 0;
  const int vec_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  k_dequant_legacy<T><<<grid > 0 ? grid : 1, kDqThreads, 0, s>>>(W, nblocks, out, vec_in, vec_out);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_mul_mat_t(const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                             uint64_t limit_ns, cudaStream_t s) {
  const int64_t rows_per_cta = 8;  // 8 warps
  const int grid = static_cast<int>(
      std::min<int64_t>((M + rows_per_cta - 1) / rows_per_cta, static_cast<int64_t>(device_info().sm_count) * 16));
  // The fast kernel needs 4-byte aligned rows for Q4_1 (2-byte for Q8_0), 16-byte aligned x rows and
  // int sizes; anything else takes the byte kernel.
  const int64_t row_bytes = (K / kQK) * Fmt<T>::kBytes;
  const uintptr_t wa = reinterpret_cast<uintptr_t>(W), xa = reinterpret_cast<uintptr_t>(X);
  const bool fast = ((wa | static_cast<uintptr_t>(row_bytes)) & (T == GQ_TYPE_Q4_1 ? 3 : 1)) == 0 && (xa & 15) == 0 &&
                    K % 4 == 0 && M < (int64_t(1) << 31) && K < (int64_t(1) << 31) && N < (int64_t(1) << 31);
  const int rb = static_cast<int>(row_bytes);
  int bulk_warps = 0;
  // (one pass over the rows: with more tokens the plain kernel re-reads W from L2 faster)
  if (fast && N <= kTok && (wa & 15) == 0 && row_bytes % 16 == 0 && row_bytes <= 96 * 1024) {
    bulk_warps = std::min(kBulkMaxWarps, static_cast<int>((200 * 1024) / (2 * row_bytes)));
  }
  if (bulk_warps > 0) {
    auto kern = k_mul_mat_legacy_bulk<T>;
    const int smem = 2 * bulk_warps * rb;
    cudaError_t e = kernel_smem(reinterpret_cast<const void*>(kern), 200 * 1024, false);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = kernel_occupancy(reinterpret_cast<const void*>(kern), 32 * bulk_warps, smem, &occ);
    if (e != cudaSuccess) return e;
    const int64_t ctas = std::min<int64_t>((M + bulk_warps - 1) / bulk_warps,
                                           static_cast<int64_t>(device_info().sm_count) * std::max(occ, 1));
    kern<<<static_cast<unsigned>(ctas), 32 * bulk_warps, smem, s>>>(W, static_cast<int>(M), static_cast<int>(K), X,
                                                                     static_cast<int>(N), Y, limit_ns,
                                                                     device_error_word());
  } else if (fast)
    k_mul_mat_legacy<T><<<grid > 0 ? grid : 1, 256, 0, s>>>(W, static_cast<int>(M), static_cast<int>(K), X,
                                                             static_cast<int>(N), Y);
  else
    k_mul_mat_legacy_bytes<T><<<grid > 0 ? grid : 1, 256, 0, s>>>(W, M, K, X, N, Y);
  return cudaGetLastError();
}

}  // namespace

int type_block_bytes(int type) {
  switch (type) {
    case GQ_TYPE_Q4_0: return kBlockBytes;
    case GQ_TYPE_Q4_1: return Fmt<GQ_TYPE_Q4_1>::kBytes;
    case GQ_TYPE_Q8_0: return Fmt<GQ_TYPE_Q8_0>::kBytes;
    case GQ_TYPE_Q4_K: return 144;
    case GQ_TYPE_Q5_0: return Fmt<GQ_TYPE_Q5_0>::kBytes;
    case GQ_TYPE_Q5_1: return Fmt<GQ_TYPE_Q5_1>::kBytes;
  }
  return 0;
}

int type_block_weights(int type) { return type == GQ_TYPE_Q4_K ? 256 : kQK; }

uint64_t type_row_bytes(int type, int64_t K) {
  const int bw = type_block_weights(type);
  if (K < 0 || K % bw) return 0;
  return static_cast<uint64_t>(K / bw) * static_cast<uint64_t>(type_block_bytes(type));
}

cudaError_t launch_dequant_legacy(int type, const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s) {
  if (type == GQ_TYPE_Q4_1) return launch_dequant_t<GQ_TYPE_Q4_1>(W, nblocks, out, s);
  if (type == GQ_TYPE_Q5_0) return launch_dequant_t<GQ_TYPE_Q5_0>(W, nblocks, out, s);
  if (type == GQ_TYPE_Q5_1) return launch_dequant_t<GQ_TYPE_Q5_1>(W, nblocks, out, s);
  return launch_dequant_t<GQ_TYPE_Q8_0>(W, nblocks, out, s);
}

cudaError_t launch_mul_mat_legacy(int type, const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N,
                                  float* Y, uint64_t wait_limit_ns, cudaStream_t s) {
  if (type == GQ_TYPE_Q4_1) return launch_mul_mat_t<GQ_TYPE_Q4_1>(W, M, K, X, N, Y, wait_limit_ns, s);
  if (type == GQ_TYPE_Q5_0) return launch_mul_mat_t<GQ_TYPE_Q5_0>(W, M, K, X, N, Y, wait_limit_ns, s);
  if (type == GQ_TYPE_Q5_1) return launch_mul_mat_t<GQ_TYPE_Q5_1>(W, M, K, X, N, Y, wait_limit_ns, s);
  return launch_mul_mat_t<GQ_TYPE_Q8_0>(W, M, K, X, N, Y, wait_limit_ns, s);
}

}  // namespace gq
