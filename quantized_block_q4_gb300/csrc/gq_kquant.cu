// KK: Q4_K, the 4-bit k-quant: dequantisation (bit-exact) and the MUL_MAT
// kernel for shapes and alignments the fast kernels do not take.
//
// "Architecture and module overview", quantisation-format section and the
// error-model paragraph of its weight-loading section: k-quants group 256
// weights per block and keep the block's scales and mins hierarchically inside
// it, an upper level in 6 bits and a lower one in 4; "GGUF loading, mmap and
// tensor placement": a Q4_K tensor takes ne[0]/256 x block-size bytes.  The
// layout taken (the one GGUF files carry), a 144-byte super-block:
//   bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 sixteen 6-bit fields (sc_j, m_j of
//   the 8 sub-blocks of 32 weights), 16-143 qs[128]; weight 64c + l (l < 32)
//   is the low nibble of qs[32c + l] in sub-block 2c, weight 64c + 32 + l its
//   high nibble in sub-block 2c + 1;  w = d*sc_j*q - dmin*m_j.
// (The packing of the 6-bit fields is spelled out in gq_q4k.cuh.)
// In fp32, d*sc_j (<= 17 significant bits) times q (4 bits) and dmin*m_j are
// exact, so one fused multiply-add gives the weight rounded once: the value
// the dequantisation must produce, bit for bit.
#include <algorithm>
#include <cuda_fp16.h>

#include "gq_internal.h"
#include "gq_ptx.cuh"
#include "gq_q4k.cuh"

namespace gq {
namespace {

constexpr int kSuperWeights = kQ4KWeights;
constexpr int kSuperBytes = kQ4KBytes;

__device__ __forceinline__ float half_bits(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h & 0xFFFFu)));
}

// The 8 weights of lane part i (0..31) of a super-block: weights 8i .. 8i+7,
// i.e. chunk c = i / 8, sub-block 2c (i % 8 < 4, low nibbles) or 2c + 1 (high
// nibbles), code bytes 32c + 8 (i % 4) .. + 7.  ALIGNED: the super-block is
// 16-byte aligned (vector loads); otherwise byte loads.
template <bool ALIGNED>
__device__ __forceinline__ void q4k_part(const uint8_t* __restrict__ blk, int i, float (&w)[8]) {
  const int c = i >> 3, hi = (i >> 2) & 1, l0 = 8 * (i & 3);
  uint8_t hdr[16];
  uint8_t qs[8];
  if constexpr (ALIGNED) {
    const uint4 h = __ldg(reinterpret_cast<const uint4*>(blk));
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 32 * c + l0));
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
    for (int k = 0; k < 16; ++k) hdr[k] = static_cast<uint8_t>(hw[k >> 2] >> (8 * (k & 3)));
#pragma unroll
    for (int k = 0; k < 8; ++k) qs[k] = static_cast<uint8_t>((k < 4 ? q.x : q.y) >> (8 * (k & 3)));
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) hdr[k] = __ldg(blk + k);
#pragma unroll
    for (int k = 0; k < 8; ++k) qs[k] = __ldg(blk + 16 + 32 * c + l0 + k);
  }
  const float d = half_bits(hdr[0] | (hdr[1] << 8));
  const float dmin = half_bits(hdr[2] | (hdr[3] << 8));
  auto word = [&](int o) -> uint32_t {
    return hdr[o] | (hdr[o + 1] << 8) | (hdr[o + 2] << 16) | (static_cast<uint32_t>(hdr[o + 3]) << 24);
  };
  uint32_t sc, mn;
  q4k_scale_min_rt(word(4), word(8), word(12), 2 * c + hi, sc, mn);
  const float d1 = d * static_cast<float>(sc);     // exact
  const float m1 = dmin * static_cast<float>(mn);  // exact
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = hi ? (qs[k] >> 4) : (qs[k] & 15);
    w[k] = __fmaf_rn(d1, static_cast<float>(q), -m1);  // d1*q exact: one rounding
  }
}

constexpr int kDqThreads = 256;

// Weights 4q .. 4q+3 of a 16-byte aligned super-block (q = 0..63): chunk c =
// q / 16, sub-block 2c (q % 16 < 8, low nibbles) or 2c + 1 (high nibbles),
// code bytes 32c + 4 (q % 8) .. + 3.
__device__ __forceinline__ float4 q4k_quad(const uint8_t* __restrict__ blk, uint4 h, int q) {
  const int c = q >> 4, hi = (q >> 3) & 1;
  const uint32_t codes = __ldg(reinterpret_cast<const uint32_t*>(blk + 16 + 32 * c + 4 * (q & 7)));
  uint32_t sc, mn;
  q4k_scale_min_rt(h.y, h.z, h.w, 2 * c + hi, sc, mn);
  const float d1 = half_bits(h.x) * static_cast<float>(sc);       // exact
  const float m1 = half_bits(h.x >> 16) * static_cast<float>(mn);  // exact
  const uint32_t v = hi ? codes >> 4 : codes;
  float4 r;
  r.x = __fmaf_rn(d1, static_cast<float>(v & 15), -m1);  // d1*q exact: one rounding
  r.y = __fmaf_rn(d1, static_cast<float>((v >> 8) & 15), -m1);
  r.z = __fmaf_rn(d1, static_cast<float>((v >> 16) & 15), -m1);
  r.w = __fmaf_rn(d1, static_cast<float>((v >> 24) & 15), -m1);
  return r;
}

// 16-byte aligned W and out: a warp per super-block and step, lane i writing
// weights 4i .. 4i+3 and 128 + 4i .. 128 + 4i + 3, so that each float4 store
// instruction covers 512 contiguous bytes (whole sectors).
__global__ void __launch_bounds__(kDqThreads) k_dequant_q4_k_vec(const uint8_t* __restrict__ W, int64_t nsuper,
                                                                 float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kDqThreads / 32);
  for (int64_t sb = static_cast<int64_t>(blockIdx.x) * (kDqThreads / 32) + (threadIdx.x >> 5); sb < nsuper;
       sb += warps) {
    const uint8_t* blk = W + sb * kSuperBytes;
    const uint4 h = __ldg(reinterpret_cast<const uint4*>(blk));  // d | dmin << 16, then the field words
    const float4 a = q4k_quad(blk, h, lane);
    const float4 b = q4k_quad(blk, h, 32 + lane);
    float4* dst = reinterpret_cast<float4*>(out + sb * kSuperWeights);
    dst[lane] = a;
    dst[32 + lane] = b;
  }
}

// Any alignment: one thread per 8 weights, 32 threads per super-block.
template <bool ALIGNED, bool VEC_OUT>
__global__ void __launch_bounds__(kDqThreads) k_dequant_q4_k(const uint8_t* __restrict__ W, int64_t nsuper,
                                                             float* __restrict__ out) {
  const int64_t parts = nsuper * 32;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kDqThreads;
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * kDqThreads + threadIdx.x; p < parts; p += stride) {
    const int64_t sb = p >> 5;
    const int i = static_cast<int>(p & 31);
    float w[8];
    q4k_part<ALIGNED>(W + sb * kSuperBytes, i, w);
    float* dst = out + sb * kSuperWeights + 8 * i;
    if constexpr (VEC_OUT) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) dst[k] = w[k];
    }
  }
}

// MUL_MAT for any alignment: one warp per weight row; lane i decodes its 8
// weights of each super-block once and applies them to every token (x loads
// of 8 consecutive floats, vector loads when X is 16-byte aligned).
template <bool ALIGNED, bool VEC_X>
__global__ void __launch_bounds__(256) k_mul_mat_q4_k(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                                      const float* __restrict__ X, int64_t N, float* __restrict__ Y) {
  constexpr int kTok = 8;
  const int lane = threadIdx.x & 31;
  const int64_t nsb = K / kSuperWeights;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t m = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint8_t* row = W + m * nsb * kSuperBytes;
    for (int64_t n0 = 0; n0 < N; n0 += kTok) {
      const int nt = static_cast<int>(N - n0 < kTok ? N - n0 : kTok);
      float acc[kTok] = {};
      for (int64_t sb = 0; sb < nsb; ++sb) {
        float w[8];
        q4k_part<ALIGNED>(row + sb * kSuperBytes, lane, w);
        const int64_t k0 = sb * kSuperWeights + 8 * lane;
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t < nt) {
            const float* xr = X + (n0 + t) * K + k0;
            float xv[8];
            if constexpr (VEC_X) {
              const float4 a = __ldg(reinterpret_cast<const float4*>(xr));
              const float4 b = __ldg(reinterpret_cast<const float4*>(xr) + 1);
              xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
              xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) xv[k] = __ldg(xr + k);
            }
            float a = acc[t];
#pragma unroll
            for (int k = 0; k < 8; ++k) a = fmaf(w[k], xv[k], a);
            acc[t] = a;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        if (lane == 0 && t < nt) Y[(n0 + t) * M + m] = a;
      }
    }
  }
}

}  // namespace

cudaError_t launch_dequant_q4_k(const uint8_t* W, int64_t nsuper, float* out, cudaStream_t s) {
  const int64_t want = (nsuper * 32 + kDqThreads - 1) / kDqThreads;
  const int grid = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>(want, static_cast<int64_t>(device_info().sm_count) * 8)));
  const bool a = (reinterpret_cast<uintptr_t>(W) & 15) == 0, v = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  if (a && v) {
    const int vgrid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>((nsuper + 7) / 8, static_cast<int64_t>(device_info().sm_count) * 8)));
    k_dequant_q4_k_vec<<<vgrid, kDqThreads, 0, s>>>(W, nsuper, out);
  } else if (a)
    k_dequant_q4_k<true, false><<<grid, kDqThreads, 0, s>>>(W, nsuper, out);
  else if (v)
    k_dequant_q4_k<false, true><<<grid, kDqThreads, 0, s>>>(W, nsuper, out);
  else
    k_dequant_q4_k<false, false><<<grid, kDqThreads, 0, s>>>(W, nsuper, out);
  return cudaGetLastError();
}

cudaError_t launch_mul_mat_q4_k(const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                                cudaStream_t s) {
  const int grid = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>((M + 7) / 8, static_cast<int64_t>(device_info().sm_count) * 16)));
  const bool a = (reinterpret_cast<uintptr_t>(W) & 15) == 0, v = (reinterpret_cast<uintptr_t>(X) & 15) == 0;
  if (a && v)
    k_mul_mat_q4_k<true, true><<<grid, 256, 0, s>>>(W, M, K, X, N, Y);
  else if (a)
    k_mul_mat_q4_k<true, false><<<grid, 256, 0, s>>>(W, M, K, X, N, Y);
  else if (v)
    k_mul_mat_q4_k<false, true><<<grid, 256, 0, s>>>(W, M, K, X, N, Y);
  else
    k_mul_mat_q4_k<false, false><<<grid, 256, 0, s>>>(W, M, K, X, N, Y);
  return cudaGetLastError();
}

}  // namespace gq
