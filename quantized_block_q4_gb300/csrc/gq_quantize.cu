// KQ: fp32 weights -> Q4_0 blocks, the step before MUL_MAT.
//
// Follows the block-quantisation formula q(w) = clip(round(w/s) + z, q_min,
// q_max), w_hat = s*(q - z) ("Architecture and module overview",
// weight-loading section) with z = 8 and q in [0, 15].  The pages leave the
// choice of s open; the rule used (the same one the library documents):
//   m = the weight of largest magnitude in the block, sign kept, the first on
//   ties; d = binary16(m / -8), round to nearest even (an all-zero block
//   stores d = +0); q = clip(rint(w / d) + 8, 0, 15) with the quotient an IEEE
//   fp32 division rounded to nearest even, q = 8 when d == 0 or the quotient is
//   NaN.  The low nibble of qs[j] is element j, the high nibble element j+16.
// One thread per block (the fp32 rows are contiguous and K % 32 == 0, so block
// b starts at float 32*b); a warp stages its 32 packed blocks (576 bytes) in
// shared memory and writes them out with coalesced 16-byte stores.  HBM-bound:
// 128 bytes read and 18 written per block.
#include <algorithm>
#include <cuda_fp16.h>

#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ void quantize_one(const float (&w)[32], uint8_t* dst) {
  float amax = 0.f, m = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float a = fabsf(w[j]);
    if (a > amax) {
      amax = a;
      m = w[j];
    }
  }
  const uint16_t d_bits = amax > 0.f ? __half_as_ushort(__float2half_rn(m / -8.0f)) : static_cast<uint16_t>(0);
  const float d = __half2float(__ushort_as_half(d_bits));
  // rint(w / d) with the IEEE quotient: w * RN(1/d) is within 2 ulps of the
  // rounded quotient (|w / d| <= 8.01), so the two can round to different
  // integers only next to a half-integer; there the division itself decides.
  const float r = __frcp_rn(d);
  uint32_t q[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (d == 0.f) {
      q[j] = 8;
    } else {
      float u = w[j] * r;
      float h = rintf(u);
      if (fabsf(u - h) > 0.5f - 1e-4f) h = rintf(__fdiv_rn(w[j], d));
      const float t = h + 8.0f;
      q[j] = (t != t) ? 8u : (t < 0.f ? 0u : (t > 15.f ? 15u : static_cast<uint32_t>(t)));
    }
  }
  // 18 bytes at an even offset: nine 16-bit stores
  uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
  d16[0] = d_bits;
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const uint32_t b0 = q[j] | (q[j + 16] << 4), b1 = q[j + 1] | (q[j + 17] << 4);
    d16[1 + j / 2] = static_cast<uint16_t>(b0 | (b1 << 8));
  }
}

__global__ void __launch_bounds__(kQThreads)
    k_quantize_q4_0(const float* __restrict__ W, int64_t nblocks, uint8_t* __restrict__ out, int vec_in,
                    int vec_out) {
  __shared__ __align__(16) uint8_t stage[kQThreads / 32][32 * 18];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b0 = (static_cast<int64_t>(blockIdx.x) * kQThreads) + warp * 32;  // first block of this warp
  const int64_t b = b0 + lane;
  if (b < nblocks) {
    float w[32];
    const float* src = W + b * 32;
    if (vec_in) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src) + i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = __ldg(src + i);
    }
    quantize_one(w, &stage[warp][lane * 18]);
  }
  __syncwarp();
  if (b0 >= nblocks) return;
  const int nb = nblocks - b0 < 32 ? static_cast<int>(nblocks - b0) : 32;
  uint8_t* dst = out + b0 * 18;
  if (vec_out && nb == 32) {  // 576 bytes, 16-byte aligned: 36 uint4
    const uint4* s4 = reinterpret_cast<const uint4*>(stage[warp]);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[lane] = s4[lane];
    if (lane < 4) d4[32 + lane] = s4[32 + lane];
  } else {
    for (int i = lane; i < nb * 18; i += 32) dst[i] = stage[warp][i];
  }
}

}  // namespace

cudaError_t launch_quantize(const float* W, int64_t M, int64_t K, uint8_t* out, cudaStream_t s) {
  const int64_t nblocks = M * (K / 32);
  const int64_t grid = (nblocks + kQThreads - 1) / kQThreads;
  const int vec_in = (reinterpret_cast<uintptr_t>(W) & 15) == 0;
  const int vec_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  k_quantize_q4_0<<<static_cast<unsigned>(grid), kQThreads, 0, s>>>(W, nblocks, out, vec_in, vec_out);
  return cudaGetLastError();
}

}  // namespace gq
