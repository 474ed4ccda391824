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
// b starts at float 32*b); a warp reads its 32 blocks (4 KB) with coalesced
// 16-byte loads through shared memory, and stages its 32 packed blocks (576
// bytes) there to write them out with coalesced 16-byte stores.  HBM-bound:
// 128 bytes read and 18 written per block.
#include <algorithm>
#include <cuda_fp16.h>

#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kQThreads = 256;

// The exact quotient's code, for the rare element whose w * RN(1/d) lies next
// to a half-integer (out of line, so that the usual loop stays short).
__device__ __noinline__ uint32_t code_by_division(float w, float d) {
  const int qi = __float2int_rn(__fdiv_rn(w, d)) + 8;  // a NaN quotient converts to 0: code 8
  return static_cast<uint32_t>(min(max(qi, 0), 15));
}

__device__ __forceinline__ void quantize_one(const float (&w)[32], uint8_t* dst) {
  // m: the first weight of largest magnitude (NaNs never win the comparison)
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(w[j]));
  float m = 0.f;
#pragma unroll
  for (int j = 31; j >= 0; --j) m = fabsf(w[j]) == amax ? w[j] : m;
  const uint16_t d_bits = amax > 0.f ? __half_as_ushort(__float2half_rn(m / -8.0f)) : static_cast<uint16_t>(0);
  const float d = __half2float(__ushort_as_half(d_bits));
  uint32_t packed[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};  // d == 0: every code 8
  if (d != 0.f) {
    // rint(w / d) with the IEEE quotient: w * RN(1/d) is within 2 ulps of the
    // rounded quotient (|w / d| <= 8.01), so the two can round to different
    // integers only next to a half-integer; there the division itself decides.
    // A NaN quotient (w NaN, or w and d infinite) converts to 0: code 8.
    const float r = __frcp_rn(d);
    uint32_t q[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float u = w[j] * r;
      const float h = rintf(u);
      if (fabsf(u - h) > 0.5f - 1e-4f) {
        q[j] = code_by_division(w[j], d);
      } else {
        const int qi = static_cast<int>(h) + 8;
        q[j] = static_cast<uint32_t>(min(max(qi, 0), 15));
      }
    }
    // byte b of the codes: element b in the low nibble, element b + 16 in the high one
#pragma unroll
    for (int i = 0; i < 4; ++i)
      packed[i] = (q[4 * i] | (q[4 * i + 16] << 4)) | ((q[4 * i + 1] | (q[4 * i + 17] << 4)) << 8) |
                  ((q[4 * i + 2] | (q[4 * i + 18] << 4)) << 16) | ((q[4 * i + 3] | (q[4 * i + 19] << 4)) << 24);
  }
  // 18 bytes at an even offset: nine 16-bit stores
  uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
  d16[0] = d_bits;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    d16[1 + 2 * i] = static_cast<uint16_t>(packed[i]);
    d16[2 + 2 * i] = static_cast<uint16_t>(packed[i] >> 16);
  }
}

__global__ void __launch_bounds__(kQThreads)
    k_quantize_q4_0(const float* __restrict__ W, int64_t nblocks, uint8_t* __restrict__ out, int vec_in,
                    int vec_out) {
  __shared__ __align__(16) uint8_t stage[kQThreads / 32][32 * 18];
  // A warp's 32 blocks of fp32 weights, read with coalesced 16-byte loads;
  // rows padded to 36 floats, so that both the row-major writes and each
  // lane's reads of its own block are free of bank conflicts.
  __shared__ __align__(16) float xin[kQThreads / 32][32 * 36];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b0 = (static_cast<int64_t>(blockIdx.x) * kQThreads) + warp * 32;  // first block of this warp
  const int64_t b = b0 + lane;
  if (vec_in && b0 + 32 <= nblocks) {
    const float4* src4 = reinterpret_cast<const float4*>(W + b0 * 32);  // 1024 contiguous floats
    float* xs = xin[warp];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = 4 * (32 * i + lane);  // first float of this load within the warp's blocks
      *reinterpret_cast<float4*>(xs + (f >> 5) * 36 + (f & 31)) = __ldg(src4 + 32 * i + lane);
    }
    __syncwarp();
    float w[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(xs + lane * 36 + 4 * i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    quantize_one(w, &stage[warp][lane * 18]);
  } else if (b < nblocks) {
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
