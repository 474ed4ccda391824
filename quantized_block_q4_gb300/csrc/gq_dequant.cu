// K1: Q4_0 blocks -> fp32 weights, bit-exact.
//
// Block layout ("Binding GGUF weights to the compute graph", section 2.3):
// ggml_half d, then uint8_t qs[16]; 18 bytes per 32 weights.  Decoding follows
// w = d*(q - 8) with the low nibble of qs[j] as element j and the high nibble
// as element j+16.  The product of an fp16 value (11 significant bits) and an
// integer in [-8, 7] fits in fp32 exactly, so the result is independent of
// rounding mode; d*(q-8) is evaluated literally so that q = 8 with d < 0 gives
// -0.0.
//
// The W matrix is contiguous, so row boundaries do not matter here: the kernel
// walks the flat block array.  Eight blocks are 144 bytes = 9 x 16 bytes, so
// tiles of whole 8-block groups keep every global load 16-byte aligned when W
// is.  A tile is staged through shared memory with coalesced 16-byte loads;
// each thread then emits float4 outputs, consecutive threads writing
// consecutive 16-byte chunks (the kernel is bound by these writes: 128 bytes
// out per 18 bytes in).
#include <algorithm>
#include <cuda_fp16.h>

#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kThreads = 256;
constexpr int kTileBlocks = 256;                       // 32 groups of 8 blocks
constexpr int kTileBytes = kTileBlocks * kBlockBytes;  // 4608 = 288 x 16

__device__ __forceinline__ float dq(float d, uint32_t q) { return d * static_cast<float>(static_cast<int>(q) - 8); }

__global__ void __launch_bounds__(kThreads) k_dequant_vec(const uint8_t* __restrict__ W, int64_t nblocks,
                                                          float* __restrict__ out) {
  __shared__ __align__(16) uint8_t tile[kTileBytes];
  const int64_t ntiles = (nblocks + kTileBlocks - 1) / kTileBlocks;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t b0 = t * kTileBlocks;
    const int nb = static_cast<int>(nblocks - b0 < kTileBlocks ? nblocks - b0 : kTileBlocks);
    const int nbytes = nb * kBlockBytes;
    const uint8_t* src = W + b0 * kBlockBytes;  // 16-byte aligned: b0 is a multiple of 8 blocks
    __syncthreads();
    for (int c = threadIdx.x; c * 16 < nbytes; c += kThreads) {
      if (c * 16 + 16 <= nbytes) {
        *reinterpret_cast<uint4*>(tile + c * 16) = __ldg(reinterpret_cast<const uint4*>(src + c * 16));
      } else {
        for (int i = c * 16; i < nbytes; ++i) tile[i] = src[i];
      }
    }
    __syncthreads();
    // nb * 8 float4 outputs: o -> block o/8, part o%8 (elements 4*part .. 4*part+3)
    float4* dst = reinterpret_cast<float4*>(out + b0 * kQK);
    for (int o = threadIdx.x; o < nb * 8; o += kThreads) {
      const int b = o >> 3, part = o & 7;
      const uint8_t* blk = tile + b * kBlockBytes;
      const uint16_t dbits = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
      const float d = __half2float(__ushort_as_half(dbits));
      const uint8_t* q = blk + 2 + 4 * (part & 3);
      const int sh = (part & 4) ? 4 : 0;  // parts 4..7 are the high nibbles (elements 16..31)
      float4 v;
      v.x = dq(d, (q[0] >> sh) & 0xF);
      v.y = dq(d, (q[1] >> sh) & 0xF);
      v.z = dq(d, (q[2] >> sh) & 0xF);
      v.w = dq(d, (q[3] >> sh) & 0xF);
      dst[o] = v;
    }
  }
}

// Any alignment: one thread per block, byte loads, scalar stores.
__global__ void k_dequant_bytes(const uint8_t* __restrict__ W, int64_t nblocks, float* __restrict__ out) {
  for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < nblocks;
       b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint8_t* blk = W + b * kBlockBytes;
    const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(blk[0] | (blk[1] << 8))));
    float* o = out + b * kQK;
    for (int j = 0; j < 16; ++j) {
      const uint32_t byte = blk[2 + j];
      o[j] = dq(d, byte & 0xF);
      o[j + 16] = dq(d, byte >> 4);
    }
  }
}

}  // namespace

cudaError_t launch_dequant_vec(const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s) {
  const int64_t ntiles = (nblocks + kTileBlocks - 1) / kTileBlocks;
  const int grid = static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(device_info().sm_count) * 8));
  k_dequant_vec<<<grid, kThreads, 0, s>>>(W, nblocks, out);
  return cudaGetLastError();
}

cudaError_t launch_dequant_bytes(const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s) {
  const int grid =
      static_cast<int>(std::min<int64_t>((nblocks + 255) / 256, static_cast<int64_t>(device_info().sm_count) * 16));
  k_dequant_bytes<<<grid, 256, 0, s>>>(W, nblocks, out);
  return cudaGetLastError();
}

}  // namespace gq
