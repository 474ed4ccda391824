// KP: the GPU repack of Q4_0 weights for the fast kernels.
//
// ggml rows may carry a padded stride (nb[1]) and K need only be a multiple of
// 32 ("ggml compute graph and memory allocator", the ggml_tensor section on
// ne/nb; "Binding GGUF weights to the compute graph", section 2.3).  The TMA
// kernels want rows whose width is a multiple of 256 weights (8 blocks = 144
// bytes = 9 x 16 bytes, so every row and every 256-k box is 16-byte aligned).
// gq_prepare_q4_0 copies each row into that layout and appends zero blocks
// (d = +0, every code 8: weights +0) up to the next multiple of 256 weights.
// The block bytes are copied unchanged, so the prepared matrix holds the same
// weights; the zero blocks meet zero x in the kernels and add exact zeros.
#include <algorithm>

#include "gq_internal.h"

namespace gq {
namespace {

// Byte j of a prepared row: byte j of the source row while j < K/32*18, then
// the zero-block pattern (00 00 88 .. 88; the source row is whole blocks, so
// j % 18 is the byte's place in its block).
__device__ __forceinline__ uint32_t prepared_byte(const uint8_t* src, int j, int src_row_bytes) {
  return j < src_row_bytes ? src[j] : (static_cast<uint32_t>(j) % kBlockBytes < 2 ? 0u : 0x88u);
}

// One warp per row, a lane per 16 output bytes at a time.  WORDS: the source
// rows start 4-byte aligned (W and the row stride), so every 16 bytes that lie
// inside the source row come as four word loads; the rest of the row (the
// source's last partial 16 bytes and the zero blocks, under 160 bytes) goes
// byte by byte.
constexpr int kPrepWarps = 8;
template <bool WORDS>
__global__ void __launch_bounds__(32 * kPrepWarps)
    k_prepare_q4_0(const uint8_t* __restrict__ W, int64_t M, int src_row_bytes, int64_t row_stride,
                   int dst_row_bytes, uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int words_end = WORDS ? src_row_bytes / 16 * 16 : 0;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kPrepWarps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kPrepWarps + (threadIdx.x >> 5); r < M; r += warps) {
    const uint8_t* src = W + r * row_stride;
    uint8_t* dst = out + r * dst_row_bytes;
#pragma unroll 4
    for (int j0 = 16 * lane; j0 < words_end; j0 += 16 * 32) {
      const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src + j0);
      *reinterpret_cast<uint4*>(dst + j0) = make_uint4(__ldg(s4), __ldg(s4 + 1), __ldg(s4 + 2), __ldg(s4 + 3));
    }
    for (int j0 = words_end + 16 * lane; j0 < dst_row_bytes; j0 += 16 * 32) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) v |= prepared_byte(src, j0 + 4 * q + b, src_row_bytes) << (8 * b);
        w[q] = v;
      }
      *reinterpret_cast<uint4*>(dst + j0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

int64_t prepared_row_bytes(int64_t K) { return (K + 255) / 256 * 144; }

cudaError_t launch_prepare_q4_0(const uint8_t* W, int64_t M, int64_t K, int64_t row_stride, uint8_t* out,
                                cudaStream_t s) {
  const int dst = static_cast<int>(prepared_row_bytes(K));
  const int src = static_cast<int>((K / kQK) * kBlockBytes);
  const int grid = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>((M + kPrepWarps - 1) / kPrepWarps, static_cast<int64_t>(device_info().sm_count) * 16)));
  const bool words = (reinterpret_cast<uintptr_t>(W) & 3) == 0 && row_stride % 4 == 0;
  if (words)
    k_prepare_q4_0<true><<<grid, 32 * kPrepWarps, 0, s>>>(W, M, src, row_stride, dst, out);
  else
    k_prepare_q4_0<false><<<grid, 32 * kPrepWarps, 0, s>>>(W, M, src, row_stride, dst, out);
  return cudaGetLastError();
}

}  // namespace gq
