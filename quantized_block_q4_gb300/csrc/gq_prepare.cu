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

// One thread per 16 output bytes: byte j of prepared row r is byte j of the
// source row while j < K/32*18, then the zero-block pattern (00 00 88 .. 88).
__global__ void k_prepare_q4_0(const uint8_t* __restrict__ W, int64_t M, int64_t src_row_bytes,
                               int64_t row_stride, int64_t dst_row_bytes, uint8_t* __restrict__ out) {
  const int64_t chunks_per_row = dst_row_bytes / 16;
  const int64_t total = M * chunks_per_row;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = c / chunks_per_row, j0 = (c % chunks_per_row) * 16;
    const uint8_t* src = W + r * row_stride;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t v = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t j = j0 + 4 * q + b;
        const uint32_t byte = j < src_row_bytes ? src[j] : ((j % kBlockBytes) < 2 ? 0u : 0x88u);
        v |= byte << (8 * b);
      }
      w[q] = v;
    }
    *reinterpret_cast<uint4*>(out + r * dst_row_bytes + j0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

int64_t prepared_row_bytes(int64_t K) { return (K + 255) / 256 * 144; }

cudaError_t launch_prepare_q4_0(const uint8_t* W, int64_t M, int64_t K, int64_t row_stride, uint8_t* out,
                                cudaStream_t s) {
  const int64_t dst = prepared_row_bytes(K);
  const int64_t total = M * (dst / 16);
  const int grid = static_cast<int>(std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(device_info().sm_count) * 16));
  k_prepare_q4_0<<<grid > 0 ? grid : 1, 256, 0, s>>>(W, M, (K / kQK) * kBlockBytes, row_stride, dst, out);
  return cudaGetLastError();
}

}  // namespace gq
