// K0: fp32 -> bf16 conversion of the activations, and K3: the prefill
// MUL_MAT on tcgen05 tensor cores (in progress).
#include <algorithm>
#include <cuda_bf16.h>

#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {
namespace {

// 8 elements per thread per step: two float4 loads, one 16-byte store.
__global__ void k_f32_to_bf16(const float* __restrict__ x, uint16_t* __restrict__ y, int64_t n) {
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

cudaError_t launch_f32_to_bf16(const float* x, uint16_t* y, int64_t n, cudaStream_t s) {
  const int64_t work = (n + 7) / 8;
  const int grid =
      static_cast<int>(std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(device_info().sm_count) * 8));
  k_f32_to_bf16<<<grid > 0 ? grid : 1, 256, 0, s>>>(x, y, n);
  return cudaGetLastError();
}

void prefill_boxes(uint32_t* w_box_x_bytes, uint32_t* w_box_rows, uint32_t* x_box_k, uint32_t* x_box_rows) {
  *w_box_x_bytes = 144;
  *w_box_rows = 128;
  *x_box_k = 64;
  *x_box_rows = 256;
}

cudaError_t launch_prefill(const CUtensorMap*, const CUtensorMap*, int64_t, int64_t, int64_t, float*, uint64_t,
                           cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace gq
