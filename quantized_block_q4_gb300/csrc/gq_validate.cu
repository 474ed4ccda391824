// KV: row-data validation of block-quantised weights ("GGUF loading, mmap
// and tensor placement", the section on --check-tensors and parallel
// validation: ggml_validate_row_data checks each row's scale factors and
// integers).  Reading: a block is invalid when one of its
// fp16 scale fields is NaN or infinite (exponent bits all ones) -- d for
// every format, m for Q4_1 and Q5_1 and dmin for Q4_K; the 4-, 5-, 6- and 8-bit
// fields are always valid.  A Q4_K block is a 256-weight super-block.
//
// One pass over the flat block array (rows are contiguous, so row boundaries
// do not matter): each thread tests the blocks it strides over with byte
// loads of the scales' high bytes (any alignment), a warp sums its count and
// takes its smallest bad index with shuffles, and lane 0 folds them into the
// caller's result with one 64-bit atomic add and one atomic min.  Every sector of W
// holds a scale byte, so the pass streams the whole matrix: HBM-bound at the
// weight bytes.  A one-thread kernel resets the result first; under
// programmatic dependent launch the scan starts while it runs and waits for
// it only before its atomics.
#include <algorithm>

#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {
namespace {

constexpr int kVThreads = 256;

// An fp16 value is NaN or infinite exactly when its five exponent bits (bits
// 10..14, i.e. bits 2..6 of the little-endian high byte) are all ones.
__device__ __forceinline__ bool half_not_finite(uint32_t hi_byte) { return (hi_byte & 0x7Cu) == 0x7Cu; }

// Waits for the kernel before (which may still read the previous result, and
// which the scan must follow), then lets the scan start.
__global__ void k_validate_init(unsigned long long* __restrict__ result) {
  pdl_wait();
  pdl_launch_dependents();
  result[0] = 0ull;
  result[1] = ~0ull;
}

__global__ void __launch_bounds__(kVThreads)
    k_validate(const uint8_t* __restrict__ W, uint64_t nblocks, int block_bytes, int check_min,
               unsigned long long* __restrict__ result) {
  unsigned long long count = 0, first = ~0ull;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kVThreads;
  for (uint64_t b = static_cast<uint64_t>(blockIdx.x) * kVThreads + threadIdx.x; b < nblocks; b += stride) {
    const uint8_t* p = W + b * static_cast<uint64_t>(block_bytes);
    bool bad = half_not_finite(__ldg(p + 1));
    if (check_min) bad |= half_not_finite(__ldg(p + 3));
    if (bad) {
      ++count;
      first = first < b ? first : b;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    count += __shfl_xor_sync(0xFFFFFFFFu, count, o);
    const unsigned long long f = __shfl_xor_sync(0xFFFFFFFFu, first, o);
    first = f < first ? f : first;
  }
  pdl_wait();  // the reset of the result has landed
  if ((threadIdx.x & 31) == 0 && count) {
    atomicAdd(&result[0], count);
    atomicMin(&result[1], first);
  }
}

}  // namespace

cudaError_t launch_validate(const uint8_t* W, int64_t nblocks, int type, unsigned long long* result, int pdl,
                            cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_validate_init, result);
  if (e != cudaSuccess || nblocks == 0) return e;
  const int64_t want = (nblocks + kVThreads - 1) / kVThreads;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(want, static_cast<int64_t>(device_info().sm_count) * 8)));
  cfg.blockDim = dim3(kVThreads);
  // Q4_1's and Q5_1's min offset and Q4_K's dmin sit in bytes 2-3, as the second fp16 field
  return cudaLaunchKernelEx(&cfg, k_validate, W, static_cast<uint64_t>(nblocks), type_block_bytes(type),
                            (type == GQ_TYPE_Q4_1 || type == GQ_TYPE_Q4_K || type == GQ_TYPE_Q5_1) ? 1 : 0, result);
}

}  // namespace gq
