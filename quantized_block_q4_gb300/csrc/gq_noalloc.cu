// gq_mul_mat_q4_0_noalloc: the tensor-core MUL_MAT with no device allocation.
//
// gq_mul_mat_q4_0 gets the bf16 copy of the activations that its tensor-core
// kernel reads from cudaMallocAsync.  Some callers cannot let a library do
// that: a serving process whose memory pool owns all device memory up front, a
// framework that hands out memory only from its own arena, or a hot loop that
// must never enter the driver's allocator.  For them this entry point keeps the
// bf16 copy in one fixed array compiled into the library:
//
//  * The array is a file-scope __device__ variable of kMaxElems bf16 values
//    (12 MiB).  It is reserved on each device where the library's kernels are
//    first loaded (lazily, on first use of the library on that device, under
//    CUDA's default lazy module loading) and stays until that device's context
//    is destroyed, whether or not this entry point is ever called.
//  * Host code may not use the array's name as a device address (on the host it
//    names a shadow variable).  The first call on a device, with that device
//    current, asks the runtime for the real address with cudaGetSymbolAddress
//    and caches it per device.  Make that first call before any stream capture
//    begins.  The cached address belongs to that context: resetting the device
//    (cudaDeviceReset) after the first call is not supported.
//  * All calls share the one array and it keeps whatever the last call wrote.
//    Each call overwrites the N*K elements it later reads, so nothing needs to
//    start at zero; calls whose work overlaps on the GPU (on different streams
//    or devices sharing a context) race on the array.
#include <mutex>

#include "gq.h"
#include "gq_internal.h"

namespace {

constexpr int64_t kMaxElems = int64_t(6) << 20;  // 6 Mi bf16 values = 12 MiB
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) uint16_t g_noalloc_x_bf16[kMaxElems];

namespace {

std::mutex g_mu;
uint16_t* g_addr[kMaxDevices] = {};

// Device address of the array on the current device (set up once per device).
gq_status scratch_address(uint16_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return gq::api_fail(GQ_ERR_CUDA, "gq_mul_mat_q4_0_noalloc: no usable current device");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_x_bf16);
    if (e != cudaSuccess || p == nullptr)
      return gq::api_fail(GQ_ERR_CUDA, "gq_mul_mat_q4_0_noalloc: cudaGetSymbolAddress of the static array failed");
    g_addr[dev] = static_cast<uint16_t*>(p);
  }
  *out = g_addr[dev];
  return GQ_OK;
}

}  // namespace

extern "C" gq_status gq_mul_mat_q4_0_noalloc(const void* W, int64_t M, int64_t K, const float* X, int64_t N,
                                             float* Y, void* stream) {
  gq::api_clear_error();
  gq_status st = gq::api_check_mm_shape(M, K, N);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!W || !X || !Y) return gq::api_fail(GQ_ERR_NULL, "gq_mul_mat_q4_0_noalloc: W, X and Y must not be NULL");
  if (K == 0 || K % 256)
    return gq::api_fail(GQ_ERR_SHAPE, "gq_mul_mat_q4_0_noalloc: needs K > 0 and K % 256 == 0");
  if (N * K > kMaxElems)
    return gq::api_fail(GQ_ERR_SHAPE,
                        "gq_mul_mat_q4_0_noalloc: N*K exceeds the static scratch (6291456 bf16 values, 12 MiB)");
  if (reinterpret_cast<uintptr_t>(W) % 16 || reinterpret_cast<uintptr_t>(X) % 4 ||
      reinterpret_cast<uintptr_t>(Y) % 4)
    return gq::api_fail(GQ_ERR_ALIGN, "gq_mul_mat_q4_0_noalloc: W must be 16-byte, X and Y 4-byte aligned");
  st = gq::api_check_device();
  if (st != GQ_OK) return st;
  uint16_t* xb = nullptr;
  st = scratch_address(&xb);
  if (st != GQ_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = gq::launch_f32_to_bf16(X, xb, N * K, s, gq::api_pdl());
  if (e != cudaSuccess) return gq::api_fail(GQ_ERR_CUDA, "gq_mul_mat_q4_0_noalloc: conversion launch failed");
  return gq::api_prefill_bf16(W, M, K, xb, N, Y, false, s);
}
