// The C ABI of include/gq.h: argument checks, dispatch, tensor maps, errors.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "gq.h"
#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {

__device__ uint32_t g_dev_error = 0;

namespace {

constexpr int kMaxDevices = 64;
thread_local std::string t_last_error;

std::atomic<int64_t> g_prefill_min_n{16};  // N >= 16: the tensor-core kernel is faster
std::atomic<int64_t> g_force_generic{0};
std::atomic<int64_t> g_wait_limit_ns{2000000000LL};
std::atomic<int64_t> g_early_w{0};
std::atomic<int64_t> g_decode_variant{0};
std::atomic<int64_t> g_pdl{1};
std::atomic<int64_t> g_moe_path{0};
std::atomic<int64_t> g_test_drop{0};

gq_status fail(gq_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gq_status fail(gq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

gq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D tiled tensor map: dim0 innermost (elements), dim1 rows, row stride in bytes.
gq_status make_tmap(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t row_stride, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d, dims %llu x %llu, box %u x %u)",
                static_cast<int>(r), static_cast<unsigned long long>(dim0), static_cast<unsigned long long>(dim1),
                box0, box1);
  return GQ_OK;
}

gq_status check_device() {
  const DeviceInfo& di = device_info();
  if (di.device < 0) return fail(GQ_ERR_CUDA, "no current CUDA device");
  if (!(di.cc_major == 10 && di.cc_minor == 3))
    return fail(GQ_ERR_UNSUPPORTED, "device %d is compute capability %d.%d; this library is built for sm_103a",
                di.device, di.cc_major, di.cc_minor);
  return GQ_OK;
}

// Shapes shared by the mul_mat entry points.  Kernels index with 32-bit ints.
gq_status check_mm_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K < 0 || N < 0)
    return fail(GQ_ERR_SHAPE, "negative size (M=%lld K=%lld N=%lld)", (long long)M, (long long)K, (long long)N);
  if (K % kQK) return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of 32", (long long)K);
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || K > lim || N > lim)
    return fail(GQ_ERR_SHAPE, "a size exceeds 2^31-1 (M=%lld K=%lld N=%lld)", (long long)M, (long long)K,
                (long long)N);
  // products must fit comfortably in 63 bits of bytes
  const unsigned __int128 wb = (unsigned __int128)M * (K / kQK) * kBlockBytes;
  const unsigned __int128 xb = (unsigned __int128)N * K * 4, yb = (unsigned __int128)N * M * 4;
  const unsigned __int128 cap = (unsigned __int128)1 << 62;
  if (wb > cap || xb > cap || yb > cap) return fail(GQ_ERR_SHAPE, "tensor size overflows");
  return GQ_OK;
}

}  // namespace

uint32_t* device_error_word() {
  static std::atomic<uint32_t*> ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  uint32_t* p = ptrs[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lk(mu);
    p = ptrs[dev].load(std::memory_order_relaxed);
    if (!p) {
      void* a = nullptr;
      if (cudaGetSymbolAddress(&a, g_dev_error) != cudaSuccess) return nullptr;
      p = static_cast<uint32_t*>(a);
      ptrs[dev].store(p, std::memory_order_release);
    }
  }
  return p;
}

const DeviceInfo& device_info() {
  static DeviceInfo infos[kMaxDevices];
  static std::atomic<bool> ready[kMaxDevices] = {};
  static std::mutex mu;
  static const DeviceInfo none;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return none;
  if (!ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev].load(std::memory_order_relaxed)) {
      DeviceInfo d;
      int v = 0;
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
      d.sm_count = v;
      cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
      cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
      cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      d.smem_optin = static_cast<size_t>(v);
      d.device = dev;
      infos[dev] = d;
      ready[dev].store(true, std::memory_order_release);
    }
  }
  return infos[dev];
}

namespace {
std::mutex g_attr_mu;
std::map<std::pair<const void*, int>, size_t> g_smem_set;                    // (kernel, device) -> bytes
std::map<std::tuple<const void*, int, int, size_t>, int> g_occupancy;        // (kernel, device, threads, smem)
}  // namespace

cudaError_t kernel_smem(const void* kernel, size_t bytes, bool max_shared) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  size_t& have = g_smem_set[{kernel, dev}];
  if (bytes <= have && (have > 0 || !max_shared)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (max_shared) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  have = std::max(have, bytes);
  return cudaSuccess;
}

cudaError_t kernel_occupancy(const void* kernel, int threads, size_t smem, int* blocks) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  auto it = g_occupancy.find({kernel, dev, threads, smem});
  if (it == g_occupancy.end()) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    it = g_occupancy.emplace(std::make_tuple(kernel, dev, threads, smem), occ > 0 ? occ : 1).first;
  }
  *blocks = it->second;
  return cudaSuccess;
}

// Stream-ordered scratch from a pool the library owns (one per device), which
// keeps freed memory for the next call instead of returning it to the driver
// at every synchronisation; the caller's own default pool is left alone.
static cudaMemPool_t scratch_pool() {
  static cudaMemPool_t pools[kMaxDevices];
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[dev] = p;
  }
  return pools[dev];
}

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
  cudaMemPool_t pool = scratch_pool();
  return pool ? cudaMallocFromPoolAsync(p, bytes, pool, s) : cudaMallocAsync(p, bytes, s);
}

cudaError_t scratch_free(void* p, cudaStream_t s) { return cudaFreeAsync(p, s); }

}  // namespace gq

using namespace gq;

// W_row_bytes: the stride of W's rows (K/32*18, or the prepared layout's
// ceil(K/256)*144, whose zero blocks pad each row to whole 256-k boxes).
static gq_status mul_mat_decode(const void* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                                cudaStream_t s, int64_t W_row_bytes = 0) {
  CUtensorMap tm;
  uint32_t bx = 0, by = 0;
  const int variant = static_cast<int>(g_decode_variant.load());
  decode_w_box(N, variant, &bx, &by);
  const uint64_t row_bytes =
      W_row_bytes > 0 ? static_cast<uint64_t>(W_row_bytes) : static_cast<uint64_t>(K / kQK) * kBlockBytes;
  gq_status st = make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, static_cast<uint64_t>(M), row_bytes,
                           bx, by, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;
  cudaError_t e = launch_decode(&tm, DecodeBox{bx, by}, X, N, M, K, Y, static_cast<uint64_t>(g_wait_limit_ns.load()),
                                static_cast<int>(g_early_w.load()), variant, static_cast<int>(g_pdl.load()), s);
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "decode launch");
}

// Kw: the width of W's rows in weights (K, or K rounded up to 256 for the
// prepared layout; x beyond K reads as zeros through the tensor map).
// x_static: the caller's promise (GQ_OPT_X_STATIC) about Xb; only for the
// entry point whose Xb is the caller's (the other paths convert X right before).
static gq_status mul_mat_prefill_bf16(const void* W, int64_t M, int64_t K, const uint16_t* Xb, int64_t N, float* Y,
                                      bool allow_scratch, cudaStream_t s, int type = GQ_TYPE_Q4_0, int64_t Kw = 0,
                                      bool x_static = false) {
  CUtensorMap tmW, tmX;
  uint32_t wbx, web, wby, xbk, xbr;
  if (Kw <= 0) Kw = K;
  prefill_boxes(N, M, Kw, allow_scratch, x_static && g_pdl.load() != 0, type, &wbx, &web, &wby, &xbk, &xbr);
  const uint64_t row_bytes = type_row_bytes(type, Kw);
  gq_status st = make_tmap(&tmW, web == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, W,
                           row_bytes / web, static_cast<uint64_t>(M), row_bytes, wbx, wby, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GQ_OK) return st;
  st = make_tmap(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xb, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                 static_cast<uint64_t>(K) * 2, xbk, xbr, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GQ_OK) return st;
  cudaError_t e = launch_prefill(&tmW, &tmX, N, M, Kw, Y, static_cast<uint64_t>(g_wait_limit_ns.load()), allow_scratch,
                                 static_cast<int>(g_early_w.load()), x_static ? 1 : 0, static_cast<int>(g_pdl.load()),
                                 s, type);
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "prefill launch");
}

namespace gq {
gq_status api_fail(gq_status st, const char* msg) { return fail(st, "%s", msg); }
int test_drop() { return static_cast<int>(g_test_drop.load()); }
void api_clear_error() { t_last_error.clear(); }
gq_status api_check_device() { return check_device(); }
int api_pdl() { return static_cast<int>(g_pdl.load()); }
gq_status api_check_mm_shape(int64_t M, int64_t K, int64_t N) { return check_mm_shape(M, K, N); }
gq_status api_prefill_bf16(const void* W, int64_t M, int64_t K, const uint16_t* X_bf16, int64_t N, float* Y,
                           bool allow_scratch, cudaStream_t s) {
  return mul_mat_prefill_bf16(W, M, K, X_bf16, N, Y, allow_scratch, s);
}
}  // namespace gq

extern "C" {

size_t gq_q4_0_nbytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0 || K % kQK) return 0;
  return static_cast<size_t>(M) * static_cast<size_t>(K / kQK) * kBlockBytes;
}

gq_status gq_dequant_q4_0(const void* W, int64_t M, int64_t K, float* out, void* stream) {
  t_last_error.clear();
  if (M < 0 || K < 0) return fail(GQ_ERR_SHAPE, "negative size");
  if (K % kQK) return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of 32", (long long)K);
  if (M == 0 || K == 0) return GQ_OK;
  if (!W || !out) return fail(GQ_ERR_NULL, "W and out must not be NULL");
  if ((unsigned __int128)M * K * 4 > ((unsigned __int128)1 << 62)) return fail(GQ_ERR_SHAPE, "size overflows");
  gq_status st = check_device();
  if (st != GQ_OK) return st;
  const int64_t nblocks = M * (K / kQK);
  auto s = static_cast<cudaStream_t>(stream);
  cudaError_t e = (aligned(W, 16) && aligned(out, 16))
                      ? launch_dequant_vec(static_cast<const uint8_t*>(W), nblocks, out, s)
                      : launch_dequant_bytes(static_cast<const uint8_t*>(W), nblocks, out, s);
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "dequant launch");
}

size_t gq_type_nbytes(gq_type type, int64_t M, int64_t K) {
  if (type_block_bytes(type) == 0 || M < 0 || K < 0 || K % type_block_weights(type)) return 0;
  return static_cast<size_t>(M) * static_cast<size_t>(type_row_bytes(type, K));
}

gq_status gq_dequant(gq_type type, const void* W, int64_t M, int64_t K, float* out, void* stream) {
  if (type == GQ_TYPE_Q4_0) return gq_dequant_q4_0(W, M, K, out, stream);
  t_last_error.clear();
  if (type_block_bytes(type) == 0) return fail(GQ_ERR_SHAPE, "unknown block type %d", static_cast<int>(type));
  if (M < 0 || K < 0) return fail(GQ_ERR_SHAPE, "negative size");
  const int bw = type_block_weights(type);
  if (K % bw) return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of %d", (long long)K, bw);
  if (M == 0 || K == 0) return GQ_OK;
  if (!W || !out) return fail(GQ_ERR_NULL, "W and out must not be NULL");
  if ((unsigned __int128)M * K * 4 > ((unsigned __int128)1 << 62)) return fail(GQ_ERR_SHAPE, "size overflows");
  if (!aligned(out, 4)) return fail(GQ_ERR_ALIGN, "out must be 4-byte aligned");
  gq_status st = check_device();
  if (st != GQ_OK) return st;
  cudaError_t e = type == GQ_TYPE_Q4_K
                      ? launch_dequant_q4_k(static_cast<const uint8_t*>(W), M * (K / bw), out,
                                            static_cast<cudaStream_t>(stream))
                      : launch_dequant_legacy(type, static_cast<const uint8_t*>(W), M * (K / kQK), out,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "dequant launch");
}

gq_status gq_validate(gq_type type, const void* W, int64_t M, int64_t K, uint64_t* result, void* stream) {
  t_last_error.clear();
  if (type_block_bytes(type) == 0) return fail(GQ_ERR_SHAPE, "unknown block type %d", static_cast<int>(type));
  if (M < 0 || K < 0) return fail(GQ_ERR_SHAPE, "negative size");
  const int bw = type_block_weights(type);
  if (K % bw) return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of %d", (long long)K, bw);
  if (!result) return fail(GQ_ERR_NULL, "result must not be NULL");
  if (!aligned(result, 8)) return fail(GQ_ERR_ALIGN, "result must be 8-byte aligned");
  if (M > 0 && K > 0 && !W) return fail(GQ_ERR_NULL, "W must not be NULL");
  if ((unsigned __int128)M * K > ((unsigned __int128)1 << 62)) return fail(GQ_ERR_SHAPE, "size overflows");
  gq_status st = check_device();
  if (st != GQ_OK) return st;
  cudaError_t e = launch_validate(static_cast<const uint8_t*>(W), M * (K / bw), type,
                                  reinterpret_cast<unsigned long long*>(result), static_cast<int>(g_pdl.load()),
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "validate launch");
}

gq_status gq_validate_q4_0(const void* W, int64_t M, int64_t K, uint64_t* result, void* stream) {
  return gq_validate(GQ_TYPE_Q4_0, W, M, K, result, stream);
}

gq_status gq_mul_mat(gq_type type, const void* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                     void* stream) {
  if (type == GQ_TYPE_Q4_0) return gq_mul_mat_q4_0(W, M, K, X, N, Y, stream);
  t_last_error.clear();
  if (type_block_bytes(type) == 0) return fail(GQ_ERR_SHAPE, "unknown block type %d", static_cast<int>(type));
  gq_status st = check_mm_shape(M, K, N);
  if (st != GQ_OK) return st;
  if (K % type_block_weights(type))
    return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of %d", (long long)K, type_block_weights(type));
  if (M == 0 || N == 0) return GQ_OK;
  if (!Y) return fail(GQ_ERR_NULL, "Y must not be NULL");
  st = check_device();
  if (st != GQ_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(N) * M * sizeof(float), s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "memset");
  }
  if (!W || !X) return fail(GQ_ERR_NULL, "W and X must not be NULL");
  if (!aligned(X, 4) || !aligned(Y, 4)) return fail(GQ_ERR_ALIGN, "X and Y must be 4-byte aligned");
  // Fast paths as for Q4_0: the mma.sync decode kernel below the tensor-core
  // threshold, the tcgen05 kernel from it on; the scalar kernel otherwise.
  const bool fast = K % 256 == 0 && aligned(W, 16) && aligned(X, 16) && aligned(Y, 16) && !g_force_generic.load();
  const bool tc = fast && N >= g_prefill_min_n.load();
  if (fast && !tc && N < 16) {
    // the decode kernel on this block format: a box row is 256 k of a weight
    // row (Q4_1 160 bytes, Q4_K 144; Q8_0's 272 bytes as 16-bit elements)
    CUtensorMap tm;
    const uint64_t row_bytes = type_row_bytes(type, K);
    const uint32_t box_bytes = static_cast<uint32_t>(type_row_bytes(type, 256));
    const bool wide = box_bytes > 256;
    st = make_tmap(&tm, wide ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, W,
                   row_bytes / (wide ? 2 : 1), static_cast<uint64_t>(M), row_bytes, box_bytes / (wide ? 2 : 1), 32,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != GQ_OK) return st;
    cudaError_t e = launch_decode_legacy(type, &tm, DecodeBox{box_bytes, 32}, X, N, M, K, Y, static_cast<uint64_t>(g_wait_limit_ns.load()),
                                         static_cast<int>(g_early_w.load()), static_cast<int>(g_pdl.load()), s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "decode launch");
  }
  if (!tc) {
    cudaError_t e = type == GQ_TYPE_Q4_K
                        ? launch_mul_mat_q4_k(static_cast<const uint8_t*>(W), M, K, X, N, Y, s)
                        : launch_mul_mat_legacy(type, static_cast<const uint8_t*>(W), M, K, X, N, Y,
                                                static_cast<uint64_t>(g_wait_limit_ns.load()), s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "mul_mat launch");
  }
  // X -> bf16 scratch, then the tensor-core kernel with this block format
  const size_t xbytes = static_cast<size_t>(N) * K * sizeof(uint16_t);
  void* xb = nullptr;
  cudaError_t e = scratch_alloc(&xb, xbytes, s);
  if (e != cudaSuccess) return fail(GQ_ERR_ALLOC, "scratch allocation (%zu bytes): %s", xbytes, cudaGetErrorString(e));
  e = launch_f32_to_bf16(X, static_cast<uint16_t*>(xb), N * K, s, static_cast<int>(g_pdl.load()));
  if (e != cudaSuccess) {
    scratch_free(xb, s);
    return cuda_fail(e, "f32->bf16 launch");
  }
  st = mul_mat_prefill_bf16(W, M, K, static_cast<const uint16_t*>(xb), N, Y, true, s, type);
  e = scratch_free(xb, s);
  if (st != GQ_OK) return st;
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "scratch free");
}

gq_status gq_quantize_q4_0(const float* W, int64_t M, int64_t K, void* out, void* stream) {
  t_last_error.clear();
  if (M < 0 || K < 0) return fail(GQ_ERR_SHAPE, "negative size");
  if (K % kQK) return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of 32", (long long)K);
  if (M == 0 || K == 0) return GQ_OK;
  if (!W || !out) return fail(GQ_ERR_NULL, "W and out must not be NULL");
  if (!aligned(W, 4)) return fail(GQ_ERR_ALIGN, "W must be 4-byte aligned");
  if ((unsigned __int128)M * K * 4 > ((unsigned __int128)1 << 62)) return fail(GQ_ERR_SHAPE, "size overflows");
  gq_status st = check_device();
  if (st != GQ_OK) return st;
  cudaError_t e = launch_quantize(W, M, K, static_cast<uint8_t*>(out), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "quantize launch");
}

gq_status gq_mul_mat_q4_0(const void* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y, void* stream) {
  t_last_error.clear();
  gq_status st = check_mm_shape(M, K, N);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!Y) return fail(GQ_ERR_NULL, "Y must not be NULL");
  st = check_device();
  if (st != GQ_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // empty sum
    cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(N) * M * sizeof(float), s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "memset");
  }
  if (!W || !X) return fail(GQ_ERR_NULL, "W and X must not be NULL");
  if (!aligned(X, 4) || !aligned(Y, 4)) return fail(GQ_ERR_ALIGN, "X and Y must be 4-byte aligned");

  const bool fast = (K % 256 == 0) && aligned(W, 16) && aligned(X, 16) && aligned(Y, 16);
  if (!fast || g_force_generic.load()) {
    cudaError_t e = launch_generic(static_cast<const uint8_t*>(W), M, K, X, N, Y, s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "generic launch");
  }
  if (N < g_prefill_min_n.load() && N <= 64) return mul_mat_decode(W, M, K, X, N, Y, s);

  // Prefill: X -> bf16 scratch (stream-ordered), then the tensor-core kernel.
  const size_t xbytes = static_cast<size_t>(N) * K * sizeof(uint16_t);
  void* xb = nullptr;
  cudaError_t e = scratch_alloc(&xb, xbytes, s);
  if (e != cudaSuccess) return fail(GQ_ERR_ALLOC, "scratch allocation (%zu bytes): %s", xbytes, cudaGetErrorString(e));
  e = launch_f32_to_bf16(X, static_cast<uint16_t*>(xb), N * K, s, static_cast<int>(g_pdl.load()));
  if (e != cudaSuccess) {
    scratch_free(xb, s);
    return cuda_fail(e, "f32->bf16 launch");
  }
  st = mul_mat_prefill_bf16(W, M, K, static_cast<const uint16_t*>(xb), N, Y, true, s);
  e = scratch_free(xb, s);
  if (st != GQ_OK) return st;
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "scratch free");
}

gq_status gq_mul_mat_id_q4_0(const void* W, int64_t n_expert, int64_t M, int64_t K, const float* X, int64_t n_ids,
                             const int32_t* ids, int64_t T, float* Y, void* stream) {
  t_last_error.clear();
  if (n_expert < 1) return fail(GQ_ERR_SHAPE, "n_expert=%lld must be >= 1", (long long)n_expert);
  if (n_ids < 0 || T < 0) return fail(GQ_ERR_SHAPE, "negative size (n_ids=%lld T=%lld)", (long long)n_ids, (long long)T);
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (n_ids > lim || T > lim || (T > 0 && n_ids > lim / T))
    return fail(GQ_ERR_SHAPE, "T*n_ids exceeds 2^31-1 (n_ids=%lld T=%lld)", (long long)n_ids, (long long)T);
  const int64_t P = T * n_ids;  // (token, slot) pairs
  gq_status st = check_mm_shape(M, K, P);
  if (st != GQ_OK) return st;
  if (n_expert > lim || (unsigned __int128)n_expert * M * (K / kQK) * kBlockBytes > ((unsigned __int128)1 << 62))
    return fail(GQ_ERR_SHAPE, "n_expert=%lld: weight size overflows", (long long)n_expert);
  if (M == 0 || P == 0) return GQ_OK;
  if (!Y || !ids) return fail(GQ_ERR_NULL, "ids and Y must not be NULL");
  if (K > 0 && (!W || !X)) return fail(GQ_ERR_NULL, "W and X must not be NULL");
  if (!aligned(X, 4) || !aligned(Y, 4) || !aligned(ids, 4))
    return fail(GQ_ERR_ALIGN, "X, Y and ids must be 4-byte aligned");
  st = check_device();
  if (st != GQ_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);

  const bool fast = K > 0 && K % 256 == 0 && aligned(W, 16) && aligned(X, 16) && aligned(Y, 16) &&
                    moe_route_supported(n_expert) && n_expert * M <= lim;
  if (!fast || g_force_generic.load()) {
    cudaError_t e = launch_generic_id(static_cast<const uint8_t*>(W), n_expert, M, K, X, ids, P, Y, s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "generic MUL_MAT_ID launch");
  }
  const int64_t used = std::min(n_expert, P);
  const int64_t path = g_moe_path.load();
  const bool tc = path == 2 || (path == 0 && P >= 16 * used);
  const int cap = decode_moe_cap(P, n_expert, T);
  const int64_t n_mtiles = (M + 127) / 128;
  if (tc && n_mtiles * ((P + kMoeBN - 1) / kMoeBN + used) > lim)
    return fail(GQ_ERR_SHAPE, "too many tensor-core work items");

  const uint64_t limit = static_cast<uint64_t>(g_wait_limit_ns.load());
  const int pdl = static_cast<int>(g_pdl.load());
  const uint64_t row_bytes = static_cast<uint64_t>(K / kQK) * kBlockBytes;
  if (!tc && cap == 1) {
    // A single token: every slot is a one-token group of its own, so the
    // decode kernel reads the ids itself -- no routing kernel, no scratch.
    MoeRoute rt{};
    rt.ids = ids;
    rt.np = static_cast<int32_t>(P);
    rt.ne = static_cast<int32_t>(n_expert);
    CUtensorMap tm;
    uint32_t bx = 0, by = 0;
    decode_moe_w_box(cap, &bx, &by);
    st = make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, static_cast<uint64_t>(n_expert * M), row_bytes,
                   bx, by, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != GQ_OK) return st;
    const cudaError_t e = launch_decode_moe(&tm, DecodeBox{bx, by}, X, cap, n_expert, M, K, P, rt, Y, limit, pdl, s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "MUL_MAT_ID decode launch");
  }

  const size_t route_bytes = (moe_route_ints(n_expert, P, cap) * sizeof(int32_t) + 255) / 256 * 256;
  const size_t xg_bytes = tc ? static_cast<size_t>(P) * K * sizeof(uint16_t) : 0;
  void* scratch = nullptr;
  cudaError_t e = scratch_alloc(&scratch, route_bytes + xg_bytes, s);
  if (e != cudaSuccess)
    return fail(GQ_ERR_ALLOC, "scratch allocation (%zu bytes): %s", route_bytes + xg_bytes, cudaGetErrorString(e));
  const MoeRoute rt = moe_route_layout(static_cast<int32_t*>(scratch), n_expert, P, cap);
  const char* what = "MUL_MAT_ID routing launch";
  e = launch_moe_route(ids, P, n_expert, n_mtiles, kMoeBN, cap, rt, Y, M, pdl, s);
  if (e == cudaSuccess && !tc) {
    CUtensorMap tm;
    uint32_t bx = 0, by = 0;
    decode_moe_w_box(cap, &bx, &by);
    st = make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, static_cast<uint64_t>(n_expert * M), row_bytes,
                   bx, by, CU_TENSOR_MAP_SWIZZLE_NONE);
    what = "MUL_MAT_ID decode launch";
    if (st == GQ_OK) e = launch_decode_moe(&tm, DecodeBox{bx, by}, X, cap, n_expert, M, K, P, rt, Y, limit, pdl, s);
  } else if (e == cudaSuccess) {
    uint16_t* xg = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(scratch) + route_bytes);
    CUtensorMap tmW, tmX;
    st = make_tmap(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, static_cast<uint64_t>(n_expert * M), row_bytes,
                   144, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == GQ_OK)
      st = make_tmap(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xg, static_cast<uint64_t>(K), static_cast<uint64_t>(P),
                     static_cast<uint64_t>(K) * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == GQ_OK) {
      what = "MUL_MAT_ID gather launch";
      e = launch_moe_gather_bf16(X, P, K, rt, xg, pdl, s);
      if (e == cudaSuccess) {
        what = "MUL_MAT_ID tensor-core launch";
        e = launch_prefill_moe(&tmW, &tmX, n_expert, M, K, P, rt, Y, limit, pdl, s);
      }
    }
  }
  const cudaError_t f = scratch_free(scratch, s);
  if (st != GQ_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, what);
  return f == cudaSuccess ? GQ_OK : cuda_fail(f, "scratch free");
}

size_t gq_prepared_q4_0_nbytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0 || K % kQK) return 0;
  return static_cast<size_t>(M) * static_cast<size_t>(prepared_row_bytes(K));
}

gq_status gq_prepare_q4_0(const void* W, int64_t M, int64_t K, int64_t row_stride, void* out, void* stream) {
  t_last_error.clear();
  if (M < 0 || K < 0) return fail(GQ_ERR_SHAPE, "negative size");
  if (K % kQK) return fail(GQ_ERR_SHAPE, "K=%lld is not a multiple of 32", (long long)K);
  const int64_t src_row = (K / kQK) * kBlockBytes;
  if (row_stride == 0) row_stride = src_row;
  if (row_stride < src_row)
    return fail(GQ_ERR_SHAPE, "row_stride=%lld is shorter than a row (%lld bytes)", (long long)row_stride,
                (long long)src_row);
  if (M == 0 || K == 0) return GQ_OK;
  if (!W || !out) return fail(GQ_ERR_NULL, "W and out must not be NULL");
  if (!aligned(out, 16)) return fail(GQ_ERR_ALIGN, "out must be 16-byte aligned");
  if ((unsigned __int128)M * row_stride > ((unsigned __int128)1 << 62)) return fail(GQ_ERR_SHAPE, "size overflows");
  if (prepared_row_bytes(K) > INT32_MAX)
    return fail(GQ_ERR_SHAPE, "K=%lld: a prepared row would exceed 2^31 bytes", (long long)K);
  gq_status st = check_device();
  if (st != GQ_OK) return st;
  cudaError_t e = launch_prepare_q4_0(static_cast<const uint8_t*>(W), M, K, row_stride, static_cast<uint8_t*>(out),
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "prepare launch");
}

gq_status gq_mul_mat_q4_0_prepared(const void* Wp, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                                   void* stream) {
  t_last_error.clear();
  gq_status st = check_mm_shape(M, K, N);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!Y) return fail(GQ_ERR_NULL, "Y must not be NULL");
  st = check_device();
  if (st != GQ_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(N) * M * sizeof(float), s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "memset");
  }
  if (!Wp || !X) return fail(GQ_ERR_NULL, "Wp and X must not be NULL");
  if (!aligned(Wp, 16) || !aligned(X, 16) || !aligned(Y, 16))
    return fail(GQ_ERR_ALIGN, "Wp, X and Y must be 16-byte aligned");
  const int64_t Kw = (K + 255) / 256 * 256;
  if (N < g_prefill_min_n.load() && N <= 64) return mul_mat_decode(Wp, M, K, X, N, Y, s, prepared_row_bytes(K));
  if (K < 256) {
    // Fewer than 256 terms: bf16 operands (relative 2^-9 each) do not average
    // below the 1e-3 * sum|w x| tolerance; the decode kernel (exact W, fp16 x)
    // runs in chunks of 64 tokens instead.
    for (int64_t n0 = 0; n0 < N; n0 += 64) {
      st = mul_mat_decode(Wp, M, K, X + n0 * K, std::min<int64_t>(64, N - n0), Y + n0 * M, s, prepared_row_bytes(K));
      if (st != GQ_OK) return st;
    }
    return GQ_OK;
  }
  const size_t xbytes = static_cast<size_t>(N) * K * sizeof(uint16_t);
  void* xb = nullptr;
  cudaError_t e = scratch_alloc(&xb, xbytes, s);
  if (e != cudaSuccess) return fail(GQ_ERR_ALLOC, "scratch allocation (%zu bytes): %s", xbytes, cudaGetErrorString(e));
  e = launch_f32_to_bf16(X, static_cast<uint16_t*>(xb), N * K, s, static_cast<int>(g_pdl.load()));
  if (e != cudaSuccess) {
    scratch_free(xb, s);
    return cuda_fail(e, "f32->bf16 launch");
  }
  st = mul_mat_prefill_bf16(Wp, M, K, static_cast<const uint16_t*>(xb), N, Y, true, s, GQ_TYPE_Q4_0, Kw);
  e = scratch_free(xb, s);
  if (st != GQ_OK) return st;
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "scratch free");
}

gq_status gq_mul_mat_q4_0_bf16x(const void* W, int64_t M, int64_t K, const uint16_t* X_bf16, int64_t N, float* Y,
                                void* stream) {
  t_last_error.clear();
  gq_status st = check_mm_shape(M, K, N);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!Y) return fail(GQ_ERR_NULL, "Y must not be NULL");
  st = check_device();
  if (st != GQ_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(N) * M * sizeof(float), s);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e, "memset");
  }
  if (!W || !X_bf16) return fail(GQ_ERR_NULL, "W and X_bf16 must not be NULL");
  if (K % 256) return fail(GQ_ERR_SHAPE, "the bf16-activation path needs K %% 256 == 0 (K=%lld)", (long long)K);
  if (!aligned(W, 16) || !aligned(X_bf16, 16) || !aligned(Y, 16))
    return fail(GQ_ERR_ALIGN, "W, X_bf16 and Y must be 16-byte aligned");
  return mul_mat_prefill_bf16(W, M, K, X_bf16, N, Y, true, s, GQ_TYPE_Q4_0, 0, get_decode_x_static() != 0);
}

gq_status gq_f32_to_bf16(const float* x, uint16_t* y, int64_t n, void* stream) {
  t_last_error.clear();
  if (n < 0) return fail(GQ_ERR_SHAPE, "negative size");
  if (n == 0) return GQ_OK;
  if (!x || !y) return fail(GQ_ERR_NULL, "x and y must not be NULL");
  if (!aligned(x, 4) || !aligned(y, 2)) return fail(GQ_ERR_ALIGN, "x must be 4-byte and y 2-byte aligned");
  gq_status st = check_device();
  if (st != GQ_OK) return st;
  cudaError_t e = launch_f32_to_bf16(x, y, n, static_cast<cudaStream_t>(stream), static_cast<int>(g_pdl.load()));
  return e == cudaSuccess ? GQ_OK : cuda_fail(e, "f32->bf16 launch");
}

gq_status gq_sync_status(void* stream) {
  t_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t* w = device_error_word();
  if (!w) return fail(GQ_ERR_CUDA, "device error word unavailable");
  uint32_t v = 0;
  e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (v) {
    const uint32_t zero = 0;
    cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (v & DEVERR_TIMEOUT)
      return fail(GQ_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait gave up (device error bits 0x%x)", v);
    return fail(GQ_ERR_BAD_INDEX, "an expert id was outside [0, n_expert) (device error bits 0x%x)", v);
  }
  return GQ_OK;
}

gq_status gq_set_option(gq_option opt, int64_t value) {
  t_last_error.clear();
  switch (opt) {
    case GQ_OPT_PREFILL_MIN_N:
      if (value < 1) return fail(GQ_ERR_SHAPE, "prefill threshold must be >= 1");
      g_prefill_min_n = value;
      return GQ_OK;
    case GQ_OPT_FORCE_GENERIC:
      g_force_generic = value ? 1 : 0;
      return GQ_OK;
    case GQ_OPT_WAIT_LIMIT_NS:
      if (value < 1000) return fail(GQ_ERR_SHAPE, "wait limit must be >= 1000 ns");
      g_wait_limit_ns = value;
      return GQ_OK;
    case GQ_OPT_WEIGHTS_STATIC:
      g_early_w = value ? 1 : 0;
      return GQ_OK;
    case GQ_OPT_DECODE_VARIANT:
      if (value < 0 || value > 4) return fail(GQ_ERR_SHAPE, "decode variant must be 0..4");
      g_decode_variant = value;
      return GQ_OK;
    case GQ_OPT_PDL:
      g_pdl = value ? 1 : 0;
      return GQ_OK;
    case GQ_OPT_PREFILL_TILE_N:
      if (value != 0 && value != 128 && value != 256) return fail(GQ_ERR_SHAPE, "tile width must be 0, 128 or 256");
      set_prefill_bn_override(static_cast<int>(value));
      return GQ_OK;
    case GQ_OPT_PREFILL_PAIR:
      set_prefill_pair_mode(static_cast<int>(value));
      return GQ_OK;
    case GQ_OPT_PREFILL_STREAMK:
      if (value < 0 || value > 4096) return fail(GQ_ERR_SHAPE, "k-split setting must be 0..4096");
      set_prefill_streamk(value);
      return GQ_OK;
    case GQ_OPT_PREFILL_SLOTS:
      if (value < 0 || value > 65536) return fail(GQ_ERR_SHAPE, "slot count must be 0..65536");
      set_prefill_slots(value);
      return GQ_OK;
    case GQ_OPT_DECODE_EARLY_STAGES:
      if (value < 1 || value > 64) return fail(GQ_ERR_SHAPE, "early stage count must be 1..64");
      set_decode_early_stages(static_cast<int>(value));
      return GQ_OK;
    case GQ_OPT_X_STATIC:
      set_decode_x_static(static_cast<int>(value));
      return GQ_OK;
    case GQ_OPT_MOE_PATH:
      if (value < 0 || value > 2) return fail(GQ_ERR_SHAPE, "MUL_MAT_ID path must be 0, 1 or 2");
      g_moe_path = value;
      return GQ_OK;
    case GQ_OPT_TEST_DROP_ARRIVE:
      if (value < 0 || value > 2) return fail(GQ_ERR_SHAPE, "test drop must be 0 (off), 1 (decode) or 2 (tensor core)");
      g_test_drop = value;
      return GQ_OK;
  }
  return fail(GQ_ERR_SHAPE, "unknown option %d", static_cast<int>(opt));
}

int64_t gq_get_option(gq_option opt) {
  switch (opt) {
    case GQ_OPT_PREFILL_MIN_N: return g_prefill_min_n.load();
    case GQ_OPT_FORCE_GENERIC: return g_force_generic.load();
    case GQ_OPT_WAIT_LIMIT_NS: return g_wait_limit_ns.load();
    case GQ_OPT_WEIGHTS_STATIC: return g_early_w.load();
    case GQ_OPT_DECODE_VARIANT: return g_decode_variant.load();
    case GQ_OPT_PDL: return g_pdl.load();
    case GQ_OPT_PREFILL_TILE_N: return get_prefill_bn_override();
    case GQ_OPT_PREFILL_PAIR: return get_prefill_pair_mode();
    case GQ_OPT_PREFILL_STREAMK: return get_prefill_streamk();
    case GQ_OPT_PREFILL_SLOTS: return get_prefill_slots();
    case GQ_OPT_DECODE_EARLY_STAGES: return get_decode_early_stages();
    case GQ_OPT_X_STATIC: return get_decode_x_static();
    case GQ_OPT_MOE_PATH: return g_moe_path.load();
    case GQ_OPT_TEST_DROP_ARRIVE: return g_test_drop.load();
  }
  return -1;
}

const char* gq_last_error(void) { return t_last_error.c_str(); }

const char* gq_status_string(gq_status s) {
  switch (s) {
    case GQ_OK: return "GQ_OK";
    case GQ_ERR_NULL: return "GQ_ERR_NULL";
    case GQ_ERR_SHAPE: return "GQ_ERR_SHAPE";
    case GQ_ERR_ALIGN: return "GQ_ERR_ALIGN";
    case GQ_ERR_CUDA: return "GQ_ERR_CUDA";
    case GQ_ERR_ALLOC: return "GQ_ERR_ALLOC";
    case GQ_ERR_DEVICE_TIMEOUT: return "GQ_ERR_DEVICE_TIMEOUT";
    case GQ_ERR_UNSUPPORTED: return "GQ_ERR_UNSUPPORTED";
    case GQ_ERR_BAD_INDEX: return "GQ_ERR_BAD_INDEX";
  }
  return "unknown gq_status";
}

int gq_version(void) { return 100; }

}  // extern "C"
