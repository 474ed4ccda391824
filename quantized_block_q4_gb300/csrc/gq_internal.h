// Internal interface between the C ABI (gq_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gq.h"

namespace gq {

constexpr int kQK = 32;          // weights per block_q4_0
constexpr int kBlockBytes = 18;  // fp16 d + 16 bytes of codes

// Device-side error word (defined in gq_api.cu).
uint32_t* device_error_word();

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};
const DeviceInfo& device_info();  // current device, cached

// Kernel launch attributes of the current device, set once per (kernel,
// device) and cached; safe to call from several host threads at once.
// Raise the kernel's dynamic shared-memory limit to at least `bytes` (and, with
// max_shared, prefer all of the unified L1 / shared storage as shared memory).
cudaError_t kernel_smem(const void* kernel, size_t bytes, bool max_shared);
// Resident blocks per SM for `threads` threads and `smem` bytes (at least 1).
cudaError_t kernel_occupancy(const void* kernel, int threads, size_t smem, int* blocks);

// Stream-ordered scratch from the library's own per-device pool (gq_api.cu).
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s);
cudaError_t scratch_free(void* p, cudaStream_t s);

// ---- K1: Q4_0 blocks -> fp32, bit-exact (gq_dequant.cu)
cudaError_t launch_dequant_vec(const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s);
cudaError_t launch_dequant_bytes(const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s);

// ---- K2: decode / small-N mul_mat (gq_decode.cu).  Needs K % 256 == 0,
// W 16-byte aligned, N <= 64.
// The W box a decode tensor map was encoded with (rows, and bytes of a box
// row); the launch is refused (cudaErrorInvalidValue) unless it is the box the
// chosen tile layout expects (decode_w_box / decode_moe_w_box, or 32 rows of
// 256 weights for the other block formats).
struct DecodeBox {
  uint32_t row_bytes = 0;
  uint32_t rows = 0;
};
cudaError_t launch_decode(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int64_t N, int64_t M, int64_t K,
                          float* Y, uint64_t wait_limit_ns, int early_w, int variant, int pdl, cudaStream_t s);
// Q4_1 / Q8_0, N <= 15: the decode kernel on 20- / 34-byte blocks; tmW boxes of
// 32 rows x 160 bytes (Q4_1, 8-bit elements) or 32 rows x 136 16-bit elements (Q8_0).
cudaError_t launch_decode_legacy(int type, const CUtensorMap* tmW, const DecodeBox& box, const float* X, int64_t N, int64_t M, int64_t K,
                                 float* Y, uint64_t wait_limit_ns, int early_w, int pdl, cudaStream_t s);
// TMA box the decode kernel expects for W (rows of raw blocks viewed as bytes).
void decode_w_box(int64_t N, int variant, uint32_t* box_x_bytes, uint32_t* box_rows);

// ---- generic fallback mul_mat: any K % 32 == 0, any alignment, any N.
cudaError_t launch_generic(const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                           cudaStream_t s);

void set_decode_early_stages(int n);  // W stages streamed before the dependency (with WEIGHTS_STATIC)
int get_decode_early_stages();
void set_decode_x_static(int on);      // GQ_OPT_X_STATIC: X is not written by kernels that may still run (read early)
int get_decode_x_static();

// ---- KQ: fp32 -> Q4_0 blocks (gq_quantize.cu).  K % 32 == 0, W 4-byte aligned.
cudaError_t launch_quantize(const float* W, int64_t M, int64_t K, uint8_t* out, cudaStream_t s);

// ---- K0: fp32 -> bf16 (round to nearest even) (gq_prefill.cu)
// pdl: launch with programmatic dependent launch (the kernel waits for the one before).
cudaError_t launch_f32_to_bf16(const float* x, uint16_t* y, int64_t n, cudaStream_t s, int pdl);

// ---- K3: prefill mul_mat on tcgen05 (gq_prefill.cu).  Needs K % 256 == 0.
// allow_scratch: the launch may take stream-ordered scratch for the partial
// sums of tiles split along k (else, or if that allocation fails, whole tiles).
// type: block format of W (GQ_TYPE_*; Q4_1 and Q8_0 run the 1-CTA kernels).
// pdl: launch with programmatic dependent launch (every role waits for the
// kernel before; with early_w the first raw W chunks stream before that; with
// x_static only Y and the k-split scratch wait for it).
cudaError_t launch_prefill(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t N, int64_t M,
                           int64_t K, float* Y, uint64_t wait_limit_ns, bool allow_scratch, int early_w,
                           int x_static, int pdl, cudaStream_t s, int type = GQ_TYPE_Q4_0);
void set_prefill_streamk(int64_t v);   // 0 whole tiles only, 1 by shape (default), n >= 2: every tile in n pieces
int64_t get_prefill_streamk();
void set_prefill_slots(int64_t v);     // 0: SM count; n: plan for n SMs (test aid)
int64_t get_prefill_slots();
void set_prefill_bn_override(int bn);  // 0 = by shape, else 128 or 256
void set_prefill_pair_mode(int on);    // 1: 2-SM pair kernel for N > 128 (default 0)
int get_prefill_pair_mode();
int get_prefill_bn_override();
// TMA boxes of the prefill kernel: W rows of one 256-k chunk as w_box_x
// elements of w_elem_bytes each (1, or 2 when the chunk is wider than 256 bytes).
// The tile width depends on the shape, on whether tiles may be split
// (allow_split) and on whether the launch overlaps its neighbours on the
// stream (overlap: pdl and x_static), so the same arguments must reach
// launch_prefill.
void prefill_boxes(int64_t N, int64_t M, int64_t K, bool allow_split, bool overlap, int type, uint32_t* w_box_x,
                   uint32_t* w_elem_bytes, uint32_t* w_box_rows, uint32_t* x_box_k, uint32_t* x_box_rows);

// ---- KR / KG: MUL_MAT_ID routing and activation gather (gq_moe.cu)
// Routing tables in device memory, written by the routing kernel.
struct MoeRoute {
  int32_t* meta;        // [0] tensor-core work items, [1] decode groups, [2] routed pairs, [3] bad ids
  int32_t* off;         // [E + 2]: expert e's pairs are perm[off[e] .. off[e+1]); bad ids from off[E]
  int32_t* item_start;  // [E + 1]: first tensor-core work item (expert, row tile, token tile) of expert e
  int32_t* groups;      // [3 * max groups]: decode group = (expert, first sorted position, tokens <= cap)
  int32_t* perm;        // [P]: sorted position -> pair index t * S + s (stable within an expert)
  // Direct decode groups (no routing tables; the decode kernel only): when
  // ids is set, group g is pair g alone, with expert ids[g] (np groups of one
  // token; an id outside [0, ne) gives a NaN row and DEVERR_BAD_ID).
  const int32_t* ids;
  int32_t np, ne;
};
size_t moe_route_ints(int64_t E, int64_t P, int cap);
MoeRoute moe_route_layout(int32_t* base, int64_t E, int64_t P, int cap);
bool moe_route_supported(int64_t E);
cudaError_t launch_moe_route(const int32_t* ids, int64_t P, int64_t E, int64_t n_mtiles, int bn, int cap,
                             const MoeRoute& rt, float* Y, int64_t M, int pdl, cudaStream_t s);
cudaError_t launch_moe_gather_bf16(const float* X, int64_t P, int64_t K, const MoeRoute& rt, uint16_t* Xg,
                                   int pdl, cudaStream_t s);
cudaError_t launch_generic_id(const uint8_t* W, int64_t E, int64_t M, int64_t K, const float* X,
                              const int32_t* ids, int64_t P, float* Y, cudaStream_t s);
// Tensor-core MUL_MAT_ID over the routed pairs (gq_prefill.cu): tmW covers the
// E * M weight rows, tmX the gathered bf16 rows with 64-row boxes.
constexpr int kMoeBN = 256;   // tokens per tensor-core work item
cudaError_t launch_prefill_moe(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t E, int64_t M, int64_t K,
                               int64_t P, const MoeRoute& rt, float* Y, uint64_t wait_limit_ns, int pdl,
                               cudaStream_t s);
// Decode MUL_MAT_ID over the decode groups (gq_decode.cu); returns the group
// capacity the launch will use through decode_moe_cap first.
int decode_moe_cap(int64_t P, int64_t E, int64_t T);
void decode_moe_w_box(int cap, uint32_t* box_x_bytes, uint32_t* box_rows);
cudaError_t launch_decode_moe(const CUtensorMap* tmW, const DecodeBox& box, const float* X, int cap, int64_t E, int64_t M, int64_t K,
                              int64_t P, const MoeRoute& rt, float* Y, uint64_t wait_limit_ns, int pdl,
                              cudaStream_t s);

// ---- KL: Q4_1 / Q8_0 dequantisation and MUL_MAT (gq_legacy.cu)
int type_block_bytes(int type);    // bytes per block: 18 / 20 / 34 / 144 (Q4_K), 0 for an unknown type
int type_block_weights(int type);  // weights per block: 32, or 256 for Q4_K
uint64_t type_row_bytes(int type, int64_t K);  // bytes of a row of K weights; 0 unless K % block weights == 0
cudaError_t launch_dequant_legacy(int type, const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s);

// ---- KV: row-data validation (gq_validate.cu).  result[0] = blocks with a
// non-finite scale field, result[1] = the smallest such flat block index (or
// all ones); both reset on the stream first (pdl: the scan overlaps the reset).
cudaError_t launch_validate(const uint8_t* W, int64_t nblocks, int type, unsigned long long* result, int pdl,
                            cudaStream_t s);
cudaError_t launch_mul_mat_legacy(int type, const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N,
                                  float* Y, uint64_t wait_limit_ns, cudaStream_t s);

// ---- KK: Q4_K dequantisation (bit-exact) and the any-alignment MUL_MAT (gq_kquant.cu)
cudaError_t launch_dequant_q4_k(const uint8_t* W, int64_t nsuper, float* out, cudaStream_t s);
cudaError_t launch_mul_mat_q4_k(const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                                cudaStream_t s);

// ---- KP: Q4_0 repack into rows of a multiple of 256 weights (gq_prepare.cu)
int64_t prepared_row_bytes(int64_t K);  // ceil(K / 256) * 144
cudaError_t launch_prepare_q4_0(const uint8_t* W, int64_t M, int64_t K, int64_t row_stride, uint8_t* out,
                                cudaStream_t s);

// ---- helpers of the C ABI (gq_api.cu) for entry points defined in other files
gq_status api_fail(gq_status st, const char* msg);  // records the per-thread error text
void api_clear_error();
// GQ_OPT_TEST_DROP_ARRIVE: 1 = the decode kernel, 2 = the tensor-core kernel
// leaves one W copy of CTA 0 unissued (its consumers' bounded wait runs out).
int test_drop();                              // clears it (every entry point starts with this)
gq_status api_check_device();
int api_pdl();  // GQ_OPT_PDL
gq_status api_check_mm_shape(int64_t M, int64_t K, int64_t N);
gq_status api_prefill_bf16(const void* W, int64_t M, int64_t K, const uint16_t* X_bf16, int64_t N, float* Y,
                           bool allow_scratch, cudaStream_t s);

}  // namespace gq
