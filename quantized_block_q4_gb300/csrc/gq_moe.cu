// KR / KG: routing and activation gather of MUL_MAT_ID, and its generic
// fallback kernel.
//
// MUL_MAT_ID ("GGUF loading, mmap and tensor placement", step six, the
// MUL_MAT_ID probe: w ne = [K, M, n_expert], b ne = [K, n_ids, tokens], ids ne
// = [n_ids, tokens]) computes, for every (token t, slot s) pair,
//   Y[t][s][m] = sum_k w_e[m][k] * X[t][s][k],  e = ids[t][s].
// Instead of one MUL_MAT per pair, the pairs are sorted by expert so that each
// expert's weights are read once for all the tokens routed to it:
//   KR  one CTA: a stable counting sort of the P = T*S pairs by expert id (per-
//       warp histograms, an exclusive scan over (expert, warp), then a second
//       pass that places each pair, ranks within a warp from __match_any_sync).
//       It also lays out the work of the matmul kernels: tensor-core work items
//       (expert, 128-row tile, 256-token tile) and decode groups (expert, up to
//       `cap` tokens).  Ids outside [0, n_expert) are sorted after all experts,
//       their Y rows are set to NaN and the device error word gets DEVERR_BAD_ID.
//   KG  many CTAs: Xg[pos] = bf16(X[perm[pos]]) for the routed pairs in sorted
//       order, so that each expert's tokens are consecutive bf16 rows that the
//       tensor-core kernel loads with TMA.
// Results do not depend on the order of pairs within an expert (each output
// row is its own dot product), but the sort is stable anyway, so launches are
// reproducible bit for bit.
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {
namespace {

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__global__ void k_moe_route(const int32_t* __restrict__ ids, int P, int E, int n_mtiles, int bn, int cap,
                            MoeRoute rt, float* __restrict__ Y, int M, uint32_t* err) {
  extern __shared__ int sh[];
  __shared__ int wtot[32][3];
  __shared__ int tot[3];
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int EB = E + 1;           // bucket E collects the ids outside [0, E)
  int* hist = sh;                 // [nw][EB]: pass-1 counts, then each warp's next sorted position
  int* cnt = sh + nw * EB;        // [EB]: pairs per bucket
  pdl_wait();  // ids may come from the previous kernel
  pdl_launch_dependents();  // after the wait: a later launch cannot overtake the kernels ahead of this one

  for (int i = threadIdx.x; i < nw * EB; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  // Warp w takes the contiguous range [r0, r1) of pairs, in order.
  const int r0 = static_cast<int>(static_cast<int64_t>(P) * warp / nw);
  const int r1 = static_cast<int>(static_cast<int64_t>(P) * (warp + 1) / nw);
  auto bucket = [&](int i) -> int {
    if (i >= r1) return -1;
    const int v = __ldg(ids + i);
    return (v >= 0 && v < E) ? v : E;
  };
  for (int base = r0; base < r1; base += 32) {
    const int e = bucket(base + lane);
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) hist[warp * EB + e] += __popc(peers);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < EB; b += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int v = hist[w * EB + b];
      hist[w * EB + b] = run;
      run += v;
    }
    cnt[b] = run;
  }
  __syncthreads();

  // Exclusive scans over the buckets of (pairs, tensor-core items, decode
  // groups); thread t covers a contiguous run of buckets.
  auto items_of = [&](int b) { return b < E ? n_mtiles * ceil_div(cnt[b], bn) : 0; };
  auto groups_of = [&](int b) { return b < E ? ceil_div(cnt[b], cap) : 0; };
  const int chunk = (EB + blockDim.x - 1) / blockDim.x;
  const int b0 = min(EB, static_cast<int>(threadIdx.x) * chunk), b1 = min(EB, b0 + chunk);
  int s0 = 0, s1 = 0, s2 = 0;
  for (int b = b0; b < b1; ++b) {
    s0 += cnt[b];
    s1 += items_of(b);
    s2 += groups_of(b);
  }
  int i0 = s0, i1 = s1, i2 = s2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a0 = __shfl_up_sync(0xFFFFFFFFu, i0, o);
    const int a1 = __shfl_up_sync(0xFFFFFFFFu, i1, o);
    const int a2 = __shfl_up_sync(0xFFFFFFFFu, i2, o);
    if (lane >= o) {
      i0 += a0;
      i1 += a1;
      i2 += a2;
    }
  }
  if (lane == 31) {
    wtot[warp][0] = i0;
    wtot[warp][1] = i1;
    wtot[warp][2] = i2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0, c = 0, d = 0;
    for (int w = 0; w < nw; ++w) {
      const int x0 = wtot[w][0], x1 = wtot[w][1], x2 = wtot[w][2];
      wtot[w][0] = a;
      wtot[w][1] = c;
      wtot[w][2] = d;
      a += x0;
      c += x1;
      d += x2;
    }
    tot[0] = a;
    tot[1] = c;
    tot[2] = d;
  }
  __syncthreads();
  int e0 = wtot[warp][0] + i0 - s0, e1 = wtot[warp][1] + i1 - s1, e2 = wtot[warp][2] + i2 - s2;
  for (int b = b0; b < b1; ++b) {
    const int c = cnt[b];
    rt.off[b] = e0;
    if (b < E) {
      rt.item_start[b] = e1;
      for (int k = 0; k * cap < c; ++k) {
        int* g = rt.groups + 3 * (e2 + k);
        g[0] = b;
        g[1] = e0 + k * cap;
        g[2] = min(cap, c - k * cap);
      }
    }
    for (int w = 0; w < nw; ++w) hist[w * EB + b] += e0;
    e0 += c;
    e1 += items_of(b);
    e2 += groups_of(b);
  }
  if (threadIdx.x == 0) {
    rt.off[EB] = P;
    rt.item_start[E] = tot[1];
    rt.meta[0] = tot[1];
    rt.meta[1] = tot[2];
    rt.meta[2] = P - cnt[E];
    rt.meta[3] = cnt[E];
  }
  __syncthreads();

  // Pass 2: place each pair; within a warp's step, equal ids keep lane order.
  for (int base = r0; base < r1; base += 32) {
    const int i = base + lane;
    const int e = bucket(i);
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    int pos = 0;
    if (e >= 0) pos = hist[warp * EB + e] + __popc(peers & ((1u << lane) - 1u));
    __syncwarp();
    if (e >= 0) {
      rt.perm[pos] = i;
      if (lane == __ffs(peers) - 1) hist[warp * EB + e] += __popc(peers);
    }
    __syncwarp();
  }

  const int nbad = cnt[E];
  if (nbad > 0) {
    __syncthreads();  // every perm entry written
    if (threadIdx.x == 0) atomicOr(err, DEVERR_BAD_ID);
    const int first = P - nbad;
    for (int64_t j = threadIdx.x; j < static_cast<int64_t>(nbad) * M; j += blockDim.x) {
      const int pr = rt.perm[first + static_cast<int>(j / M)];
      Y[static_cast<size_t>(pr) * M + static_cast<size_t>(j % M)] = __int_as_float(0x7FC00000);
    }
  }
}

// Xg[pos][:] = bf16(X[perm[pos]][:]) for pos < routed pairs.  K % 8 == 0 and
// X, Xg 16-byte aligned: 8 elements per thread step.
__global__ void k_moe_gather_bf16(const float* __restrict__ X, int64_t K, const MoeRoute rt,
                                  uint16_t* __restrict__ Xg) {
  pdl_wait();
  pdl_launch_dependents();
  const int routed = rt.meta[2];
  const int64_t k8 = K / 8;
  for (int pos = blockIdx.x; pos < routed; pos += gridDim.x) {
    const float4* src = reinterpret_cast<const float4*>(X + static_cast<size_t>(rt.perm[pos]) * K);
    uint4* dst = reinterpret_cast<uint4*>(Xg + static_cast<size_t>(pos) * K);
    for (int64_t j = threadIdx.x; j < k8; j += blockDim.x) {
      const float4 a = __ldg(src + 2 * j), b = __ldg(src + 2 * j + 1);
      __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
      uint4 o;
      o.x = *reinterpret_cast<uint32_t*>(&p0);
      o.y = *reinterpret_cast<uint32_t*>(&p1);
      o.z = *reinterpret_cast<uint32_t*>(&p2);
      o.w = *reinterpret_cast<uint32_t*>(&p3);
      dst[j] = o;
    }
  }
}

// Fallback for any K % 32 == 0 and any alignment: one warp per (pair, row),
// ids read directly (no routing).  An id outside [0, E) gives a NaN row and
// DEVERR_BAD_ID.
__global__ void k_generic_id_q4_0(const uint8_t* __restrict__ W, int E, int64_t M, int64_t K,
                                  const float* __restrict__ X, const int32_t* __restrict__ ids, int64_t P,
                                  float* __restrict__ Y, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / kQK;
  const int64_t row_bytes = nb * kBlockBytes;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); idx < P * M;
       idx += warps) {
    const int64_t p = idx / M, m = idx % M;
    const int e = ids[p];
    if (e < 0 || e >= E) {
      if (lane == 0) {
        Y[p * M + m] = __int_as_float(0x7FC00000);
        atomicOr(err, DEVERR_BAD_ID);
      }
      continue;
    }
    const uint8_t* row = W + (static_cast<int64_t>(e) * M + m) * row_bytes;
    const float* x = X + p * K;
    float acc = 0.f;
    for (int64_t b = lane; b < nb; b += 32) {
      const uint8_t* blk = row + b * kBlockBytes;
      const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(blk[0] | (blk[1] << 8))));
      float part = 0.f;
      for (int j = 0; j < 16; ++j) {
        const uint32_t byte = blk[2 + j];
        part = fmaf(static_cast<float>(static_cast<int>(byte & 0xF) - 8), x[b * kQK + j], part);
        part = fmaf(static_cast<float>(static_cast<int>(byte >> 4) - 8), x[b * kQK + j + 16], part);
      }
      acc = fmaf(d, part, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) Y[p * M + m] = acc;
  }
}

// Warps of the routing CTA: per-warp histograms of E + 1 ints must fit in
// shared memory next to one count per bucket.
int route_warps(int E) {
  const int budget_ints = (200 * 1024) / 4;
  const int nw = budget_ints / (E + 1) - 1;
  return std::min(32, nw);
}

}  // namespace

size_t moe_route_ints(int64_t E, int64_t P, int cap) {
  const int64_t max_groups = std::min(E, P) + P / std::max(cap, 1) + 1;
  return 4 + static_cast<size_t>(E + 2) + static_cast<size_t>(E + 1) + 3 * static_cast<size_t>(max_groups) +
         static_cast<size_t>(P);
}

MoeRoute moe_route_layout(int32_t* base, int64_t E, int64_t P, int cap) {
  const int64_t max_groups = std::min(E, P) + P / std::max(cap, 1) + 1;
  MoeRoute rt{};  // ids = nullptr: routed groups
  rt.meta = base;
  rt.off = rt.meta + 4;
  rt.item_start = rt.off + (E + 2);
  rt.groups = rt.item_start + (E + 1);
  rt.perm = rt.groups + 3 * max_groups;
  return rt;
}

bool moe_route_supported(int64_t E) { return E >= 1 && route_warps(static_cast<int>(E)) >= 1; }

cudaError_t launch_moe_route(const int32_t* ids, int64_t P, int64_t E, int64_t n_mtiles, int bn, int cap,
                             const MoeRoute& rt, float* Y, int64_t M, int pdl, cudaStream_t s) {
  // One warp per 64 pairs up to the shared-memory limit: a decode batch of a
  // few pairs needs one warp and no cross-warp work.
  const int nw = std::max(1, std::min(route_warps(static_cast<int>(E)), static_cast<int>((P + 63) / 64)));
  const size_t smem = (static_cast<size_t>(nw) + 1) * static_cast<size_t>(E + 1) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = kernel_smem(reinterpret_cast<const void*>(k_moe_route), smem, false);
    if (e != cudaSuccess) return e;
  }
  // With programmatic dependent launch the routing CTA starts while the
  // previous kernel drains; it reads ids only after griddepcontrol.wait.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32 * nw);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_moe_route, ids, static_cast<int>(P), static_cast<int>(E),
                            static_cast<int>(n_mtiles), bn, cap, rt, Y, static_cast<int>(M), device_error_word());
}

cudaError_t launch_moe_gather_bf16(const float* X, int64_t P, int64_t K, const MoeRoute& rt, uint16_t* Xg,
                                   int pdl, cudaStream_t s) {
  const int grid = static_cast<int>(std::min<int64_t>(P, static_cast<int64_t>(device_info().sm_count) * 8));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_moe_gather_bf16, X, K, rt, Xg);
}

cudaError_t launch_generic_id(const uint8_t* W, int64_t E, int64_t M, int64_t K, const float* X,
                              const int32_t* ids, int64_t P, float* Y, cudaStream_t s) {
  const int64_t warps = P * M;
  const int grid = static_cast<int>(std::min<int64_t>((warps + 7) / 8, static_cast<int64_t>(device_info().sm_count) * 16));
  k_generic_id_q4_0<<<grid > 0 ? grid : 1, 256, 0, s>>>(W, static_cast<int>(E), M, K, X, ids, P, Y,
                                                          device_error_word());
  return cudaGetLastError();
}

}  // namespace gq
