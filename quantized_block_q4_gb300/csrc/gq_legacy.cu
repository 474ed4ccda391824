// KL: the other legacy block formats, Q4_1 and Q8_0: dequantisation (bit-
// exact) and MUL_MAT.
//
// "Architecture and module overview", quantisation-format section: the legacy
// formats keep one scale per block of 32 weights, Q4_1 additionally a min
// offset, Q8_0 eight bits per weight.  Layout read from that section and the
// Q4_0 struct of "Binding GGUF weights to the compute graph", section 2.3:
//   Q4_1: ggml_half d, ggml_half m, uint8_t qs[16]  (20 bytes), w = d*q + m,
//         q = 0..15, low nibble of qs[j] = element j, high nibble = j+16;
//   Q8_0: ggml_half d, int8_t qs[32]                (34 bytes), w = d*q.
// In fp32 d*q is exact (at most 11 x 8 significant bits); Q4_1 adds m with
// one rounding.  Both kernels evaluate exactly that, so dequantisation is
// bit-exact and MUL_MAT sees the same weights.
//
// MUL_MAT here is the decode-shaped kernel for these formats: one warp per
// weight row, lanes taking consecutive blocks (a warp's loads of one step
// cover 32 consecutive blocks), weights decoded to fp32 in registers and
// dotted with x in fp32 for up to kTok tokens per pass; the lanes' partial
// sums meet by shuffles.  W is read from DRAM once per pass; more tokens than
// kTok re-read it from L2.
#include <algorithm>
#include <cuda_fp16.h>

#include "gq_internal.h"

namespace gq {
namespace {

template <int T>
struct Fmt;
template <>
struct Fmt<GQ_TYPE_Q4_1> {
  static constexpr int kBytes = 20;
};
template <>
struct Fmt<GQ_TYPE_Q8_0> {
  static constexpr int kBytes = 34;
};

__device__ __forceinline__ float half_at(const uint8_t* p) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(p[0] | (p[1] << 8))));
}

// Element e (0..31) of a block held in shared or global memory.
template <int T>
__device__ __forceinline__ float weight(const uint8_t* blk, int e, float d, float m) {
  if constexpr (T == GQ_TYPE_Q4_1) {
    const uint32_t byte = blk[4 + (e & 15)];
    const uint32_t q = e < 16 ? (byte & 0xF) : (byte >> 4);
    return __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
  } else {
    (void)m;
    return __fmul_rn(d, static_cast<float>(static_cast<int8_t>(blk[2 + e])));
  }
}

constexpr int kDqThreads = 256;
constexpr int kDqTile = 256;  // blocks per tile: a multiple of 8, so 16-byte aligned tiles stay aligned

// Tiles of 256 blocks are staged in shared memory (16-byte loads when W is
// 16-byte aligned, else byte loads); each thread then writes float4 outputs,
// consecutive threads consecutive 16 bytes.
template <int T>
__global__ void __launch_bounds__(kDqThreads) k_dequant_legacy(const uint8_t* __restrict__ W, int64_t nblocks,
                                                               float* __restrict__ out, int vec_in, int vec_out) {
  constexpr int kB = Fmt<T>::kBytes;
  __shared__ __align__(16) uint8_t tile[kDqTile * kB];
  const int64_t ntiles = (nblocks + kDqTile - 1) / kDqTile;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t b0 = t * kDqTile;
    const int nb = static_cast<int>(nblocks - b0 < kDqTile ? nblocks - b0 : kDqTile);
    const int nbytes = nb * kB;
    const uint8_t* src = W + b0 * kB;
    __syncthreads();
    if (vec_in) {
      for (int c = threadIdx.x; c * 16 < nbytes; c += kDqThreads) {
        if (c * 16 + 16 <= nbytes)
          *reinterpret_cast<uint4*>(tile + c * 16) = __ldg(reinterpret_cast<const uint4*>(src + c * 16));
        else
          for (int i = c * 16; i < nbytes; ++i) tile[i] = src[i];
      }
    } else {
      for (int i = threadIdx.x; i < nbytes; i += kDqThreads) tile[i] = src[i];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < nb * 8; o += kDqThreads) {
      const int b = o >> 3, part = o & 7;
      const uint8_t* blk = tile + b * kB;
      const float d = half_at(blk);
      const float m = T == GQ_TYPE_Q4_1 ? half_at(blk + 2) : 0.f;
      float4 v;
      v.x = weight<T>(blk, 4 * part, d, m);
      v.y = weight<T>(blk, 4 * part + 1, d, m);
      v.z = weight<T>(blk, 4 * part + 2, d, m);
      v.w = weight<T>(blk, 4 * part + 3, d, m);
      float* dst = out + (b0 + b) * kQK + 4 * part;
      if (vec_out) {
        *reinterpret_cast<float4*>(dst) = v;
      } else {
        dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
      }
    }
  }
}

constexpr int kTok = 4;  // tokens per pass of the MUL_MAT kernel

// One block's 32 weights, from global memory, into registers.
template <int T>
__device__ __forceinline__ void load_block(const uint8_t* __restrict__ blk, float (&w)[32]) {
  if constexpr (T == GQ_TYPE_Q4_1) {
    // 20-byte blocks of a 4-byte aligned row: five 32-bit loads
    const uint32_t* p = reinterpret_cast<const uint32_t*>(blk);
    const uint32_t h = __ldg(p);
    const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(h & 0xFFFF)));
    const float m = __half2float(__ushort_as_half(static_cast<uint16_t>(h >> 16)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = __ldg(p + 1 + i);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t byte = (v >> (8 * j)) & 0xFF;
        w[4 * i + j] = __fadd_rn(__fmul_rn(d, static_cast<float>(byte & 0xF)), m);
        w[16 + 4 * i + j] = __fadd_rn(__fmul_rn(d, static_cast<float>(byte >> 4)), m);
      }
    }
  } else {
    // 34-byte blocks are 2-byte aligned: seventeen 16-bit loads
    const uint16_t* p = reinterpret_cast<const uint16_t*>(blk);
    const float d = __half2float(__ushort_as_half(__ldg(p)));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t v = __ldg(p + 1 + i);
      w[2 * i] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(v & 0xFF)));
      w[2 * i + 1] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(v >> 8)));
    }
  }
}

template <int T>
__global__ void __launch_bounds__(256) k_mul_mat_legacy(const uint8_t* __restrict__ W, int M, int K,
                                                        const float* __restrict__ X, int N, float* __restrict__ Y) {
  constexpr int kB = Fmt<T>::kBytes;
  const int lane = threadIdx.x & 31;
  const int nb = K / kQK;
  const int64_t row_bytes = static_cast<int64_t>(nb) * kB;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint8_t* row = W + m * row_bytes;
    for (int n0 = 0; n0 < N; n0 += kTok) {
      const int nt = N - n0 < kTok ? N - n0 : kTok;
      float acc[kTok] = {};
      for (int b = lane; b < nb; b += 32) {
        float w[32];
        load_block<T>(row + static_cast<int64_t>(b) * kB, w);
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t < nt) {
            const float4* xp = reinterpret_cast<const float4*>(X + static_cast<int64_t>(n0 + t) * K + b * kQK);
            float a = acc[t];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = __ldg(xp + i);
              a = fmaf(w[4 * i], x.x, a);
              a = fmaf(w[4 * i + 1], x.y, a);
              a = fmaf(w[4 * i + 2], x.z, a);
              a = fmaf(w[4 * i + 3], x.w, a);
            }
            acc[t] = a;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        if (lane == 0 && t < nt) Y[static_cast<int64_t>(n0 + t) * M + m] = a;
      }
    }
  }
}

// Any alignment: one warp per row, byte loads of W and scalar loads of x.
template <int T>
__global__ void k_mul_mat_legacy_bytes(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                       const float* __restrict__ X, int64_t N, float* __restrict__ Y) {
  constexpr int kB = Fmt<T>::kBytes;
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / kQK;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t m = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint8_t* row = W + m * nb * kB;
    for (int64_t n = 0; n < N; ++n) {
      const float* x = X + n * K;
      float acc = 0.f;
      for (int64_t b = lane; b < nb; b += 32) {
        const uint8_t* blk = row + b * kB;
        const float d = half_at(blk);
        const float mn = T == GQ_TYPE_Q4_1 ? half_at(blk + 2) : 0.f;
        for (int e = 0; e < kQK; ++e) acc = fmaf(weight<T>(blk, e, d, mn), x[b * kQK + e], acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (lane == 0) Y[n * M + m] = acc;
    }
  }
}

template <int T>
cudaError_t launch_dequant_t(const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s) {
  const int64_t ntiles = (nblocks + kDqTile - 1) / kDqTile;
  const int grid = static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(device_info().sm_count) * 8));
  const int vec_in = (reinterpret_cast<uintptr_t>(W) & 15) == 0;
  const int vec_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  k_dequant_legacy<T><<<grid > 0 ? grid : 1, kDqThreads, 0, s>>>(W, nblocks, out, vec_in, vec_out);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_mul_mat_t(const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N, float* Y,
                             cudaStream_t s) {
  const int64_t rows_per_cta = 8;  // 8 warps
  const int grid = static_cast<int>(
      std::min<int64_t>((M + rows_per_cta - 1) / rows_per_cta, static_cast<int64_t>(device_info().sm_count) * 16));
  // The fast kernel needs 4-byte aligned rows for Q4_1 (2-byte for Q8_0), 16-byte aligned x rows and
  // int sizes; anything else takes the byte kernel.
  const int64_t row_bytes = (K / kQK) * Fmt<T>::kBytes;
  const uintptr_t wa = reinterpret_cast<uintptr_t>(W), xa = reinterpret_cast<uintptr_t>(X);
  const bool fast = ((wa | static_cast<uintptr_t>(row_bytes)) & (T == GQ_TYPE_Q4_1 ? 3 : 1)) == 0 && (xa & 15) == 0 &&
                    K % 4 == 0 && M < (int64_t(1) << 31) && K < (int64_t(1) << 31) && N < (int64_t(1) << 31);
  if (fast)
    k_mul_mat_legacy<T><<<grid > 0 ? grid : 1, 256, 0, s>>>(W, static_cast<int>(M), static_cast<int>(K), X,
                                                             static_cast<int>(N), Y);
  else
    k_mul_mat_legacy_bytes<T><<<grid > 0 ? grid : 1, 256, 0, s>>>(W, M, K, X, N, Y);
  return cudaGetLastError();
}

}  // namespace

int type_block_bytes(int type) {
  switch (type) {
    case GQ_TYPE_Q4_0: return kBlockBytes;
    case GQ_TYPE_Q4_1: return Fmt<GQ_TYPE_Q4_1>::kBytes;
    case GQ_TYPE_Q8_0: return Fmt<GQ_TYPE_Q8_0>::kBytes;
  }
  return 0;
}

cudaError_t launch_dequant_legacy(int type, const uint8_t* W, int64_t nblocks, float* out, cudaStream_t s) {
  if (type == GQ_TYPE_Q4_1) return launch_dequant_t<GQ_TYPE_Q4_1>(W, nblocks, out, s);
  return launch_dequant_t<GQ_TYPE_Q8_0>(W, nblocks, out, s);
}

cudaError_t launch_mul_mat_legacy(int type, const uint8_t* W, int64_t M, int64_t K, const float* X, int64_t N,
                                  float* Y, cudaStream_t s) {
  if (type == GQ_TYPE_Q4_1) return launch_mul_mat_t<GQ_TYPE_Q4_1>(W, M, K, X, N, Y, s);
  return launch_mul_mat_t<GQ_TYPE_Q8_0>(W, M, K, X, N, Y, s);
}

}  // namespace gq
