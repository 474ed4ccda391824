// K0: fp32 -> bf16 conversion of the activations, and K3: the prefill
// MUL_MAT against Q4_0 weights on tcgen05 tensor cores.
//
// K3 computes Y[n][m] = sum_k w[m][k] * x[n][k] for a 128-row x BN-token tile
// per CTA ("GGUF loading, mmap and tensor placement", step six: the MUL_MAT
// probe with a 512-token batch; "Binding GGUF weights to the compute graph",
// section 2.3: the kernel reads the blocks and dequantises them itself).
// Roles (192 threads):
//   warp 0  TMA producer: raw W rows (128 x 144 bytes = 256 weights each) and
//           bf16 x tiles (BN x 64, 128-byte swizzle) into shared-memory rings.
//   warp 1  allocates BN TMEM columns; one thread issues tcgen05.mma
//           (M=128, N=BN, K=16, bf16 x bf16 -> fp32 in TMEM) and commits to
//           the rings' "empty" barriers.
//   warps 2-5  dequantise: thread i owns W row i of the tile, expands its two
//           blocks per 64-k step to w = d*(q-8) in fp32 (exact), rounds once to
//           bf16 and writes the 128-byte-swizzled K-major A tile; then read the
//           accumulator with tcgen05.ld (warp w reads TMEM lanes 32*(w%4)..)
//           and store fp32 Y, consecutive lanes writing consecutive m.
// Every wait is bounded; a timeout sets the device error word, the roles
// drain what they issued, TMEM is released and the CTA exits.
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

namespace {

template <int BN>
struct PrefillCfg {
  static constexpr int kBM = 128;
  static constexpr int kBK = 64;        // k per MMA stage: one 128-byte row of bf16
  static constexpr int kRawK = 256;     // k per raw W stage
  static constexpr int kRawRow = 144;   // bytes of 8 blocks
  static constexpr int RS = 2, AS = 4, BS = (BN == 256 ? 3 : 4);
  static constexpr int kRawBytes = kBM * kRawRow;  // 18432
  static constexpr int kABytes = kBM * 128;        // 16384
  static constexpr int kBBytes = BN * 128;
  static constexpr int kOffB = 0;
  static constexpr int kOffA = kOffB + BS * kBBytes;
  static constexpr int kOffRaw = kOffA + AS * kABytes;
  static constexpr int kOffBar = kOffRaw + RS * kRawBytes;
  static constexpr int kNBar = 2 * RS + 2 * AS + 2 * BS + 1;
  static constexpr int kOffTmem = kOffBar + kNBar * 8;
  static constexpr int kOffAbort = kOffTmem + 8;
  static constexpr int kSmem = kOffAbort + 8 + 1024;  // + slack to align the base to 1024
  static constexpr int kThreads = 192;
};

// Two 4-bit codes -> bf16x2 of d*(q-8): exact in fp32, one rounding to bf16.
__device__ __forceinline__ uint32_t deq_pair(uint32_t q0, uint32_t q1, float d) {
  const float f0 = __uint_as_float(0x4B000000u | q0) - 8388616.0f;  // 2^23 + q - (2^23 + 8) = q - 8
  const float f1 = __uint_as_float(0x4B000000u | q1) - 8388616.0f;
  __nv_bfloat162 h = __floats2bfloat162_rn(f0 * d, f1 * d);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 8 codes from two words of code bytes (low or high nibbles) -> 8 bf16.
__device__ __forceinline__ uint4 deq_chunk(uint32_t qa, uint32_t qb, int sh, float d) {
  uint4 o;
  o.x = deq_pair((qa >> sh) & 0xF, (qa >> (sh + 8)) & 0xF, d);
  o.y = deq_pair((qa >> (sh + 16)) & 0xF, (qa >> (sh + 24)) & 0xF, d);
  o.z = deq_pair((qb >> sh) & 0xF, (qb >> (sh + 8)) & 0xF, d);
  o.w = deq_pair((qb >> (sh + 16)) & 0xF, (qb >> (sh + 24)) & 0xF, d);
  return o;
}

// Bounded wait on the last phase issued into each slot of a ring (drain path).
__device__ __forceinline__ void drain_ring(uint64_t* full, int slots, uint32_t issued, uint64_t limit_ns) {
  for (int s = 0; s < slots; ++s) {
    if (static_cast<uint32_t>(s) >= issued) break;
    const uint32_t last = ((issued - 1 - s) / slots) * slots + s;  // largest index < issued in slot s
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&full[s]), (last / slots) & 1) && globaltimer_ns() - t0 < limit_ns) {
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    k_prefill_q4_0(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int N, int M,
                   int K, float* __restrict__ Y, uint64_t limit_ns, uint32_t* err) {
  using C = PrefillCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + C::RS;
  uint64_t* a_full = raw_empty + C::RS;
  uint64_t* a_empty = a_full + C::AS;
  uint64_t* b_full = a_empty + C::AS;
  uint64_t* b_empty = b_full + C::BS;
  uint64_t* acc_full = b_empty + C::BS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntn = (N + BN - 1) / BN;
  const int m0 = (blockIdx.x / ntn) * C::kBM;
  const int n0 = (blockIdx.x % ntn) * BN;
  const int nk = K / C::kBK;
  const int nr = K / C::kRawK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RS; ++i) {
      mbar_init(smem_u32(&raw_full[i]), 1);
      mbar_init(smem_u32(&raw_empty[i]), 4);
    }
    for (int i = 0; i < C::AS; ++i) {
      mbar_init(smem_u32(&a_full[i]), 4);
      mbar_init(smem_u32(&a_empty[i]), 1);
    }
    for (int i = 0; i < C::BS; ++i) {
      mbar_init(smem_u32(&b_full[i]), 1);
      mbar_init(smem_u32(&b_empty[i]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      uint32_t nraw = 0, nb = 0;
      bool ok = true;
      for (int ks = 0; ks < nk && ok; ++ks) {
        if ((ks & 3) == 0) {
          const int r = ks >> 2, slot = r % C::RS;
          if (!mbar_wait_bounded(smem_u32(&raw_empty[slot]), ((r / C::RS) & 1) ^ 1, limit_ns, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&raw_full[slot]), C::kRawBytes);
          tma_load_2d(sbase + C::kOffRaw + slot * C::kRawBytes, &tmW, r * C::kRawRow, m0, smem_u32(&raw_full[slot]));
          ++nraw;
        }
        const int slot = ks % C::BS;
        if (!mbar_wait_bounded(smem_u32(&b_empty[slot]), ((ks / C::BS) & 1) ^ 1, limit_ns, abort_flag, err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&b_full[slot]), C::kBBytes);
        tma_load_2d(sbase + C::kOffB + slot * C::kBBytes, &tmX, ks * C::kBK, n0, smem_u32(&b_full[slot]));
        ++nb;
      }
      if (!ok) {
        drain_ring(raw_full, C::RS, nraw, limit_ns);
        drain_ring(b_full, C::BS, nb, limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16_f32(128, BN);
      for (int ks = 0; ks < nk; ++ks) {
        const int as = ks % C::AS, bs = ks % C::BS;
        if (!mbar_wait_bounded(smem_u32(&a_full[as]), (ks / C::AS) & 1, limit_ns, abort_flag, err)) break;
        if (!mbar_wait_bounded(smem_u32(&b_full[bs]), (ks / C::BS) & 1, limit_ns, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t a_addr = sbase + C::kOffA + as * C::kABytes;
        const uint32_t b_addr = sbase + C::kOffB + bs * C::kBBytes;
#pragma unroll
        for (int kk = 0; kk < C::kBK / 16; ++kk)
          umma_bf16_ss(tmem_base, umma_desc_sw128(a_addr + kk * 32), umma_desc_sw128(b_addr + kk * 32), idesc,
                       (ks | kk) != 0);
        umma_commit(smem_u32(&a_empty[as]));
        umma_commit(smem_u32(&b_empty[bs]));
      }
      umma_commit(smem_u32(acc_full));
      // Do not leave while MMAs issued by this thread may still run.
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(acc_full), 0) && globaltimer_ns() - t0 < limit_ns) {
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // W row within the tile == TMEM lane
    bool live = true;
    for (int r = 0; r < nr; ++r) {
      const int rslot = r % C::RS;
      if (live) live = mbar_wait_bounded(smem_u32(&raw_full[rslot]), (r / C::RS) & 1, limit_ns, abort_flag, err);
      live = __all_sync(0xFFFFFFFFu, live);
      uint32_t w[36];
      if (live) {
        const uint4* src = reinterpret_cast<const uint4*>(smem + C::kOffRaw + rslot * C::kRawBytes + row * C::kRawRow);
#pragma unroll
        for (int i = 0; i < 9; ++i) {
          const uint4 v = src[i];
          w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
      }
      __syncwarp();
      if (live && lane == 0) mbar_arrive(smem_u32(&raw_empty[rslot]));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ks = r * 4 + j, as = ks % C::AS;
        if (live) live = mbar_wait_bounded(smem_u32(&a_empty[as]), ((ks / C::AS) & 1) ^ 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        if (live) {
          // blocks 2j (even) and 2j+1 (odd) of the raw row = words 9j .. 9j+8
          const uint32_t W0 = w[9 * j], W1 = w[9 * j + 1], W2 = w[9 * j + 2], W3 = w[9 * j + 3], W4 = w[9 * j + 4];
          const float d0 = __half2float(__ushort_as_half(static_cast<uint16_t>(W0 & 0xFFFFu)));
          const float d1 = __half2float(__ushort_as_half(static_cast<uint16_t>(W4 >> 16)));
          const uint32_t q0[4] = {prmt(W0, W1, 0x5432u), prmt(W1, W2, 0x5432u), prmt(W2, W3, 0x5432u),
                                  prmt(W3, W4, 0x5432u)};
          const uint32_t q1[4] = {w[9 * j + 5], w[9 * j + 6], w[9 * j + 7], w[9 * j + 8]};
          uint8_t* arow = smem + C::kOffA + as * C::kABytes + row * 128;
          const int sw = row & 7;
          // chunk c holds k = 8c .. 8c+7 of this 64-k step
          *reinterpret_cast<uint4*>(arow + ((0 ^ sw) << 4)) = deq_chunk(q0[0], q0[1], 0, d0);
          *reinterpret_cast<uint4*>(arow + ((1 ^ sw) << 4)) = deq_chunk(q0[2], q0[3], 0, d0);
          *reinterpret_cast<uint4*>(arow + ((2 ^ sw) << 4)) = deq_chunk(q0[0], q0[1], 4, d0);
          *reinterpret_cast<uint4*>(arow + ((3 ^ sw) << 4)) = deq_chunk(q0[2], q0[3], 4, d0);
          *reinterpret_cast<uint4*>(arow + ((4 ^ sw) << 4)) = deq_chunk(q1[0], q1[1], 0, d1);
          *reinterpret_cast<uint4*>(arow + ((5 ^ sw) << 4)) = deq_chunk(q1[2], q1[3], 0, d1);
          *reinterpret_cast<uint4*>(arow + ((6 ^ sw) << 4)) = deq_chunk(q1[0], q1[1], 4, d1);
          *reinterpret_cast<uint4*>(arow + ((7 ^ sw) << 4)) = deq_chunk(q1[2], q1[3], 4, d1);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (live && lane == 0) mbar_arrive(smem_u32(&a_full[as]));
      }
    }
    // epilogue
    if (live) live = mbar_wait_bounded(smem_u32(acc_full), 0, limit_ns, abort_flag, err);
    live = __all_sync(0xFFFFFFFFu, live);
    tc_fence_after();
    if (live) {
      const int m = m0 + row;
#pragma unroll 1
      for (int cb = 0; cb < BN / 32; ++cb) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + cb * 32, v);
        tmem_ld_wait();
        if (m < M) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int n = n0 + cb * 32 + jj;
            if (n < N) Y[static_cast<size_t>(n) * M + m] = __uint_as_float(v[jj]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, BN);
  }
}

template <int BN>
cudaError_t launch_prefill_bn(const CUtensorMap* tmW, const CUtensorMap* tmX, int N, int M, int K, float* Y,
                              uint64_t limit_ns, cudaStream_t s) {
  using C = PrefillCfg<BN>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill_q4_0<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int grid = ((M + C::kBM - 1) / C::kBM) * ((N + BN - 1) / BN);
  k_prefill_q4_0<BN><<<grid, C::kThreads, C::kSmem, s>>>(*tmW, *tmX, N, M, K, Y, limit_ns, device_error_word());
  return cudaGetLastError();
}

int prefill_bn(int64_t N) { return N <= 128 ? 128 : 256; }

}  // namespace

void prefill_boxes(int64_t N, uint32_t* w_box_x_bytes, uint32_t* w_box_rows, uint32_t* x_box_k,
                   uint32_t* x_box_rows) {
  *w_box_x_bytes = 144;
  *w_box_rows = 128;
  *x_box_k = 64;
  *x_box_rows = static_cast<uint32_t>(prefill_bn(N));
}

cudaError_t launch_prefill(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t N, int64_t M, int64_t K,
                           float* Y, uint64_t wait_limit_ns, cudaStream_t s) {
  const int n = static_cast<int>(N), m = static_cast<int>(M), k = static_cast<int>(K);
  if (prefill_bn(N) == 128) return launch_prefill_bn<128>(tmW, tmX, n, m, k, Y, wait_limit_ns, s);
  return launch_prefill_bn<256>(tmW, tmX, n, m, k, Y, wait_limit_ns, s);
}

}  // namespace gq
