// K0: fp32 -> bf16 conversion of the activations, and K3: the prefill
// MUL_MAT against Q4_0 weights on tcgen05 tensor cores.
//
// K3 computes Y[n][m] = sum_k w[m][k] * x[n][k] for a 128-row x BN-token tile
// per CTA ("GGUF loading, mmap and tensor placement", step six: the MUL_MAT
// probe with a 512-token batch; "Binding GGUF weights to the compute graph",
// section 2.3: the kernel reads the blocks and dequantises them itself).
// Roles (320 threads):
//   warp 0  TMA producer: raw W rows (128 x 144 bytes = 256 weights each) and
//           bf16 x tiles (BN x 64, 128-byte swizzle) into shared-memory rings.
//   warp 1  allocates 512 TMEM columns: the fp32 accumulator (BN columns) and
//           a ring of A stages (32 columns = 64 bf16 k each).  One thread
//           issues tcgen05.mma with A read from tensor memory and B (x) from
//           shared memory (M=128, N=BN, K=16, bf16 x bf16 -> fp32) and
//           commits to the rings' "empty" barriers.
//   warps 2-9  dequantise: warps 2-5 take the even 64-k steps, warps 6-9 the
//           odd ones; a thread owns one W row of the tile, i.e. one TMEM lane,
//           and stores RN_bf16(d*(q-8)) for the step's 64 weights into its
//           lane with one tcgen05.st.  Then they read the accumulator with
//           tcgen05.ld (warp w reads TMEM lanes 32*(w%4)..; the two groups
//           split the columns) and store fp32 Y, consecutive lanes writing
//           consecutive m.
// Dequantisation to bf16 with a single rounding, in bf16x2 arithmetic: the
// fp16 scale is split exactly as d = d_hi + d_lo (both bf16; d_lo holds the
// last 3 bits), q - 8 is formed exactly as (128 + q) - 136 from the bit
// pattern 0x4300 | q, q'*d_lo is exact in bf16, and one fused
// fma.rn.bf16x2(q', d_hi, q'*d_lo) rounds d*(q-8) once.
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
  static constexpr int RS = 3, BS = (BN == 256 ? 5 : 8);
  static constexpr int kACols = kBK / 2;               // TMEM columns per A stage
  static constexpr int AS = (512 - BN) / kACols;       // A stages in the rest of TMEM
  static constexpr int kTmemCols = 512;
  static constexpr int kRawBytes = kBM * kRawRow;  // 18432
  static constexpr int kBBytes = BN * 128;
  static constexpr int kOffB = 0;
  static constexpr int kOffRaw = kOffB + BS * kBBytes;
  static constexpr int kOffBar = kOffRaw + RS * kRawBytes;
  static constexpr int kNBar = 2 * RS + 2 * AS + 2 * BS + 1;
  static constexpr int kOffTmem = kOffBar + kNBar * 8;
  static constexpr int kOffAbort = kOffTmem + 8;
  static constexpr int kSmem = kOffAbort + 8 + 1024;  // + slack to align the base to 1024
  static constexpr int kDeqWarps = 8;
  static constexpr int kThreads = 32 * (2 + kDeqWarps);
};

__device__ __forceinline__ uint32_t scale_pair(uint32_t qp, uint32_t dhi2, uint32_t dlo2) {
  return bfma2_u32(qp, dhi2, bmul2_u32(qp, dlo2));
}

// Four consecutive code bytes c0..c3 -> bf16x2 pairs of RN(d*(q-8)):
// lo01 = (c0.lo, c1.lo), lo23 = (c2.lo, c3.lo), hi01 = (c0.hi, c1.hi), hi23 = (c2.hi, c3.hi).
__device__ __forceinline__ void word_to_bf16(uint32_t q, uint32_t dhi2, uint32_t dlo2, uint32_t& lo01,
                                             uint32_t& lo23, uint32_t& hi01, uint32_t& hi23) {
  const uint32_t kMagic = 0x43004300u;  // bf16 128 in both halves
  const uint32_t kSub = 0x43084308u;    // bf16 136
  const uint32_t p = prmt(q, 0u, 0x3120u);  // bytes c0 c2 c1 c3
  lo01 = scale_pair(bsub2_u32(lop3_and_or(p, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
  lo23 = scale_pair(bsub2_u32(lop3_and_or(p >> 8, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
  hi01 = scale_pair(bsub2_u32(lop3_and_or(p >> 4, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
  hi23 = scale_pair(bsub2_u32(lop3_and_or(p >> 12, 0x000F000Fu, kMagic), kSub), dhi2, dlo2);
}

// Exact split of an fp16 scale into bf16 d_hi + d_lo, each broadcast to both halves.
__device__ __forceinline__ void split_scale(uint32_t d_bits, uint32_t& dhi2, uint32_t& dlo2) {
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(d_bits)));
  const __nv_bfloat16 hi = __float2bfloat16_rn(d);
  const __nv_bfloat16 lo = __float2bfloat16_rn(d - __bfloat162float(hi));  // exact: at most 3 bits remain
  const uint32_t h = *reinterpret_cast<const uint16_t*>(&hi), l = *reinterpret_cast<const uint16_t*>(&lo);
  dhi2 = h | (h << 16);
  dlo2 = l | (l << 16);
}

// One block's 16 code bytes (4 words, k-consecutive) -> 16 bf16x2 words
// holding k = 0..31 of the block in order (o[i] = k 2i, 2i+1).
__device__ __forceinline__ void block_words(const uint32_t (&q)[4], uint32_t d_bits, uint32_t* o) {
  uint32_t dhi2, dlo2;
  split_scale(d_bits, dhi2, dlo2);
  // low nibbles of bytes 0..15 are k 0..15, high nibbles are k 16..31
  word_to_bf16(q[0], dhi2, dlo2, o[0], o[1], o[8], o[9]);
  word_to_bf16(q[1], dhi2, dlo2, o[2], o[3], o[10], o[11]);
  word_to_bf16(q[2], dhi2, dlo2, o[4], o[5], o[12], o[13]);
  word_to_bf16(q[3], dhi2, dlo2, o[6], o[7], o[14], o[15]);
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
__global__ void __launch_bounds__(PrefillCfg<BN>::kThreads, 1)
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
      mbar_init(smem_u32(&raw_empty[i]), C::kDeqWarps);
    }
    for (int i = 0; i < C::AS; ++i) {
      mbar_init(smem_u32(&a_full[i]), 4);  // the 4 warps of the group that owns this k step
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
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
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
        const uint32_t a_tmem = tmem_base + BN + as * C::kACols;
        const uint32_t b_addr = sbase + C::kOffB + bs * C::kBBytes;
#pragma unroll
        for (int kk = 0; kk < C::kBK / 16; ++kk)
          umma_bf16_ts(tmem_base, a_tmem + kk * 8, umma_desc_sw128(b_addr + kk * 32), idesc, (ks | kk) != 0);
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
    const int grp = (warp - 2) >> 2;   // 0: even 64-k steps, 1: odd 64-k steps
    const int row = quad * 32 + lane;  // W row within the tile == TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    bool live = true;
    for (int r = 0; r < nr; ++r) {
      const int rslot = r % C::RS;
      if (live) live = mbar_wait_bounded(smem_u32(&raw_full[rslot]), (r / C::RS) & 1, limit_ns, abort_flag, err);
      live = __all_sync(0xFFFFFFFFu, live);
      uint32_t w[36];  // the whole raw row: 8 blocks
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
      for (int j = 0; j < 4; ++j) {  // pair j of the raw row = 64-k step 4r + j
        if ((j & 1) != grp) continue;  // warp-uniform: the groups alternate steps
        const int ks = r * 4 + j, as = ks % C::AS;
        if (live) live = mbar_wait_bounded(smem_u32(&a_empty[as]), ((ks / C::AS) & 1) ^ 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        if (live) {
          // blocks 2j (even) and 2j+1 (odd) of the row = words 9j .. 9j+8
          const uint32_t W0 = w[9 * j], W1 = w[9 * j + 1], W2 = w[9 * j + 2], W3 = w[9 * j + 3], W4 = w[9 * j + 4];
          const uint32_t q0[4] = {prmt(W0, W1, 0x5432u), prmt(W1, W2, 0x5432u), prmt(W2, W3, 0x5432u),
                                  prmt(W3, W4, 0x5432u)};
          const uint32_t q1[4] = {w[9 * j + 5], w[9 * j + 6], w[9 * j + 7], w[9 * j + 8]};
          uint32_t o[32];
          block_words(q0, W0 & 0xFFFFu, o);
          block_words(q1, W4 >> 16, o + 16);
          tmem_st_32x32b_x32(lane_addr + BN + as * C::kACols, o);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (live && lane == 0) mbar_arrive(smem_u32(&a_full[as]));
      }
    }
    // epilogue: this group's half of the accumulator columns
    if (live) live = mbar_wait_bounded(smem_u32(acc_full), 0, limit_ns, abort_flag, err);
    live = __all_sync(0xFFFFFFFFu, live);
    tc_fence_after();
    if (live) {
      const int m = m0 + row;
#pragma unroll 1
      for (int cb = grp * (BN / 64); cb < (grp + 1) * (BN / 64); ++cb) {
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
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// 2-SM variant: a cluster of two CTAs computes a 256 x 256 tile.  CTA r of the
// pair dequantises W rows m0 + 128r .. +127 into its own TMEM and loads x rows
// n0 + 128r .. +127 (half of the B tile) into its own shared memory; the
// leader (r = 0) issues tcgen05.mma.cta_group::2 (M = 256, N = 256), which
// reads A and B from both CTAs and accumulates each CTA's 128 rows in its own
// TMEM.  Each SM thus loads half as much x per flop as the 1-CTA kernel, which
// is bound by that traffic.  Hand-offs:
//   x half of CTA r  -> TMA completing on the leader's b_full (cta_group::2);
//   A stage of CTA r -> its dequant warps arrive on the leader's a_full;
//   MMA completion   -> multicast commit to both CTAs' empty / acc barriers.
struct Prefill2Cfg {
  static constexpr int kBM = 128;       // rows per CTA (256 per pair)
  static constexpr int kBN = 256;       // tokens per pair tile
  static constexpr int kBK = 64;
  static constexpr int kRawK = 256;
  static constexpr int kRawRow = 144;
  static constexpr int RS = 3, BS = 8;
  static constexpr int kACols = kBK / 2;
  static constexpr int AS = (512 - kBN) / kACols;  // 8
  static constexpr int kTmemCols = 512;
  static constexpr int kRawBytes = kBM * kRawRow;        // 18432
  static constexpr int kBBytes = (kBN / 2) * 128;        // 16384: this CTA's half of the x tile
  static constexpr int kOffB = 0;
  static constexpr int kOffRaw = kOffB + BS * kBBytes;
  static constexpr int kOffBar = kOffRaw + RS * kRawBytes;
  static constexpr int kNBar = 2 * RS + 2 * AS + 2 * BS + 1;
  static constexpr int kOffTmem = kOffBar + kNBar * 8;
  static constexpr int kOffAbort = kOffTmem + 8;
  static constexpr int kSmem = kOffAbort + 8 + 1024;
  static constexpr int kDeqWarps = 8;
  static constexpr int kThreads = 32 * (2 + kDeqWarps);
};

__global__ void __launch_bounds__(Prefill2Cfg::kThreads, 1)
    k_prefill2_q4_0(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int N, int M,
                    int K, float* __restrict__ Y, uint64_t limit_ns, uint32_t* err) {
  using C = Prefill2Cfg;
  constexpr int BN = C::kBN;
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
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int ntn = (N + BN - 1) / BN;
  const int m0 = (pair / ntn) * 2 * C::kBM + static_cast<int>(rank) * C::kBM;
  const int n0 = (pair % ntn) * BN;
  const int nk = K / C::kBK;
  const int nr = K / C::kRawK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RS; ++i) {
      mbar_init(smem_u32(&raw_full[i]), 1);
      mbar_init(smem_u32(&raw_empty[i]), C::kDeqWarps);
    }
    for (int i = 0; i < C::AS; ++i) {
      mbar_init(smem_u32(&a_full[i]), 8);  // 4 warps of the owning group in each CTA (leader's copy is used)
      mbar_init(smem_u32(&a_empty[i]), 1);
    }
    for (int i = 0; i < C::BS; ++i) {
      mbar_init(smem_u32(&b_full[i]), 1);  // leader's expect_tx; both halves complete bytes on it
      mbar_init(smem_u32(&b_empty[i]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      uint32_t nraw = 0;
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
        const uint32_t leader_full = mapa_shared(smem_u32(&b_full[slot]), 0);
        if (leader) mbar_arrive_expect_tx(smem_u32(&b_full[slot]), 2 * C::kBBytes);
        tma_load_2d_pair(sbase + C::kOffB + slot * C::kBBytes, &tmX, ks * C::kBK, n0 + static_cast<int>(rank) * (BN / 2),
                         leader_full);
      }
      if (!ok) drain_ring(raw_full, C::RS, nraw, limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16_f32(256, BN);
      for (int ks = 0; ks < nk; ++ks) {
        const int as = ks % C::AS, bs = ks % C::BS;
        if (!mbar_wait_bounded(smem_u32(&a_full[as]), (ks / C::AS) & 1, limit_ns, abort_flag, err)) break;
        if (!mbar_wait_bounded(smem_u32(&b_full[bs]), (ks / C::BS) & 1, limit_ns, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t a_tmem = tmem_base + BN + as * C::kACols;
        const uint32_t b_addr = sbase + C::kOffB + bs * C::kBBytes;
#pragma unroll
        for (int kk = 0; kk < C::kBK / 16; ++kk)
          umma_bf16_ts_pair(tmem_base, a_tmem + kk * 8, umma_desc_sw128(b_addr + kk * 32), idesc, (ks | kk) != 0);
        umma_commit_pair(smem_u32(&a_empty[as]), 3);
        umma_commit_pair(smem_u32(&b_empty[bs]), 3);
      }
      umma_commit_pair(smem_u32(acc_full), 3);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(acc_full), 0) && globaltimer_ns() - t0 < limit_ns) {
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue (both CTAs)
    const int quad = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
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
        if ((j & 1) != grp) continue;
        const int ks = r * 4 + j, as = ks % C::AS;
        if (live) live = mbar_wait_bounded(smem_u32(&a_empty[as]), ((ks / C::AS) & 1) ^ 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        if (live) {
          const uint32_t W0 = w[9 * j], W1 = w[9 * j + 1], W2 = w[9 * j + 2], W3 = w[9 * j + 3], W4 = w[9 * j + 4];
          const uint32_t q0[4] = {prmt(W0, W1, 0x5432u), prmt(W1, W2, 0x5432u), prmt(W2, W3, 0x5432u),
                                  prmt(W3, W4, 0x5432u)};
          const uint32_t q1[4] = {w[9 * j + 5], w[9 * j + 6], w[9 * j + 7], w[9 * j + 8]};
          uint32_t o[32];
          block_words(q0, W0 & 0xFFFFu, o);
          block_words(q1, W4 >> 16, o + 16);
          tmem_st_32x32b_x32(lane_addr + BN + as * C::kACols, o);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (live && lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&a_full[as]), 0));
      }
    }
    if (live) live = mbar_wait_bounded(smem_u32(acc_full), 0, limit_ns, abort_flag, err);
    live = __all_sync(0xFFFFFFFFu, live);
    tc_fence_after();
    if (live) {
      const int m = m0 + row;
#pragma unroll 1
      for (int cb = grp * (BN / 64); cb < (grp + 1) * (BN / 64); ++cb) {
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
  cluster_sync();  // neither CTA frees TMEM or leaves while the pair's MMAs or remote arrivals may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

cudaError_t launch_prefill2(const CUtensorMap* tmW, const CUtensorMap* tmX, int N, int M, int K, float* Y,
                            uint64_t limit_ns, cudaStream_t s) {
  using C = Prefill2Cfg;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill2_q4_0, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int pairs = ((M + 2 * C::kBM - 1) / (2 * C::kBM)) * ((N + C::kBN - 1) / C::kBN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_prefill2_q4_0, *tmW, *tmX, N, M, K, Y, limit_ns, device_error_word());
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

int g_bn_override = 0;  // 0: choose by shape; 128 or 256: force the tile width (tuning)

int prefill_bn(int64_t N) {
  if (g_bn_override) return g_bn_override;
  return N <= 128 ? 128 : 256;
}

// 0 (default): 1-CTA kernel with 128 x prefill_bn tiles; 1: 2-SM pair kernel (256 x 256 tiles).
int g_pair_mode = 0;
bool use_pair(int64_t N) { return g_pair_mode && g_bn_override == 0 && N > 128; }

}  // namespace

void set_prefill_bn_override(int bn) { g_bn_override = bn; }
int get_prefill_bn_override() { return g_bn_override; }

void prefill_boxes(int64_t N, uint32_t* w_box_x_bytes, uint32_t* w_box_rows, uint32_t* x_box_k,
                   uint32_t* x_box_rows) {
  *w_box_x_bytes = 144;
  *w_box_rows = 128;
  *x_box_k = 64;
  *x_box_rows = use_pair(N) ? 128u : static_cast<uint32_t>(prefill_bn(N));
}

void set_prefill_pair_mode(int on) { g_pair_mode = on ? 1 : 0; }
int get_prefill_pair_mode() { return g_pair_mode; }

cudaError_t launch_prefill(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t N, int64_t M, int64_t K,
                           float* Y, uint64_t wait_limit_ns, cudaStream_t s) {
  const int n = static_cast<int>(N), m = static_cast<int>(M), k = static_cast<int>(K);
  if (use_pair(N)) return launch_prefill2(tmW, tmX, n, m, k, Y, wait_limit_ns, s);
  if (prefill_bn(N) == 128) return launch_prefill_bn<128>(tmW, tmX, n, m, k, Y, wait_limit_ns, s);
  return launch_prefill_bn<256>(tmW, tmX, n, m, k, Y, wait_limit_ns, s);
}

}  // namespace gq
