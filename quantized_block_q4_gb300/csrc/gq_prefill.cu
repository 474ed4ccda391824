// K0: fp32 -> bf16 conversion of the activations, and K3: the prefill
// MUL_MAT against Q4_0 weights on tcgen05 tensor cores.
//
// K3 computes Y[n][m] = sum_k w[m][k] * x[n][k] for a 128-row x BN-token tile
// per CTA ("GGUF loading, mmap and tensor placement", step six: the MUL_MAT
// probe with a 512-token batch; "Binding GGUF weights to the compute graph",
// section 2.3: the kernel reads the blocks and dequantises them itself).
// Roles (608 threads):
//   warp 0  TMA producer of raw W rows (128 x 144 bytes = 256 weights each)
//           into a shared-memory ring; it runs ahead of the x producer by
//           up to the ring depth (12 steps of 64 k), which hides HBM latency.
//   warp 18 TMA producer of bf16 x tiles (BN x 64, 128-byte swizzle).
//   warp 1  allocates 512 TMEM columns: the fp32 accumulator (BN columns) and
//           a ring of A stages (32 columns = 64 bf16 k each).  One thread
//           issues tcgen05.mma with A read from tensor memory and B (x) from
//           shared memory (M=128, N=BN, K=16, bf16 x bf16 -> fp32) and
//           commits to the rings' "empty" barriers.
//   warps 2-17 dequantise in four groups of four warps: group g takes the
//           64-k step g of every 256-k chunk; a thread owns one W row of the
//           tile, i.e. one TMEM lane, and stores RN_bf16(d*(q-8)) for the
//           step's 64 weights into its lane with one tcgen05.st.  Then they
//           read the accumulator with tcgen05.ld (warp w reads TMEM lanes
//           32*(w%4)..; group g takes a quarter of the columns) and store
//           fp32 Y, consecutive lanes writing consecutive m.
// Work split: a CTA runs a contiguous range of (tile, 256-k chunk) units,
// possibly several tiles (stream-K, PrefillWork below); the rings and the
// accumulator hand-off carry over from one tile to the next.
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
  static constexpr int kRawK = 256;     // k per raw W stage (one work unit)
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
  static constexpr int kNBar = 2 * RS + 2 * AS + 2 * BS + 2;
  static constexpr int kOffTmem = kOffBar + kNBar * 8;
  static constexpr int kOffAbort = kOffTmem + 8;
  static constexpr int kOffFlag = kOffAbort + 8;       // two words: "this CTA reduces the tile"
  static constexpr int kSmem = kOffFlag + 8 + 1024;   // + slack to align the base to 1024
  static constexpr int kDeqWarps = 16;  // warps 2..17, 4 groups of 4: one 64-k step of each 256-k chunk per group
  static constexpr int kXWarp = 2 + kDeqWarps;  // warp 0 loads W, warp 1 issues MMAs, the last warp loads x
  static constexpr int kThreads = 32 * (3 + kDeqWarps);
  static constexpr int kSlotFloats = BN * kBM;         // one partial tile, [column][row]
};

// Stream-K split of a launch: the T output tiles x nr chunks of 256 k are
// U = T*nr work units in tile-major order; CTA g of G takes the contiguous
// units [g*U/G, (g+1)*U/G).  A CTA thus runs one or more segments (a tile
// and a range of its chunks); only its first and last segments can cover
// part of a tile.  With G == T every CTA runs exactly one whole tile.
struct PrefillWork {
  int64_t units;  // U
  int nr;         // chunks per tile, K / 256
  int ntn;        // token tiles per 128-row block; tile t = (t / ntn, t % ntn)
  float* ws;      // 2 partial-tile slots per CTA (nullptr when no tile is split)
  int* count;     // per tile: partials published so far; zero at launch
};

__device__ __forceinline__ int64_t sk_begin(int64_t g, int64_t grid, int64_t units) { return g * units / grid; }
// The CTA whose range holds unit u.
__device__ __forceinline__ int sk_owner(int64_t u, int64_t grid, int64_t units) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}
// Partial slot of CTA g for tile t: 0 for the CTA's first tile, 1 for its last.
__device__ __forceinline__ int64_t sk_slot(int g, int64_t t, int64_t grid, const PrefillWork& wk) {
  return 2 * static_cast<int64_t>(g) + (sk_begin(g, grid, wk.units) / wk.nr == t ? 0 : 1);
}

struct Seg {
  int64_t t;  // tile
  int r0, r1; // chunk range [r0, r1) of the tile
};
__device__ __forceinline__ Seg seg_at(int64_t u, int64_t ue, int nr) {
  Seg sg;
  sg.t = u / nr;
  sg.r0 = static_cast<int>(u - sg.t * nr);
  sg.r1 = static_cast<int>(sg.r0 + ue - u < nr ? sg.r0 + ue - u : nr);
  return sg;
}

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
                   float* __restrict__ Y, const PrefillWork wk, uint64_t limit_ns, uint32_t* err) {
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
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  volatile int* reduce_flag = reinterpret_cast<volatile int*>(smem + C::kOffFlag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t grid = gridDim.x;
  const int64_t ub = sk_begin(blockIdx.x, grid, wk.units), ue = sk_begin(blockIdx.x + 1, grid, wk.units);
  const int nr = wk.nr;

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
    mbar_init(smem_u32(acc_empty), C::kDeqWarps);
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
    // ------------------------------------------------------------ W producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      uint32_t nraw = 0;
      bool ok = true;
      for (int64_t u = ub; u < ue && ok;) {
        const Seg sg = seg_at(u, ue, nr);
        const int m0 = static_cast<int>(sg.t / wk.ntn) * C::kBM;
        for (int r = sg.r0; r < sg.r1; ++r) {
          const uint32_t slot = nraw % C::RS;
          if (!mbar_wait_bounded(smem_u32(&raw_empty[slot]), ((nraw / C::RS) & 1) ^ 1, limit_ns, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&raw_full[slot]), C::kRawBytes);
          tma_load_2d(sbase + C::kOffRaw + slot * C::kRawBytes, &tmW, r * C::kRawRow, m0, smem_u32(&raw_full[slot]));
          ++nraw;
        }
        u += sg.r1 - sg.r0;
      }
      if (!ok) drain_ring(raw_full, C::RS, nraw, limit_ns);
    }
  } else if (warp == C::kXWarp) {
    // ------------------------------------------------------------ x producer
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      uint32_t nb = 0;
      bool ok = true;
      for (int64_t u = ub; u < ue && ok;) {
        const Seg sg = seg_at(u, ue, nr);
        const int n0 = static_cast<int>(sg.t % wk.ntn) * BN;
        for (int ks = 4 * sg.r0; ks < 4 * sg.r1; ++ks) {
          const uint32_t bs = nb % C::BS;
          if (!mbar_wait_bounded(smem_u32(&b_empty[bs]), ((nb / C::BS) & 1) ^ 1, limit_ns, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&b_full[bs]), C::kBBytes);
          tma_load_2d(sbase + C::kOffB + bs * C::kBBytes, &tmX, ks * C::kBK, n0, smem_u32(&b_full[bs]));
          ++nb;
        }
        u += sg.r1 - sg.r0;
      }
      if (!ok) drain_ring(b_full, C::BS, nb, limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16_f32(128, BN);
      uint32_t c = 0, seg = 0;
      bool ok = true;
      for (int64_t u = ub; u < ue && ok;) {
        const Seg sg = seg_at(u, ue, nr);
        // the previous segment's epilogue must have read the accumulator
        if (seg > 0 && !mbar_wait_bounded(smem_u32(acc_empty), (seg - 1) & 1, limit_ns, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 4 * sg.r0; ks < 4 * sg.r1; ++ks, ++c) {
          const uint32_t as = c % C::AS, bs = c % C::BS;
          if (!mbar_wait_bounded(smem_u32(&a_full[as]), (c / C::AS) & 1, limit_ns, abort_flag, err) ||
              !mbar_wait_bounded(smem_u32(&b_full[bs]), (c / C::BS) & 1, limit_ns, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + BN + as * C::kACols;
          const uint32_t b_addr = sbase + C::kOffB + bs * C::kBBytes;
#pragma unroll
          for (int kk = 0; kk < C::kBK / 16; ++kk)
            umma_bf16_ts(tmem_base, a_tmem + kk * 8, umma_desc_sw128(b_addr + kk * 32), idesc,
                         ks != 4 * sg.r0 || kk != 0);
          umma_commit(smem_u32(&a_empty[as]));
          umma_commit(smem_u32(&b_empty[bs]));
        }
        umma_commit(smem_u32(acc_full));  // also on the error path: tracks every MMA issued so far
        ++seg;
        u += sg.r1 - sg.r0;
      }
      // Do not leave while MMAs issued by this thread may still run: the last
      // commit tracks all of them.
      if (seg > 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(acc_full), (seg - 1) & 1) && globaltimer_ns() - t0 < limit_ns) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int grp = (warp - 2) >> 2;     // 64-k step grp of every 256-k chunk; then columns grp/4 of the tile
    const int row = quad * 32 + lane;    // W row within the tile == TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const bool e0 = warp == 2 && lane == 0;
    constexpr int kCbPerGrp = BN / 128;  // 32-column blocks of the accumulator per group
    const int cb0 = grp * kCbPerGrp, cb1 = cb0 + kCbPerGrp;
    // This group's 36 bytes of a raw row start at byte 36*grp: read the three
    // 16-byte words that cover them; word grp of those is the first one.
    const int raw_off = row * C::kRawRow + (36 * grp & ~15);
    bool live = true;
    uint32_t cr = 0, c = 0, seg = 0;
    for (int64_t u = ub; u < ue;) {
      const Seg sg = seg_at(u, ue, nr);
      for (int r = sg.r0; r < sg.r1; ++r, ++cr, c += 4) {
        const uint32_t rslot = cr % C::RS;
        const uint32_t as = (c + grp) % C::AS;
        if (live) live = mbar_wait_bounded(smem_u32(&raw_full[rslot]), (cr / C::RS) & 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        uint32_t v[12];
        if (live) {
          const uint4* src = reinterpret_cast<const uint4*>(smem + C::kOffRaw + rslot * C::kRawBytes + raw_off);
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            const uint4 x = src[i];
            v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
          }
        }
        __syncwarp();
        if (live && lane == 0) mbar_arrive(smem_u32(&raw_empty[rslot]));
        // Dequantise first, then wait for the A stage: only the store is left
        // between the stage becoming free and the MMA that reads it.
        uint32_t o[32];
        {
          uint32_t w[9];  // blocks 2*grp and 2*grp+1 of the row
#pragma unroll
          for (int i = 0; i < 9; ++i)
            w[i] = grp == 0 ? v[i] : grp == 1 ? v[i + 1] : grp == 2 ? v[i + 2] : v[i + 3];
          const uint32_t q0[4] = {prmt(w[0], w[1], 0x5432u), prmt(w[1], w[2], 0x5432u), prmt(w[2], w[3], 0x5432u),
                                  prmt(w[3], w[4], 0x5432u)};
          const uint32_t q1[4] = {w[5], w[6], w[7], w[8]};
          block_words(q0, w[0] & 0xFFFFu, o);
          block_words(q1, w[4] >> 16, o + 16);
        }
        if (live) live = mbar_wait_bounded(smem_u32(&a_empty[as]), (((c + grp) / C::AS) & 1) ^ 1, limit_ns, abort_flag, err);
        live = __all_sync(0xFFFFFFFFu, live);
        if (live) {
          tmem_st_32x32b_x32(lane_addr + BN + as * C::kACols, o);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (live && lane == 0) mbar_arrive(smem_u32(&a_full[as]));
      }

      // ---- epilogue of this segment: this group's quarter of the accumulator columns
      if (live) live = mbar_wait_bounded(smem_u32(acc_full), seg & 1, limit_ns, abort_flag, err);
      live = __all_sync(0xFFFFFFFFu, live);
      tc_fence_after();
      const int m = static_cast<int>(sg.t / wk.ntn) * C::kBM + row;
      const int n0 = static_cast<int>(sg.t % wk.ntn) * BN;
      if (sg.r0 == 0 && sg.r1 == nr) {
        if (live) {
#pragma unroll 1
          for (int cb = cb0; cb < cb1; ++cb) {
            uint32_t v32[32];
            tmem_ld_32x32b_x32(lane_addr + cb * 32, v32);
            tmem_ld_wait();
            if (m < M) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int n = n0 + cb * 32 + jj;
                if (n < N) Y[static_cast<size_t>(n) * M + m] = __uint_as_float(v32[jj]);
              }
            }
          }
        }
      } else {
        // Part of a split tile.  The CTA that sees every other split published
        // reduces: partial sums are added in the order of their k ranges, so
        // the result does not depend on which CTA finishes last.
        const int64_t t = sg.t;
        const int ga = sk_owner(t * nr, grid, wk.units), gb = sk_owner(t * nr + nr - 1, grid, wk.units);
        const int nsplit = gb - ga + 1;
        volatile int* flag = reduce_flag + (seg & 1);
        if (e0) *flag = live && ld_acquire_gpu(wk.count + t) == nsplit - 1;
        named_bar_sync(1, 32 * C::kDeqWarps);
        int last = *flag;
        if (!last) {
          if (live) {  // publish this split's partial tile
            float* p = wk.ws + sk_slot(blockIdx.x, t, grid, wk) * C::kSlotFloats + row;
#pragma unroll 1
            for (int cb = cb0; cb < cb1; ++cb) {
              uint32_t v32[32];
              tmem_ld_32x32b_x32(lane_addr + cb * 32, v32);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) __stcg(p + (cb * 32 + jj) * C::kBM, __uint_as_float(v32[jj]));
            }
          }
          __threadfence();
          named_bar_sync(1, 32 * C::kDeqWarps);
          if (e0) *flag = live && atomicAdd(wk.count + t, 1) == nsplit - 1;
          named_bar_sync(1, 32 * C::kDeqWarps);
          last = *flag;
        }
        if (last && live) {
          __threadfence();
#pragma unroll 1
          for (int hb = 2 * cb0; hb < 2 * cb1; ++hb) {  // 16-column halves of this group's blocks
            float acc[16];
#pragma unroll 1
            for (int g = ga; g <= gb; ++g) {
              uint32_t q[16];  // split g's partial sums of these 16 columns
              if (g == static_cast<int>(blockIdx.x)) {
                tmem_ld_32x32b_x16(lane_addr + hb * 16, q);
                tmem_ld_wait();
              } else {
                const float* p = wk.ws + sk_slot(g, t, grid, wk) * C::kSlotFloats + hb * 16 * C::kBM + row;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) q[jj] = __float_as_uint(__ldcg(p + jj * C::kBM));
              }
              if (g == ga) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) acc[jj] = __uint_as_float(q[jj]);
              } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) acc[jj] += __uint_as_float(q[jj]);
              }
            }
            if (m < M) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                const int n = n0 + hb * 16 + jj;
                if (n < N) Y[static_cast<size_t>(n) * M + m] = acc[jj];
              }
            }
          }
          if (e0) wk.count[t] = 0;  // every split has arrived: leave the counter as found
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty));
      ++seg;
      u += sg.r1 - sg.r0;
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

int64_t g_streamk = 1;  // 0: one CTA per tile; 1: stream-K when it balances the SMs better; >= 2: that many CTAs

// CTAs for T tiles of nr chunks each: T (one tile per CTA) unless spreading
// the T*nr units evenly over the SMs (at least 4 units per CTA, plus about
// 2 units' worth of time for the split tiles' fix-up) is 10% faster.
int64_t prefill_grid(int64_t T, int64_t nr, bool allow_scratch) {
  const int64_t U = T * nr;
  if (!allow_scratch || g_streamk == 0) return T;
  if (g_streamk >= 2) return std::min(g_streamk, U);
  const int64_t P = device_info().sm_count > 0 ? device_info().sm_count : 1;
  const int64_t g = std::min(P, std::max<int64_t>(1, U / 4));
  const double t_dp = static_cast<double>((T + P - 1) / P) * static_cast<double>(nr);
  const double t_sk = static_cast<double>((U + g - 1) / g) + 2.0;
  return t_sk < 0.9 * t_dp ? g : T;
}

template <int BN>
cudaError_t launch_prefill_bn(const CUtensorMap* tmW, const CUtensorMap* tmX, int N, int M, int K, float* Y,
                              uint64_t limit_ns, bool allow_scratch, cudaStream_t s) {
  using C = PrefillCfg<BN>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill_q4_0<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t ntn = (N + BN - 1) / BN;
  const int64_t T = ((M + C::kBM - 1) / C::kBM) * ntn;
  const int64_t nr = K / C::kRawK;
  int64_t grid = prefill_grid(T, nr, allow_scratch);
  PrefillWork wk{T * nr, static_cast<int>(nr), static_cast<int>(ntn), nullptr, nullptr};
  void* scratch = nullptr;
  if (T % grid != 0) {  // some tile is split across CTAs: partial-tile slots and arrival counters
    const size_t ws_bytes = static_cast<size_t>(2 * grid) * C::kSlotFloats * sizeof(float);
    const size_t bytes = ws_bytes + static_cast<size_t>(T) * sizeof(int);
    if (scratch_alloc(&scratch, bytes, s) == cudaSuccess &&
        cudaMemsetAsync(static_cast<uint8_t*>(scratch) + ws_bytes, 0, static_cast<size_t>(T) * sizeof(int), s) ==
            cudaSuccess) {
      wk.ws = static_cast<float*>(scratch);
      wk.count = reinterpret_cast<int*>(static_cast<uint8_t*>(scratch) + ws_bytes);
    } else {  // no scratch: one tile per CTA
      cudaGetLastError();
      if (scratch) scratch_free(scratch, s);
      scratch = nullptr;
      grid = T;
    }
  }
  k_prefill_q4_0<BN><<<static_cast<unsigned>(grid), C::kThreads, C::kSmem, s>>>(*tmW, *tmX, N, M, Y, wk, limit_ns,
                                                                                device_error_word());
  cudaError_t e = cudaGetLastError();
  if (scratch) {
    cudaError_t f = scratch_free(scratch, s);
    if (e == cudaSuccess) e = f;
  }
  return e;
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
void set_prefill_streamk(int64_t v) { g_streamk = v; }
int64_t get_prefill_streamk() { return g_streamk; }
int get_prefill_pair_mode() { return g_pair_mode; }

cudaError_t launch_prefill(const CUtensorMap* tmW, const CUtensorMap* tmX, int64_t N, int64_t M, int64_t K,
                           float* Y, uint64_t wait_limit_ns, bool allow_scratch, cudaStream_t s) {
  const int n = static_cast<int>(N), m = static_cast<int>(M), k = static_cast<int>(K);
  if (use_pair(N)) return launch_prefill2(tmW, tmX, n, m, k, Y, wait_limit_ns, s);
  if (prefill_bn(N) == 128) return launch_prefill_bn<128>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, s);
  return launch_prefill_bn<256>(tmW, tmX, n, m, k, Y, wait_limit_ns, allow_scratch, s);
}

}  // namespace gq
