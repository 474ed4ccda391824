// Q4_K super-block fields shared by the kernels that read Q4_K weights.
//
// A 144-byte super-block of 256 weights (the k-quant of "Architecture and
// module overview", quantisation-format section; GGUF layout): fp16 d at
// bytes 0-1, fp16 dmin at 2-3, sixteen 6-bit fields at 4-15, 128 code bytes
// at 16-143; w = d*sc_j*q - dmin*m_j for sub-block j (32 weights).  With the
// field bytes as three little-endian words F0 = bytes 4-7, F1 = 8-11,
// F2 = 12-15:
//   j < 4:  sc_j = bits 0-5 of byte j of F0,  m_j = bits 0-5 of byte j of F1;
//   j >= 4: bits 0-3 of sc_j / m_j = the low / high nibble of byte j-4 of F2,
//           bits 4-5 = the top two bits of byte j-4 of F0 / F1.
#pragma once

#include <cstdint>

namespace gq {

constexpr int kQ4KWeights = 256;  // weights per super-block
constexpr int kQ4KBytes = 144;    // bytes per super-block

template <int J>
__device__ __forceinline__ void q4k_scale_min(uint32_t F0, uint32_t F1, uint32_t F2, uint32_t& sc, uint32_t& mn) {
  static_assert(J >= 0 && J < 8, "sub-block index");
  if constexpr (J < 4) {
    sc = (F0 >> (8 * J)) & 63u;
    mn = (F1 >> (8 * J)) & 63u;
  } else {
    constexpr int sh = 8 * (J - 4);
    sc = ((F2 >> sh) & 15u) | (((F0 >> (sh + 6)) & 3u) << 4);
    mn = ((F2 >> (sh + 4)) & 15u) | (((F1 >> (sh + 6)) & 3u) << 4);
  }
}

// The same for a sub-block index known only at run time.
__device__ __forceinline__ void q4k_scale_min_rt(uint32_t F0, uint32_t F1, uint32_t F2, int j, uint32_t& sc,
                                                 uint32_t& mn) {
  const int sh = 8 * (j & 3);
  if (j < 4) {
    sc = (F0 >> sh) & 63u;
    mn = (F1 >> sh) & 63u;
  } else {
    sc = ((F2 >> sh) & 15u) | (((F0 >> (sh + 6)) & 3u) << 4);
    mn = ((F2 >> (sh + 4)) & 15u) | (((F1 >> (sh + 6)) & 3u) << 4);
  }
}

}  // namespace gq
