// Q4_K superblocks (256 elements in 144 bytes): fp16 d (bytes 0-1), fp16 dmin
// (2-3), 12 bytes of 6-bit sub-block scales and mins (4-15), 128 bytes of
// 4-bit codes (16-143; byte 32 g + l holds element 64 g + l in its low nibble
// and 64 g + 32 + l in its high nibble). Element e of sub-block j = e / 32 is
// d sc_j q - dmin m_j. This is the GGUF superblock layout, which the pages
// dispatch (aprender-serve qwen35_dequant_f32, grid (n, k.div_ceil(256)))
// without printing it.
#pragma once

#include <cstdint>

namespace apr {

// scale and min of sub-block j (0..7) from the 12 packed bytes s: bytes 0-3
// hold scales 0-3 in their low 6 bits and bytes 4-7 mins 0-3; bytes 8-11 hold
// scales 4-7 (low nibble) and mins 4-7 (high nibble), whose top two bits are
// the top two bits of bytes 0-3 and 4-7
__host__ __device__ __forceinline__ void q4k_scale_min(const uint8_t* s, uint32_t j, uint32_t& sc, uint32_t& m) {
  if (j < 4) {
    sc = s[j] & 63u;
    m = s[j + 4] & 63u;
  } else {
    sc = (s[j + 4] & 15u) | ((uint32_t)(s[j - 4] >> 6) << 4);
    m = (uint32_t)(s[j + 4] >> 4) | ((uint32_t)(s[j] >> 6) << 4);
  }
}

// the same from the three packed words w[0..2] (bytes 4-15 of the
// superblock), by register selects (no indexed array)
__device__ __forceinline__ void q4k_scale_min_w(const uint32_t* w, uint32_t j, uint32_t& sc, uint32_t& m) {
  const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
  auto byte = [&](uint32_t b) {
    const uint32_t word = b < 4 ? w0 : (b < 8 ? w1 : w2);
    return (word >> (8 * (b & 3))) & 0xFFu;
  };
  if (j < 4) {
    sc = byte(j) & 63u;
    m = byte(j + 4) & 63u;
  } else {
    sc = (byte(j + 4) & 15u) | ((byte(j - 4) >> 6) << 4);
    m = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
  }
}

}  // namespace apr
