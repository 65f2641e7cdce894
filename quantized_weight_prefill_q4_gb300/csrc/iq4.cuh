// IQ4_XS superblocks (256 elements in 136 bytes): fp16 d (bytes 0-1), a
// little-endian word of high scale bits (2-3), four bytes of low scale
// nibbles (4-7), then 128 bytes of 4-bit codes, 16 a 32-element sub-block
// (byte 8 + 16 j + l holds element 32 j + l in its low nibble and
// 32 j + 16 + l in its high nibble). Sub-block j's six-bit scale ls_j takes
// nibble j % 2 of byte 4 + j / 2 as its low bits and bits 2 j, 2 j + 1 of
// the word as its top two; a code c stands for entry c of the 16-value
// non-linear IQ4_NL code book, and the weight is d (ls_j - 32) book[c].
// This is the GGUF superblock layout and code book, which the pages dispatch
// (aprender-serve Iq4XsDequantKernel, iq4_xs_dequant_to_f32, grid
// (n, k.div_ceil(256))) without printing either.
#pragma once

#include <cstdint>

namespace apr {

// The book as bytes book[c] + 128 (all in 1 .. 241): entries 0-7, each below
// 128, and the low seven bits of entries 8-15 (each of which is 128 + its
// low seven bits)
constexpr uint32_t kIq4Lo0 = 0x3F2D1801u, kIq4Lo1 = 0x766A5D4Fu;  // -127 -104 -83 -65 | -49 -35 -22 -10
constexpr uint32_t kIq4Hi0 = 0x26190D01u, kIq4Hi1 = 0x71594535u;  // 1 13 25 38 | 53 69 89 113

// prmt.b32 in its default mode: result byte i is byte (s_i & 7) of {b, a}
// (a the low four), or, when bit 3 of selector nibble s_i is set, that byte's
// sign bit copied into all eight bits. Only the low 16 bits of s are read.
__device__ __forceinline__ uint32_t prmt_sign(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

// Byte i of the result is book[c_i] + 128 for the code c_i in nibble i of s
// (i = 0..3); bit 7 of byte i of fl must be bit 3 of c_i. Codes below 8 read
// the low table; codes of 8 and above have bit 3 set, which turns that read
// into a copy of a clear sign bit (0), while the flipped selector reads the
// high table for them and gives 0 for the others; the set bit 7 adds 128.
__device__ __forceinline__ uint32_t iq4_lookup4(uint32_t s, uint32_t fl) {
  const uint32_t lo = prmt_sign(kIq4Lo0, kIq4Lo1, s);
  const uint32_t hi = prmt_sign(kIq4Hi0, kIq4Hi1, s ^ 0x8888u);
  return lo | hi | (fl & 0x80808080u);
}

// One word x of a sub-block's code bytes 4 v .. 4 v + 3 (byte i: element
// 4 v + i in its low nibble, "A_i", and 16 + 4 v + i in its high nibble,
// "B_i"): u0 = (A0, B0, A1, B1) and u1 = (A2, B2, A3, B3) as book + 128, one a
// byte. The nibbles of x are A0 B0 A1 B1 A2 B2 A3 B3 from the bottom, so x
// and x >> 16 are the selectors themselves; the flags (bit 3 of each nibble
// at bit 7 of its byte) come from x and x << 4 byte by byte.
__device__ __forceinline__ void iq4_word(uint32_t x, uint32_t& u0, uint32_t& u1) {
  const uint32_t x4 = x << 4;
  u0 = iq4_lookup4(x, __byte_perm(x, x4, 0x1504));
  u1 = iq4_lookup4(x >> 16, __byte_perm(x, x4, 0x3726));
}

// The same for four codes held one a byte (each below 16), in their order
__device__ __forceinline__ uint32_t iq4_bytes4(uint32_t q) {
  const uint32_t t = q | (q >> 4);  // byte 0: c0 | c1 << 4, byte 2: c2 | c3 << 4
  return iq4_lookup4(__byte_perm(t, 0u, 0x4420), q << 4);
}

// ls_j - 32 of sub-block j from w0 = d | high scale bits << 16 and w1 = the
// four low-nibble bytes
__device__ __forceinline__ int iq4_scale(uint32_t w0, uint32_t w1, uint32_t j) {
  return (int)(((w1 >> (4 * j)) & 15u) | (((w0 >> (16 + 2 * j)) & 3u) << 4)) - 32;
}

}  // namespace apr
