// Decode and dot-product helpers shared by the bulk-copy GEMV kernels
// (gemv_bulk.cu, gemv_rows.cu): exact fp32 products of Q4_0 / Q8_0 codes with
// a per-CTA table of X built in shared memory.
//
// Decode without integer-to-float conversions: a 4-bit code n sitting at bit
// offset s < 23 of a 32-bit word becomes the float 2^23 + n 2^s when the
// exponent bits of 2^23 are OR-ed in, and subtracting 2^23 + 8 2^s leaves
// (n - 8) 2^s exactly (an int8 code moved to the low byte gives 2^23 + b + 128
// the same way). The 2^-s is folded into the table of X (scaled by exact powers
// of two), so one packed fp32 FMA does each product. Per block a lane sums its
// products in fp32 and scales by d.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"

namespace apr {
namespace gemv {

constexpr int XPAIR = 68;  // floats per block pair (64 columns) in the X table (64 + pad)

__device__ __forceinline__ float magic(uint32_t u) { return __uint_as_float(u | 0x4B000000u); }

// Q4_0: bit offset s at which each of the 8 codes of a payload word is read,
// in table order (lo nibble of byte m, hi nibble of byte m), m = 0..3. Codes
// must sit below bit 23 (the exponent LSB of 2^23): the lo nibbles of bytes 0-2
// and the hi nibbles of bytes 0-1 are read in place, the last three from the
// word shifted right by 12.
__host__ __device__ constexpr int q4_shift(int slot) {
  return slot == 0 ? 0 : slot == 1 ? 4 : slot == 2 ? 8 : slot == 3 ? 12 : slot == 4 ? 16 : slot == 5 ? 8
                                                                                    : slot == 6 ? 12 : 16;
}

// Table layout of one block pair (64 floats + pad): Q4_0 slot 32 blk + 8 word +
// 2 m + hi holds element 32 blk + 16 hi + 4 word + m (byte m of payload word
// `word`, low or high nibble), scaled by 2^-s with s = q4_shift(2 m + hi), in
// the order q4_word_dot consumes them; Q8_0 slot e holds element e.
// Maps element offset e (0..63) to its slot and scale exponent.
template <int QT>
__device__ __forceinline__ void elem_slot(int e, int& slot, int& s) {
  if (QT == kQ4_0) {
    const int blk = e >> 5, ee = e & 31, hi = ee >> 4, within = ee & 15, word = within >> 2, m = within & 3;
    const int q = 2 * m + hi;
    slot = 32 * blk + 8 * word + q;
    s = q4_shift(q);
  } else {
    slot = e;
    s = 0;
  }
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Products of one Q4_0 payload word with its 8 table entries (xa = slots
// 8i..8i+3, xb = 8i+4..8i+7), accumulated into acc.
// Subtracted constants 2^23 + 8 * 2^s.
constexpr float kC0 = 8388616.0f, kC4 = 8388736.0f, kC8 = 8390656.0f, kC12 = 8421376.0f, kC16 = 8912896.0f;

// Four independent accumulators (one per code pair of a word), so that the
// FMA chains stay short: the products are exact, only the order of the fp32
// sums changes. Each pair of codes takes one packed subtraction and one packed
// FMA (the f32x2 forms of sm_100 and later; each lane rounds exactly as the
// scalar instruction does), measured 2-6 % faster than the scalar forms.
__device__ __forceinline__ void q4_word_dot(uint32_t p, float4 xa, float4 xb, float2 (&acc)[4]) {
  const uint32_t p12 = p >> 12;
  const float2 f0 = make_float2(magic(p & 0xFu), magic(p & 0xF0u));
  const float2 f1 = make_float2(magic(p & 0xF00u), magic(p & 0xF000u));
  const float2 f2v = make_float2(magic(p & 0xF0000u), magic(p12 & 0xF00u));
  const float2 f3 = make_float2(magic(p12 & 0xF000u), magic(p12 & 0xF0000u));
  acc[0] = __ffma2_rn(__fadd2_rn(f0, make_float2(-kC0, -kC4)), make_float2(xa.x, xa.y), acc[0]);
  acc[1] = __ffma2_rn(__fadd2_rn(f1, make_float2(-kC8, -kC12)), make_float2(xa.z, xa.w), acc[1]);
  acc[2] = __ffma2_rn(__fadd2_rn(f2v, make_float2(-kC16, -kC8)), make_float2(xb.x, xb.y), acc[2]);
  acc[3] = __ffma2_rn(__fadd2_rn(f3, make_float2(-kC12, -kC16)), make_float2(xb.z, xb.w), acc[3]);
}

// Products of one Q8_0 payload word (4 int8, elements 4i..4i+3) with x, into
// acc[base] and acc[base + 1].
__device__ __forceinline__ void q8_word_dot(uint32_t q, float4 x, float2 (&acc)[4], int base) {
  const uint32_t u = q ^ 0x80808080u;  // byte + 128, unsigned
  const float2 fa = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                                __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)));
  const float2 fb = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                                __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)));
  const float2 c = make_float2(-8388736.0f, -8388736.0f);
  acc[base] = __ffma2_rn(__fadd2_rn(fa, c), make_float2(x.x, x.y), acc[base]);
  acc[base + 1] = __ffma2_rn(__fadd2_rn(fb, c), make_float2(x.z, x.w), acc[base + 1]);
}

// Sum of the four accumulators in a fixed order.
__device__ __forceinline__ float acc_sum(const float2 (&a)[4]) {
  return ((a[0].x + a[0].y) + (a[1].x + a[1].y)) + ((a[2].x + a[2].y) + (a[3].x + a[3].y));
}

__device__ __forceinline__ float half_bits(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }


// Builds the X table: for token t < T and block pair P < k / 64, table entry
// xt[(t * (k / 64) + P) * XPAIR + slot] = X[t][64 P + e] * 2^-s with
// (slot, s) = elem_slot(e). Threads tid = 0..nthreads-1 of the CTA take part;
// coalesced float4 loads, eight a thread in flight before any store.
template <int QT>
__device__ __forceinline__ void build_x_table(const float* __restrict__ X, int T, int k, float* xt, int tid,
                                              int nthreads) {
  const int npk = k / 64;
  const int k4 = k / 4;
  const int total4 = T * k4;
  const float4* X4 = reinterpret_cast<const float4*>(X);
  constexpr int U = 8;
  for (int base = tid; base < total4; base += U * nthreads) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * nthreads;
      v[u] = i4 < total4 ? __ldg(X4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * nthreads;
      if (i4 < total4) {
        const int t = i4 / k4;
        const int e0 = (i4 - t * k4) * 4;
        float* dst = xt + (t * npk + (e0 >> 6)) * XPAIR;
        const float vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          int slot, sh;
          elem_slot<QT>((e0 & 63) + c, slot, sh);
          dst[slot] = vv[c] * __uint_as_float((uint32_t)(127 - sh) << 23);  // exact 2^-sh
        }
      }
    }
  }
}

// acc[t] += dot(block pair at `src` (two blocks, 4-byte aligned), X table pair
// at `xp`) for t < T; `tstride` floats between the tokens' tables.
template <int QT, int TMAX>
__device__ __forceinline__ void pair_dot(const uint32_t* src, const float* xp, int T, int tstride, float (&acc)[TMAX]) {
  if constexpr (QT == kQ4_0) {
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = src[i];
    const float dA = half_bits(w[0] & 0xFFFFu), dB = half_bits(w[4] >> 16);
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const float4* xq = reinterpret_cast<const float4*>(xp + t * tstride);
        float2 aA[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
        float2 aB[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          q4_word_dot(__byte_perm(w[i], w[i + 1], 0x5432), xq[2 * i], xq[2 * i + 1], aA);
          q4_word_dot(w[5 + i], xq[8 + 2 * i], xq[8 + 2 * i + 1], aB);
        }
        acc[t] = fmaf(dA, acc_sum(aA), acc[t]);
        acc[t] = fmaf(dB, acc_sum(aB), acc[t]);
      }
    }
  } else {
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) w[i] = src[i];
    const float dA = half_bits(w[0] & 0xFFFFu), dB = half_bits(w[8] >> 16);
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const float4* xq = reinterpret_cast<const float4*>(xp + t * tstride);
        float2 aA[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
        float2 aB[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          q8_word_dot(__byte_perm(w[i], w[i + 1], 0x5432), xq[i], aA, (i & 1) * 2);
          q8_word_dot(w[9 + i], xq[8 + i], aB, (i & 1) * 2);
        }
        acc[t] = fmaf(dA, acc_sum(aA), acc[t]);
        acc[t] = fmaf(dB, acc_sum(aB), acc[t]);
      }
    }
  }
}

// acc += dot(block pair at `src`, x) with the pair's 64 table entries held in
// registers (x[slot], as in the X table) for one token.
template <int QT>
__device__ __forceinline__ void pair_dot_regs(const uint32_t* src, const float (&x)[64], float& acc) {
  float2 aA[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
  float2 aB[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
  if constexpr (QT == kQ4_0) {
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = src[i];
    const float dA = half_bits(w[0] & 0xFFFFu), dB = half_bits(w[4] >> 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q4_word_dot(__byte_perm(w[i], w[i + 1], 0x5432), make_float4(x[8 * i], x[8 * i + 1], x[8 * i + 2], x[8 * i + 3]),
                  make_float4(x[8 * i + 4], x[8 * i + 5], x[8 * i + 6], x[8 * i + 7]), aA);
      q4_word_dot(w[5 + i], make_float4(x[32 + 8 * i], x[32 + 8 * i + 1], x[32 + 8 * i + 2], x[32 + 8 * i + 3]),
                  make_float4(x[32 + 8 * i + 4], x[32 + 8 * i + 5], x[32 + 8 * i + 6], x[32 + 8 * i + 7]), aB);
    }
    acc = fmaf(dA, acc_sum(aA), acc);
    acc = fmaf(dB, acc_sum(aB), acc);
  } else {
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) w[i] = src[i];
    const float dA = half_bits(w[0] & 0xFFFFu), dB = half_bits(w[8] >> 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      q8_word_dot(__byte_perm(w[i], w[i + 1], 0x5432),
                  make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]), aA, (i & 1) * 2);
      q8_word_dot(w[9 + i], make_float4(x[32 + 4 * i], x[32 + 4 * i + 1], x[32 + 4 * i + 2], x[32 + 4 * i + 3]), aB,
                  (i & 1) * 2);
    }
    acc = fmaf(dA, acc_sum(aA), acc);
    acc = fmaf(dB, acc_sum(aB), acc);
  }
}

// Copies the 64 table entries of block pair P (one token) into registers.
__device__ __forceinline__ void load_x_pair(const float* xt, int P, float (&x)[64]) {
  const float4* src = reinterpret_cast<const float4*>(xt + P * XPAIR);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float4 v = src[j];
    x[4 * j] = v.x;
    x[4 * j + 1] = v.y;
    x[4 * j + 2] = v.z;
    x[4 * j + 3] = v.w;
  }
}

}  // namespace gemv
}  // namespace apr
