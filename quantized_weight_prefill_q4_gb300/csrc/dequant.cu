// Standalone dequant: out[n][k] = f32(d) * f32(q') (F16: f32(w); Q4_K and Q5_K:
// d sc q - dmin m rounded once; Q6_K: d sc (q - 32), exact; IQ4_XS:
// d (ls - 32) book[c], exact), bit exact against the oracle.
//
// The device dequant of aprender-serve 0.70.2 src/cuda/executor/gdn_prefill_ops.rs
// (qwen35_dequant_f32: one 32-element block per warp, one element per lane),
// kept for tests; the projections decode blocks in registers instead.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "iq4.cuh"
#include "q4k.cuh"

namespace apr {
namespace {

template <int QT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ W, int n, int k,
                                                      float* __restrict__ out) {
  constexpr int BB = QT == kQ4_0 ? 18 : 34;
  const size_t total = (size_t)n * (size_t)k;
  const size_t nb_row = (size_t)(k / 32);
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    if constexpr (QT == kF16) {  // each element its own half: widening is exact
      out[idx] = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(W)[idx]));
      continue;
    }
    if constexpr (QT == kQ6_K) {  // superblock of 256 in 210 bytes, read bytewise (2-byte aligned)
      const size_t row = idx / (size_t)k;
      const uint32_t col = (uint32_t)(idx - row * (size_t)k);
      const uint8_t* sb = W + (row * (size_t)(k / 256) + col / 256) * 210;
      const uint32_t e = col & 255u, h = e >> 7, c = (e >> 5) & 3u, l = e & 31u;
      const uint32_t lo = (sb[64 * h + 32 * (c & 1u) + l] >> (4 * (c >> 1))) & 15u;
      const uint32_t hi = (sb[128 + 32 * h + l] >> (2 * c)) & 3u;
      const float d = __half2float(__ushort_as_half((uint16_t)(sb[208] | (sb[209] << 8))));
      const int sc = (int)(int8_t)sb[192 + e / 16];
      // d sc is exact (11 + 8 bits) and so is its product with q - 32
      out[idx] = d * (float)sc * (float)((int)(lo | (hi << 4)) - 32);
      continue;
    }
    if constexpr (QT == kIQ4_XS) {  // superblock of 256 in 136 bytes, read bytewise
      const size_t row = idx / (size_t)k;
      const uint32_t col = (uint32_t)(idx - row * (size_t)k);
      const uint8_t* sb = W + (row * (size_t)(k / 256) + col / 256) * 136;
      const uint32_t e = col & 255u, j = e >> 5, l = e & 31u;
      const uint32_t c = (sb[8 + 16 * j + (l & 15u)] >> (4 * (l >> 4))) & 15u;
      // ls_j: nibble j % 2 of byte 4 + j / 2, and bits 2 (j % 4) of byte 2 + j / 4
      const int ls = (int)(((sb[4 + j / 2] >> (4 * (j & 1u))) & 15u) | (((sb[2 + j / 4] >> (2 * (j & 3u))) & 3u) << 4));
      const int v = (int)(iq4_bytes4(c) & 0xFFu) - 128;  // book[c]
      const float d = __half2float(__ushort_as_half((uint16_t)(sb[0] | (sb[1] << 8))));
      // d (ls - 32) is exact (11 + 5 bits) and so is its product with book[c]
      out[idx] = d * (float)(ls - 32) * (float)v;
      continue;
    }
    if constexpr (QT == kQ4_K || QT == kQ5_K) {  // superblock of 256 in 144 or 176 bytes
      constexpr uint32_t SBB = QT == kQ4_K ? 144 : 176, QOFF = QT == kQ4_K ? 16 : 48;
      const size_t row = idx / (size_t)k;
      const uint32_t col = (uint32_t)(idx - row * (size_t)k);
      const uint8_t* sb = W + (row * (size_t)(k / 256) + col / 256) * SBB;
      const uint32_t e = col & 255u, g = e >> 6, hi = (e >> 5) & 1u, l = e & 31u, j = 2 * g + hi;
      uint32_t sc, m;
      q4k_scale_min(sb + 4, j, sc, m);
      const float d = __half2float(__ushort_as_half((uint16_t)(sb[0] | (sb[1] << 8))));
      const float dmin = __half2float(__ushort_as_half((uint16_t)(sb[2] | (sb[3] << 8))));
      uint32_t q = (sb[QOFF + 32 * g + l] >> (4 * hi)) & 15u;
      if (QT == kQ5_K) q += ((sb[16 + l] >> j) & 1u) << 4;  // the fifth bit: bit 2 g + hi of byte l
      // d sc and dmin m are exact in fp32; one rounding of d sc q - dmin m
      out[idx] = fmaf(d * (float)sc, (float)q, -(dmin * (float)m));
      continue;
    }
    const size_t row = idx / (size_t)k;
    const uint32_t col = (uint32_t)(idx - row * (size_t)k);
    const uint8_t* blk = W + (row * nb_row + col / 32) * BB;
    const uint32_t e = col & 31u;
    const uint16_t dbits = (uint16_t)blk[0] | ((uint16_t)blk[1] << 8);
    const float d = __half2float(__ushort_as_half(dbits));  // exact widening
    int q;
    if (QT == kQ4_0) {
      const uint32_t byte = blk[2 + (e & 15u)];
      q = (int)((e < 16 ? byte : (byte >> 4)) & 0xFu) - 8;
    } else {
      q = (int)(int8_t)blk[2 + e];
    }
    out[idx] = d * (float)q;  // exact: <= 11 x 8 significant bits
  }
}

}  // namespace

cudaError_t launch_dequant(int qtype, const void* W, int n, int k, float* out, cudaStream_t s) {
  const size_t total = (size_t)n * (size_t)k;
  size_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (qtype == kIQ4_XS)
    dequant_kernel<kIQ4_XS><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  else if (qtype == kQ6_K)
    dequant_kernel<kQ6_K><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  else if (qtype == kQ5_K)
    dequant_kernel<kQ5_K><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  else if (qtype == kQ4_K)
    dequant_kernel<kQ4_K><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  else if (qtype == kF16)
    dequant_kernel<kF16><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  else if (qtype == kQ4_0)
    dequant_kernel<kQ4_0><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  else
    dequant_kernel<kQ8_0><<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, n, k, out);
  return cudaGetLastError();
}

}  // namespace apr
