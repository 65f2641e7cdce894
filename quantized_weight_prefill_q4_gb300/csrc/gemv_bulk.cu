// Small-T GEMV over Q4_0 / Q8_0 blocks, exact fp32 arithmetic, streamed with
// 1-D bulk copies (the HBM-bound form of the single-token GEMVs gemv_q4_0_pf /
// gemv_q8_0_pf of oxibonsai-kernels 0.1.4 src/gpu_backend/cuda_q_std_prefill.rs).
//
// Persistent CTAs, one per SM: a producer warp streams groups of 16 weight
// rows, 2048 columns at a time (one contiguous run of blocks per row), into a
// ring of shared-memory stages with cp.async.bulk; 8 consumer warps each own 2
// of the 16 rows, and each lane one block pair (64 columns, 36 or 68 bytes,
// always 4-byte aligned) of those rows.
//
// Decode without integer-to-float conversions: a 4-bit code n sitting at bit
// offset s < 23 of a 32-bit word becomes the float 2^23 + n 2^s when the
// exponent bits of 2^23 are OR-ed in, and subtracting 2^23 + 8 2^s leaves
// (n - 8) 2^s exactly (an int8 code moved to the low byte gives 2^23 + b + 128
// the same way). The 2^-s is folded into a per-CTA table of X (built once in
// shared memory, scaled by exact powers of two), so one packed fp32 FMA does
// each product. Per block the lane sums its products in fp32 and scales by d.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"

namespace apr {
namespace {

constexpr int NCW = 8;                // consumer warps
constexpr int RW = 2;                 // rows per consumer warp
constexpr int G = NCW * RW;           // rows per group
constexpr int KC = 2048;              // columns per chunk: 32 lanes x one block pair
constexpr int XPAIR = 68;             // floats per block pair in the X table (64 + pad)
constexpr int NTHREADS = 32 * (NCW + 1);

template <int QT, bool SWI>
struct BCfg {
  static constexpr int NM = SWI ? 2 : 1;
  static constexpr int BB = QT == kQ4_0 ? 18 : 34;
  static constexpr int CB = KC / 32 * BB;            // bytes of one row's chunk
  static constexpr int STAGE = NM * G * CB;
  static constexpr int NS = QT == kQ4_0 ? (SWI ? 3 : 4) : (SWI ? 2 : 3);
  static constexpr int RING = NS * STAGE;
};

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

__device__ __forceinline__ float2 q4_word_dot(uint32_t p, float4 xa, float4 xb, float2 acc) {
  const uint32_t p12 = p >> 12;
  const float2 v0 = __fadd2_rn(f2(magic(p & 0xFu), magic(p & 0xF0u)), f2(-kC0, -kC4));
  const float2 v1 = __fadd2_rn(f2(magic(p & 0xF00u), magic(p & 0xF000u)), f2(-kC8, -kC12));
  const float2 v2 = __fadd2_rn(f2(magic(p & 0xF0000u), magic(p12 & 0xF00u)), f2(-kC16, -kC8));
  const float2 v3 = __fadd2_rn(f2(magic(p12 & 0xF000u), magic(p12 & 0xF0000u)), f2(-kC12, -kC16));
  acc = __ffma2_rn(v0, f2(xa.x, xa.y), acc);
  acc = __ffma2_rn(v1, f2(xa.z, xa.w), acc);
  acc = __ffma2_rn(v2, f2(xb.x, xb.y), acc);
  acc = __ffma2_rn(v3, f2(xb.z, xb.w), acc);
  return acc;
}

// Products of one Q8_0 payload word (4 int8, elements 4i..4i+3) with x.
__device__ __forceinline__ float2 q8_word_dot(uint32_t q, float4 x, float2 acc) {
  const uint32_t u = q ^ 0x80808080u;  // byte + 128, unsigned
  const float2 v01 = __fadd2_rn(f2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                                   __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541))),
                                f2(-8388736.0f, -8388736.0f));
  const float2 v23 = __fadd2_rn(f2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                                   __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543))),
                                f2(-8388736.0f, -8388736.0f));
  acc = __ffma2_rn(v01, f2(x.x, x.y), acc);
  acc = __ffma2_rn(v23, f2(x.z, x.w), acc);
  return acc;
}

__device__ __forceinline__ float half_bits(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }

template <int QT, int TMAX, bool SWI>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemv_bulk_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ Wu, int n, int k,
                     const float* __restrict__ X, int T, float* Y, const float* R, unsigned* status) {
  using C = BCfg<QT, SWI>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the shared array so that
  // the compiler keeps the shared address space (shared loads, not generic)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int npk = k / 64;                                  // block pairs per row
  float* xt = reinterpret_cast<float*>(smem + C::RING);
  const int xt_floats = T * npk * XPAIR;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING + ((xt_floats * 4 + 15) & ~15));
  uint64_t* full = bars;
  uint64_t* empty = bars + C::NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * C::NS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = k / 32;
  const size_t row_bytes = (size_t)nb * C::BB;
  const int nchunks = (k + KC - 1) / KC;
  const int ngroups = (n + G - 1) / G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCW);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      int last[C::NS];
      for (int i = 0; i < C::NS; ++i) last[i] = -1;
      bool ok = true;
      int it = 0;
      for (int g = blockIdx.x; g < ngroups && ok; g += gridDim.x) {
        const int rows = min(G, n - g * G);
        for (int c = 0; c < nchunks; ++c, ++it) {
          const int st = it % C::NS;
          ok = mbar_wait(&empty[st], ((it / C::NS) & 1) ^ 1, abort_flag, status);
          if (!ok) break;
          const uint32_t bytes = (uint32_t)(min(KC / 32, nb - c * (KC / 32)) * C::BB);
          mbar_arrive_expect_tx(&full[st], bytes * rows * C::NM);
          for (int m = 0; m < C::NM; ++m)
            for (int r = 0; r < rows; ++r)
              bulk_load_1d(smem + st * C::STAGE + (m * G + r) * C::CB,
                           (m ? Wu : W) + (size_t)(g * G + r) * row_bytes + (size_t)c * C::CB, bytes, &full[st]);
          last[st] = it;
        }
      }
      if (!ok)
        for (int i = 0; i < C::NS; ++i)
          if (last[i] >= 0) mbar_wait(&full[i], (last[i] / C::NS) & 1, abort_flag + 1, status);
    }
    return;
  }

  // ------------------------------------------------ consumers: X table first
  // Coalesced float4 loads, eight per thread in flight before any store.
  {
    const int k4 = k / 4;
    const int total4 = T * k4;
    const float4* X4 = reinterpret_cast<const float4*>(X);
    constexpr int NT = NCW * 32, U = 8;
    for (int base = threadIdx.x; base < total4; base += U * NT) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i4 = base + u * NT;
        v[u] = i4 < total4 ? __ldg(X4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i4 = base + u * NT;
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
  named_sync(1, NCW * 32);

  int it = 0;
  bool ok = true;
  for (int g = blockIdx.x; g < ngroups && ok; g += gridDim.x) {
    float acc[C::NM][RW][TMAX];
#pragma unroll
    for (int m = 0; m < C::NM; ++m)
#pragma unroll
      for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int t = 0; t < TMAX; ++t) acc[m][r][t] = 0.f;
    const int row0 = g * G + warp * RW;

    for (int c = 0; c < nchunks; ++c, ++it) {
      const int st = it % C::NS;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (it / C::NS) & 1, abort_flag, status));
      if (!ok) break;
      const int pairs = min(KC / 32, nb - c * (KC / 32)) / 2;
      if (lane < pairs) {
        const int P = c * (KC / 64) + lane;
        const float* xp = xt + P * XPAIR;
#pragma unroll
        for (int m = 0; m < C::NM; ++m) {
#pragma unroll
          for (int r = 0; r < RW; ++r) {
            if (row0 + r >= n) continue;
            const uint32_t* src = reinterpret_cast<const uint32_t*>(smem + st * C::STAGE + (m * G + warp * RW + r) * C::CB +
                                                                    lane * 2 * C::BB);
            if constexpr (QT == kQ4_0) {
              uint32_t w[9];
#pragma unroll
              for (int i = 0; i < 9; ++i) w[i] = src[i];
              const float dA = half_bits(w[0] & 0xFFFFu), dB = half_bits(w[4] >> 16);
#pragma unroll
              for (int t = 0; t < TMAX; ++t) {
                if (t < T) {
                  const float4* xq = reinterpret_cast<const float4*>(xp + t * npk * XPAIR);
                  float2 aA = f2(0.f, 0.f), aB = f2(0.f, 0.f);
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    aA = q4_word_dot(__byte_perm(w[i], w[i + 1], 0x5432), xq[2 * i], xq[2 * i + 1], aA);
                    aB = q4_word_dot(w[5 + i], xq[8 + 2 * i], xq[8 + 2 * i + 1], aB);
                  }
                  acc[m][r][t] = fmaf(dA, aA.x + aA.y, acc[m][r][t]);
                  acc[m][r][t] = fmaf(dB, aB.x + aB.y, acc[m][r][t]);
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
                  const float4* xq = reinterpret_cast<const float4*>(xp + t * npk * XPAIR);
                  float2 aA = f2(0.f, 0.f), aB = f2(0.f, 0.f);
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    aA = q8_word_dot(__byte_perm(w[i], w[i + 1], 0x5432), xq[i], aA);
                    aB = q8_word_dot(w[9 + i], xq[8 + i], aB);
                  }
                  acc[m][r][t] = fmaf(dA, aA.x + aA.y, acc[m][r][t]);
                  acc[m][r][t] = fmaf(dB, aB.x + aB.y, acc[m][r][t]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) break;

    // ---- reduce over the lanes; lane t stores token t
#pragma unroll
    for (int m = 0; m < C::NM; ++m)
#pragma unroll
      for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          float v = acc[m][r][t];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          acc[m][r][t] = v;
        }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int row = row0 + r;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (lane == t && t < T && row < n) {
          const size_t o = (size_t)t * n + row;
          float y;
          if (SWI) {
            const float gt = acc[0][r][t];
            y = gt / (1.0f + expf(-gt)) * acc[C::NM - 1][r][t];
          } else {
            y = acc[0][r][t] + (R ? R[o] : 0.f);
          }
          Y[o] = y;
        }
      }
    }
  }
}

int g_num_sms[64] = {0};

template <int QT, int TMAX, bool SWI>
cudaError_t launch_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, const float* R,
                     unsigned* status, cudaStream_t s) {
  using C = BCfg<QT, SWI>;
  const size_t smem = gemv_bulk_smem(QT, k, T, SWI);
  auto kern = gemv_bulk_kernel<QT, TMAX, SWI>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int sms = 148;
  if (dev >= 0 && dev < 64) {
    if (!attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
      if (e != cudaSuccess) return e;
      attr_set[dev] = 1;
    }
    if (!g_num_sms[dev]) cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    sms = g_num_sms[dev] > 0 ? g_num_sms[dev] : 148;
  }
  const int ngroups = (n + G - 1) / G;
  const int grid = ngroups < sms ? ngroups : sms;
  (void)C::RING;
  kern<<<grid, NTHREADS, smem, s>>>((const uint8_t*)W, (const uint8_t*)Wu, n, k, X, T, Y, R, status);
  return cudaGetLastError();
}

template <int QT, bool SWI>
cudaError_t launch_q(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, const float* R,
                     unsigned* status, cudaStream_t s) {
  if (T <= 1) return launch_t<QT, 1, SWI>(W, Wu, n, k, X, T, Y, R, status, s);
  if (T <= 2) return launch_t<QT, 2, SWI>(W, Wu, n, k, X, T, Y, R, status, s);
  if (T <= 4) return launch_t<QT, 4, SWI>(W, Wu, n, k, X, T, Y, R, status, s);
  return launch_t<QT, 8, SWI>(W, Wu, n, k, X, T, Y, R, status, s);
}

}  // namespace

size_t gemv_bulk_smem(int qtype, int k, int T, bool swiglu) {
  size_t ring;
  if (qtype == kQ4_0)
    ring = swiglu ? BCfg<kQ4_0, true>::RING : BCfg<kQ4_0, false>::RING;
  else
    ring = swiglu ? BCfg<kQ8_0, true>::RING : BCfg<kQ8_0, false>::RING;
  const size_t xt = ((size_t)T * (k / 64) * XPAIR * 4 + 15) & ~(size_t)15;
  return 1024 + ring + xt + 2 * 8 * 4 + 16;
}

bool gemv_bulk_fits(int qtype, int k, int T, bool swiglu) {
  if (k % 256 != 0 || T < 1 || T > (swiglu ? 4 : 8)) return false;
  return gemv_bulk_smem(qtype, k, T, swiglu) <= 232448;
}

cudaError_t launch_gemv_bulk(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y,
                             const float* R, unsigned* status, cudaStream_t s) {
  const bool swi = Wu != nullptr;
  if (qtype == kQ4_0)
    return swi ? launch_q<kQ4_0, true>(W, Wu, n, k, X, T, Y, R, status, s)
               : launch_q<kQ4_0, false>(W, Wu, n, k, X, T, Y, R, status, s);
  return swi ? launch_q<kQ8_0, true>(W, Wu, n, k, X, T, Y, R, status, s)
             : launch_q<kQ8_0, false>(W, Wu, n, k, X, T, Y, R, status, s);
}

}  // namespace apr
