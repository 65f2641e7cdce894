// Small-T GEMV over Q4_0 / Q8_0 blocks, F16, Q4_K or Q5_K weights, exact fp32 arithmetic.
//
// Y[t][i] = sum_j X[t][j] * d_{i,j/32} * q'_{i,j} (+ R[t][i]) for T <= 16 token
// rows, or silu(g) * u for a gate/up pair. The single-token GEMVs of
// oxibonsai-kernels 0.1.4 src/gpu_backend/cuda_q_std_prefill.rs
// (gemv_q4_0_pf / gemv_q8_0_pf, launched for the last-token lm_head), widened
// to T accumulators so that one weight read serves up to 16 tokens.
//
// Layout of the work: one warp owns RW consecutive W rows at a time. The warp
// walks the row in segments of 32 blocks; each segment is copied from global
// memory with coalesced 16-byte loads (when every row starts on a 16-byte
// boundary, i.e. k % 256 == 0; 2-byte loads otherwise) into a per-warp shared
// buffer, then lane l decodes block l of the segment and multiplies it with
// the matching 32 columns of each of the T activation rows (read through the
// read-only cache; every warp of an SM walks the same columns). Per block the
// lane keeps sum_j x_j * q'_j and scales it by d once; at the end of the row
// the 32 lanes' partial sums are reduced with shuffles.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "host_common.h"
#include "iq4.cuh"
#include "q4k.cuh"

namespace apr {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// Weight loads of the streaming GEMVs: read once, so they bypass L1 and leave
// it to X, which every row reads again (measured at 4096 x 4096, T = 4:
// 30.3 -> 22.2 us for Q4_K, 30.2 -> 22.5 us for F16)
__device__ __forceinline__ uint4 ldw_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldw_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldw_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldw_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldw_u8(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void grid_dependency_wait_inline() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <int QT, int TMAX, int RW, bool VEC, bool SWI>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const uint8_t* __restrict__ W,
                                                           const uint8_t* __restrict__ Wu, int n, int k,
                                                           const float* __restrict__ X, int T,
                                                           float* Y, int ldy,
                                                           const float* R) {
  constexpr int BB = QT == kQ4_0 ? 18 : (QT == kQ8_0 ? 34 : 64);
  constexpr int SEG = 32 * BB;
  constexpr int NM = SWI ? 2 : 1;
  __shared__ __align__(16) uint8_t stage[kWarps][NM * RW][SEG];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb = k >> 5;
  const size_t row_bytes = (size_t)nb * BB;
  const int ngroups = (n + RW - 1) / RW;

  for (int grp = blockIdx.x * kWarps + warp; grp < ngroups; grp += gridDim.x * kWarps) {
    const int r0 = grp * RW;
    float acc[NM][RW][TMAX];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int t = 0; t < TMAX; ++t) acc[m][r][t] = 0.f;

    for (int s = 0; s < nb; s += 32) {
      const int nblk = min(32, nb - s);
      const int seg_bytes = nblk * BB;
      // ---- stage the segment of each row (and of the up rows)
#pragma unroll
      for (int m = 0; m < NM; ++m) {
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          const int row = r0 + r;
          if (row >= n) continue;
          const uint8_t* src = (m ? Wu : W) + (size_t)row * row_bytes + (size_t)s * BB;
          uint8_t* dst = stage[warp][m * RW + r];
          if (VEC) {
            for (int c = lane; c < seg_bytes / 16; c += 32)
              *reinterpret_cast<uint4*>(dst + c * 16) = ldg_nc_v4(src + c * 16);
          } else {
            for (int c = lane; c < seg_bytes / 2; c += 32)
              *reinterpret_cast<uint16_t*>(dst + c * 2) = __ldg(reinterpret_cast<const unsigned short*>(src) + c);
          }
        }
      }
      __syncwarp();
      if (lane < nblk) {
        const int col0 = (s + lane) * 32;
        float part[NM][RW][TMAX];
        float dsc[NM][RW];
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
          for (int r = 0; r < RW; ++r) {
            const uint8_t* blk = stage[warp][m * RW + r] + lane * BB;
            if constexpr (QT == kF16) {
              dsc[m][r] = 1.f;  // the elements are the weights
            } else {
              const uint16_t db = *reinterpret_cast<const uint16_t*>(blk);
              dsc[m][r] = __half2float(__ushort_as_half(db));
            }
#pragma unroll
            for (int t = 0; t < TMAX; ++t) part[m][r][t] = 0.f;
          }
        // Q4_0: half h covers payload bytes 8h..8h+7, i.e. elements 8h..8h+7
        // (low nibbles) and 16+8h..16+8h+7 (high nibbles).
        // Q8_0 and F16: quarter h covers elements 8h..8h+7.
        constexpr int NPART = QT == kQ4_0 ? 2 : 4;
        constexpr int NE = QT == kQ4_0 ? 16 : 8;  // elements per part
#pragma unroll
        for (int h = 0; h < NPART; ++h) {
          float wq[NM][RW][NE];
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int r = 0; r < RW; ++r) {
              const uint8_t* pay = stage[warp][m * RW + r] + lane * BB + (QT == kF16 ? 0 : 2);
              if constexpr (QT == kF16) {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(pay + 16 * h + 2 * e));
                  wq[m][r][e] = f.x;
                  wq[m][r][e + 1] = f.y;
                }
              } else if constexpr (QT == kQ4_0) {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const uint32_t two = *reinterpret_cast<const uint16_t*>(pay + 8 * h + e);
                  wq[m][r][e] = (float)((int)(two & 0xFu) - 8);
                  wq[m][r][e + 1] = (float)((int)((two >> 8) & 0xFu) - 8);
                  wq[m][r][8 + e] = (float)((int)((two >> 4) & 0xFu) - 8);
                  wq[m][r][8 + e + 1] = (float)((int)((two >> 12) & 0xFu) - 8);
                }
              } else {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const uint32_t two = *reinterpret_cast<const uint16_t*>(pay + 8 * h + e);
                  wq[m][r][e] = (float)(int8_t)(two & 0xFFu);
                  wq[m][r][e + 1] = (float)(int8_t)(two >> 8);
                }
              }
            }
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
              const float* xr = X + (size_t)t * k + col0 + 8 * h;
              const float4 a0 = __ldg(reinterpret_cast<const float4*>(xr));
              const float4 a1 = __ldg(reinterpret_cast<const float4*>(xr + 4));
              float xv[NE];
              xv[0] = a0.x; xv[1] = a0.y; xv[2] = a0.z; xv[3] = a0.w;
              xv[4] = a1.x; xv[5] = a1.y; xv[6] = a1.z; xv[7] = a1.w;
              if constexpr (NE == 16) {
                const float4 b0 = __ldg(reinterpret_cast<const float4*>(xr + 16));
                const float4 b1 = __ldg(reinterpret_cast<const float4*>(xr + 20));
                xv[8] = b0.x; xv[9] = b0.y; xv[10] = b0.z; xv[11] = b0.w;
                xv[12] = b1.x; xv[13] = b1.y; xv[14] = b1.z; xv[15] = b1.w;
              }
#pragma unroll
              for (int m = 0; m < NM; ++m)
#pragma unroll
                for (int r = 0; r < RW; ++r)
#pragma unroll
                  for (int e = 0; e < NE; ++e)
                    part[m][r][t] = fmaf(wq[m][r][e], xv[e], part[m][r][t]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
          for (int r = 0; r < RW; ++r)
#pragma unroll
            for (int t = 0; t < TMAX; ++t) acc[m][r][t] = fmaf(dsc[m][r], part[m][r][t], acc[m][r][t]);
      }
      __syncwarp();
    }

    // ---- reduce over the lanes; lane t stores token t
#pragma unroll
    for (int m = 0; m < NM; ++m)
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
      const int row = r0 + r;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (lane == t && t < T && row < n) {
          const size_t o = (size_t)t * ldy + row;
          float v;
          if (SWI)
            v = silu_mul(acc[0][r][t], acc[NM - 1][r][t]);
          else
            v = acc[0][r][t] + (R ? R[o] : 0.f);
          Y[o] = v;
        }
      }
    }
  }
}

template <int QT, int TMAX, bool SWI>
cudaError_t launch_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                     const float* R, cudaStream_t s) {
  constexpr int RW = (TMAX >= 8 || SWI) ? 1 : 2;
  const int ngroups = (n + RW - 1) / RW;
  int blocks = (ngroups + kWarps - 1) / kWarps;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const bool vec = (k % 256) == 0;
  if (vec)
    gemv_kernel<QT, TMAX, RW, true, SWI><<<blocks, kWarps * 32, 0, s>>>(
        (const uint8_t*)W, (const uint8_t*)Wu, n, k, X, T, Y, ldy, R);
  else
    gemv_kernel<QT, TMAX, RW, false, SWI><<<blocks, kWarps * 32, 0, s>>>(
        (const uint8_t*)W, (const uint8_t*)Wu, n, k, X, T, Y, ldy, R);
  return cudaGetLastError();
}

template <int QT, bool SWI>
cudaError_t launch_q(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                     const float* R, cudaStream_t s) {
  if (T <= 1) return launch_t<QT, 1, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 2) return launch_t<QT, 2, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 4) return launch_t<QT, 4, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 8) return launch_t<QT, 8, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return launch_t<QT, 16, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

// F16 weights, k % 256 == 0: a warp per weight row, each lane 16-byte chunks
// (8 halves) c = lane + 32 i of the row, eight chunks' loads in flight; X
// through the read-only cache (the same columns for every row, so it stays in
// L1); exact fp32 products (a half widens exactly). The weights of the
// warp's first chunks are requested before the dependency wait (they are
// never the output of the preceding kernel); X, R and Y after it.
// Streaming GEMVs (K-quants): superblocks whose loads are issued together before any is
// decoded, by the number of tokens (measured on 4096 and 12288 rows x 4096:
// 8 at T <= 2, 4 above; 2 took 12-40 % longer at T = 2 and 8)
__host__ __device__ constexpr int kq_unroll(int tmax) { return tmax <= 2 ? 8 : 4; }
// rows a warp takes together at T >= 2: they share each load of X (4096 x
// 4096, Q4_K: 21.9 -> 16.7 us at T = 4, 38.4 -> 25.5 us at T = 8; F16: 22.2 ->
// 17.9 us at T = 4)
__host__ __device__ constexpr int kq_rows(int tmax) { return tmax >= 2 ? 2 : 1; }

// Reduces a warp's lane partials of RB rows (NM weights each) over the warp
// and writes rows row0 .. row0 + RB - 1 below n: token t's value by lane t.
template <int TMAX, int NM, int RB, bool SWI>
__device__ __forceinline__ void kq_rows_out(float (&acc)[RB * NM][TMAX], int row0, int n, int T, int lane, float* Y,
                                            int ldy, const float* R) {
#pragma unroll
  for (int m = 0; m < RB * NM; ++m)
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      float v = acc[m][t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[m][t] = v;
    }
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    if (row0 + r >= n) break;
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (lane == t && t < T) {
        const size_t o = (size_t)t * ldy + row0 + r;
        Y[o] = SWI ? silu_mul(acc[r * NM][t], acc[r * NM + NM - 1][t]) : acc[r * NM][t] + (R ? R[o] : 0.f);
      }
    }
  }
}

constexpr int F16G = 8;  // chunks a lane loads at once

template <int TMAX, bool SWI>
__global__ void __launch_bounds__(kWarps * 32) gemv_f16_kernel(const uint16_t* __restrict__ W,
                                                               const uint16_t* __restrict__ Wu, int n, int k,
                                                               const float* __restrict__ X, int T, float* Y, int ldy,
                                                               const float* R) {
  constexpr int NM = SWI ? 2 : 1;
  constexpr int RB = kq_rows(TMAX), NS = RB * NM;  // rows together; weight rows read (row r, weight m: r NM + m)
  constexpr int G = F16G / RB;                     // chunks a lane loads at once from each weight row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = k / 8;              // 16-byte chunks a row
  const int ngroup = nchunk / (32 * G);  // groups of G chunks a lane
  const int rest = nchunk / 32 - ngroup * G;
  bool waited = false;
  for (int row0 = (blockIdx.x * kWarps + warp) * RB; row0 < n; row0 += gridDim.x * kWarps * RB) {
    float acc[NS][TMAX];
#pragma unroll
    for (int m = 0; m < NS; ++m)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[m][t] = 0.f;
    const uint4* wr[NS];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const size_t rr = (size_t)min(row0 + r, n - 1);  // a row past n repeats the last one, unstored
      wr[r * NM] = reinterpret_cast<const uint4*>(W + rr * k);
      if (SWI) wr[r * NM + 1] = reinterpret_cast<const uint4*>(Wu + rr * k);
    }
    auto chunk = [&](const uint4 (&w)[NS], int c) {
      // chunk c: columns 8c .. 8c + 7
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const float4* xr = reinterpret_cast<const float4*>(X + (size_t)t * k + 8 * c);
          const float4 a = __ldg(xr), b = __ldg(xr + 1);
#pragma unroll
          for (int m = 0; m < NS; ++m) {
            const float2 w0 = __half22float2(*reinterpret_cast<const __half2*>(&w[m].x));
            const float2 w1 = __half22float2(*reinterpret_cast<const __half2*>(&w[m].y));
            const float2 w2 = __half22float2(*reinterpret_cast<const __half2*>(&w[m].z));
            const float2 w3 = __half22float2(*reinterpret_cast<const __half2*>(&w[m].w));
            float v = acc[m][t];
            v = fmaf(w0.x, a.x, v);
            v = fmaf(w0.y, a.y, v);
            v = fmaf(w1.x, a.z, v);
            v = fmaf(w1.y, a.w, v);
            v = fmaf(w2.x, b.x, v);
            v = fmaf(w2.y, b.y, v);
            v = fmaf(w3.x, b.z, v);
            v = fmaf(w3.y, b.w, v);
            acc[m][t] = v;
          }
        }
      }
    };
    for (int gi = 0; gi < ngroup; ++gi) {
      uint4 w[G][NS];
#pragma unroll
      for (int i = 0; i < G; ++i)
#pragma unroll
        for (int m = 0; m < NS; ++m) w[i][m] = ldw_v4(wr[m] + lane + 32 * (gi * G + i));
      if (!waited) {
        grid_dependency_wait_inline();
        waited = true;
      }
#pragma unroll
      for (int i = 0; i < G; ++i) chunk(w[i], lane + 32 * (gi * G + i));
    }
    for (int i = 0; i < rest; ++i) {
      uint4 w[NS];
#pragma unroll
      for (int m = 0; m < NS; ++m) w[m] = ldw_v4(wr[m] + lane + 32 * (ngroup * G + i));
      if (!waited) {
        grid_dependency_wait_inline();
        waited = true;
      }
      chunk(w, lane + 32 * (ngroup * G + i));
    }
    kq_rows_out<TMAX, NM, RB, SWI>(acc, row0, n, T, lane, Y, ldy, R);
  }
  if (!waited) grid_dependency_wait_inline();  // a CTA without rows
}

template <int TMAX, bool SWI>
cudaError_t launch_f16_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                         const float* R, cudaStream_t s) {
  const int rows = kWarps * kq_rows(TMAX);
  long blocks = (n + rows - 1) / rows;
  const long cap = (long)num_sms() * 2;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_f16_kernel<TMAX, SWI>, static_cast<const uint16_t*>(W),
                            static_cast<const uint16_t*>(Wu), n, k, X, T, Y, ldy, R);
}

template <bool SWI>
cudaError_t launch_f16(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                       const float* R, cudaStream_t s) {
  if (T <= 1) return launch_f16_t<1, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 2) return launch_f16_t<2, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 4) return launch_f16_t<4, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 8) return launch_f16_t<8, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return launch_f16_t<16, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

// Q4_K and Q5_K weights: a warp per weight row (two rows at T >= 2), one
// 256-element superblock (144 or 176 bytes) a step; lane l takes elements 8 l .. 8 l + 7 of it: group
// g = l / 8 (64 elements), low nibbles of code bytes 32 g + 8 (l mod 4) .. for
// l mod 8 < 4 (sub-block 2 g), high nibbles of the same bytes otherwise
// (sub-block 2 g + 1); Q5_K adds bit 2 g (or 2 g + 1) of the fifth-bit bytes
// 8 (l mod 4) .. as 16. Each weight is d sc q - dmin m rounded once to fp32
// (one fma of two exact products), then exact fp32 products with X. The loads
// of several superblocks are issued before any is used.
template <int QT, int TMAX, bool SWI>
__global__ void __launch_bounds__(kWarps * 32) gemv_q4k_kernel(const uint8_t* __restrict__ W,
                                                               const uint8_t* __restrict__ Wu, int n, int k,
                                                               const float* __restrict__ X, int T, float* Y, int ldy,
                                                               const float* R) {
  constexpr int NM = SWI ? 2 : 1;
  constexpr int RB = kq_rows(TMAX), NS = RB * NM;  // rows together; weight rows read (row r, weight m: r NM + m)
  constexpr int U = kq_unroll(TMAX) / RB;
  constexpr bool FIVE = QT == kQ5_K;
  constexpr uint32_t SBB = FIVE ? 176 : 144;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = k / 256;
  const size_t row_bytes = (size_t)nsb * SBB;
  const uint32_t g = (uint32_t)lane >> 3, part = (uint32_t)lane & 7u, hi = part >> 2, j = 2 * g + hi;
  const uint32_t qoff = (FIVE ? 48 : 16) + 32 * g + 8 * (part & 3u), hoff = 16 + 8 * (part & 3u);
  bool waited = false;
  for (int row0 = (blockIdx.x * kWarps + warp) * RB; row0 < n; row0 += gridDim.x * kWarps * RB) {
    float acc[NS][TMAX];
#pragma unroll
    for (int m = 0; m < NS; ++m)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[m][t] = 0.f;
    const uint8_t* base[NS];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const size_t rr = (size_t)min(row0 + r, n - 1);  // a row past n repeats the last one, unstored
      base[r * NM] = W + rr * row_bytes;
      if (SWI) base[r * NM + 1] = Wu + rr * row_bytes;
    }
    for (int sb0 = 0; sb0 < nsb; sb0 += U) {
      uint4 h[U][NS];
      uint2 c[U][NS], f[U][NS];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int m = 0; m < NS; ++m)
          if (sb0 + u < nsb) {
            const uint8_t* sb = base[m] + (size_t)(sb0 + u) * SBB;
            h[u][m] = ldw_v4(sb);
            c[u][m] = ldw_v2(sb + qoff);
            if (FIVE) f[u][m] = ldw_v2(sb + hoff);
          }
      if (!waited) {
        grid_dependency_wait_inline();
        waited = true;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (sb0 + u >= nsb) break;
        float w[NS][8];
#pragma unroll
        for (int m = 0; m < NS; ++m) {
          const uint32_t sw[3] = {h[u][m].y, h[u][m].z, h[u][m].w};
          uint32_t sc, mn;
          q4k_scale_min_w(sw, j, sc, mn);
          const float d = __half2float(__ushort_as_half((unsigned short)(h[u][m].x & 0xFFFFu)));
          const float dmin = __half2float(__ushort_as_half((unsigned short)(h[u][m].x >> 16)));
          const float a = d * (float)sc, b = -(dmin * (float)mn);
          const uint32_t cw[2] = {c[u][m].x, c[u][m].y};
          uint32_t fw[2] = {0u, 0u};
          if (FIVE) {
            fw[0] = f[u][m].x;
            fw[1] = f[u][m].y;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            uint32_t qv = (cw[e >> 2] >> (8 * (e & 3) + 4 * hi)) & 15u;
            if (FIVE) qv += ((fw[e >> 2] >> (8 * (e & 3) + j)) & 1u) << 4;
            w[m][e] = fmaf(a, (float)qv, b);
          }
        }
        const int col = (sb0 + u) * 256 + 8 * lane;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T) {
            const float4* xr = reinterpret_cast<const float4*>(X + (size_t)t * k + col);
            const float4 xa = __ldg(xr), xb = __ldg(xr + 1);
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int m = 0; m < NS; ++m) {
              float v = acc[m][t];
#pragma unroll
              for (int e = 0; e < 8; ++e) v = fmaf(w[m][e], xv[e], v);
              acc[m][t] = v;
            }
          }
        }
      }
    }
    kq_rows_out<TMAX, NM, RB, SWI>(acc, row0, n, T, lane, Y, ldy, R);
  }
  if (!waited) grid_dependency_wait_inline();  // a CTA without rows
}

template <int QT, int TMAX, bool SWI>
cudaError_t launch_q4k_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                         const float* R, cudaStream_t s) {
  const int rows = kWarps * kq_rows(TMAX);
  long blocks = (n + rows - 1) / rows;
  const long cap = (long)num_sms() * 2;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_q4k_kernel<QT, TMAX, SWI>, static_cast<const uint8_t*>(W),
                            static_cast<const uint8_t*>(Wu), n, k, X, T, Y, ldy, R);
}

template <int QT, bool SWI>
cudaError_t launch_q4k(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                       const float* R, cudaStream_t s) {
  if (T <= 1) return launch_q4k_t<QT, 1, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 2) return launch_q4k_t<QT, 2, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 4) return launch_q4k_t<QT, 4, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 8) return launch_q4k_t<QT, 8, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return launch_q4k_t<QT, 16, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

// Q6_K: a warp per row (two rows at T >= 2), lane L decoding elements 8 L ..
// 8 L + 7 of each superblock: low nibbles from bytes 64 h + 32 (c % 2) +
// 8 (L % 4) .. (h = L / 16, c = L / 4 % 4; nibble c / 2), high bit pairs from
// bytes 128 + 32 h + 8 (L % 4) .. (bits 2 c), the int8 scale at byte
// 192 + L / 2 and d at 208.
// Rows start on 16-byte boundaries, so superblock j starts 2 (j % 2) bytes
// past a 4-byte one: an 8-byte field is read as three aligned words and
// shifted. w = d sc (q - 32) is exact in fp32; products accumulate in fp32.
template <int TMAX, bool SWI>
__global__ void __launch_bounds__(kWarps * 32) gemv_q6k_kernel(const uint8_t* __restrict__ W,
                                                               const uint8_t* __restrict__ Wu, int n, int k,
                                                               const float* __restrict__ X, int T, float* Y, int ldy,
                                                               const float* R) {
  constexpr int NM = SWI ? 2 : 1;
  constexpr int RB = kq_rows(TMAX), NS = RB * NM;  // rows together; weight rows read (row r, weight m: r NM + m)
  constexpr int U = kq_unroll(TMAX) / RB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = k / 256;
  const size_t row_bytes = (size_t)nsb * 210;
  const uint32_t h = (uint32_t)lane >> 4, c = ((uint32_t)lane >> 2) & 3u, l0 = 8u * ((uint32_t)lane & 3u);
  const uint32_t loff = 64 * h + 32 * (c & 1u) + l0, hoff = 128 + 32 * h + l0, soff = 192 + ((uint32_t)lane >> 1);
  const uint32_t lsh = 4 * (c >> 1), hsh = 2 * c;
  bool waited = false;
  for (int row0 = (blockIdx.x * kWarps + warp) * RB; row0 < n; row0 += gridDim.x * kWarps * RB) {
    float acc[NS][TMAX];
#pragma unroll
    for (int m = 0; m < NS; ++m)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[m][t] = 0.f;
    const uint8_t* base[NS];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const size_t rr = (size_t)min(row0 + r, n - 1);  // a row past n repeats the last one, unstored
      base[r * NM] = W + rr * row_bytes;
      if (SWI) base[r * NM + 1] = Wu + rr * row_bytes;
    }
    for (int sb0 = 0; sb0 < nsb; sb0 += U) {
      uint32_t lw[U][NS][3], hw[U][NS][3], scb[U][NS];
      unsigned short db[U][NS];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int m = 0; m < NS; ++m)
          if (sb0 + u < nsb) {
            const uint8_t* sb = base[m] + (size_t)(sb0 + u) * 210;
            const uint32_t sh = 2u * ((uint32_t)(sb0 + u) & 1u);
            const uint32_t* pl = reinterpret_cast<const uint32_t*>(sb + loff - sh);
            const uint32_t* ph = reinterpret_cast<const uint32_t*>(sb + hoff - sh);
#pragma unroll
            for (int v = 0; v < 3; ++v) {
              lw[u][m][v] = ldw_u32(pl + v);
              hw[u][m][v] = ldw_u32(ph + v);
            }
            scb[u][m] = ldw_u8(sb + soff);
            db[u][m] = (unsigned short)ldw_u16(sb + 208);
          }
      if (!waited) {
        grid_dependency_wait_inline();
        waited = true;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (sb0 + u >= nsb) break;
        const uint32_t s8 = 16u * ((uint32_t)(sb0 + u) & 1u);
        float w[NS][8];
#pragma unroll
        for (int m = 0; m < NS; ++m) {
          const uint32_t lo[2] = {__funnelshift_r(lw[u][m][0], lw[u][m][1], s8),
                                  __funnelshift_r(lw[u][m][1], lw[u][m][2], s8)};
          const uint32_t hi[2] = {__funnelshift_r(hw[u][m][0], hw[u][m][1], s8),
                                  __funnelshift_r(hw[u][m][1], hw[u][m][2], s8)};
          const float a = __half2float(__ushort_as_half(db[u][m])) * (float)(int)(int8_t)scb[u][m];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t qv = ((lo[e >> 2] >> (8 * (e & 3) + lsh)) & 15u) |
                                (((hi[e >> 2] >> (8 * (e & 3) + hsh)) & 3u) << 4);
            w[m][e] = a * (float)((int)qv - 32);
          }
        }
        const int col = (sb0 + u) * 256 + 8 * lane;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T) {
            const float4* xr = reinterpret_cast<const float4*>(X + (size_t)t * k + col);
            const float4 xa = __ldg(xr), xb = __ldg(xr + 1);
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int m = 0; m < NS; ++m) {
              float v = acc[m][t];
#pragma unroll
              for (int e = 0; e < 8; ++e) v = fmaf(w[m][e], xv[e], v);
              acc[m][t] = v;
            }
          }
        }
      }
    }
    kq_rows_out<TMAX, NM, RB, SWI>(acc, row0, n, T, lane, Y, ldy, R);
  }
  if (!waited) grid_dependency_wait_inline();  // a CTA without rows
}

template <int TMAX, bool SWI>
cudaError_t launch_q6k_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                         const float* R, cudaStream_t s) {
  const int rows = kWarps * kq_rows(TMAX);
  long blocks = (n + rows - 1) / rows;
  const long cap = (long)num_sms() * 2;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_q6k_kernel<TMAX, SWI>, static_cast<const uint8_t*>(W),
                            static_cast<const uint8_t*>(Wu), n, k, X, T, Y, ldy, R);
}

template <bool SWI>
cudaError_t launch_q6k(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                       const float* R, cudaStream_t s) {
  if (T <= 1) return launch_q6k_t<1, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 2) return launch_q6k_t<2, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 4) return launch_q6k_t<4, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 8) return launch_q6k_t<8, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return launch_q6k_t<16, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

// IQ4_XS: a warp per row (two rows at T >= 2), lane L decoding elements
// 8 L .. 8 L + 7 of each superblock: sub-block j = L / 4, its code bytes
// 8 + 16 j + 8 (L % 2) .. (low nibbles for L % 4 < 2, high nibbles
// otherwise), with the header's d and scale bits (bytes 0-7, one 8-byte
// load). Rows start on 16-byte boundaries and superblocks on 8-byte ones.
// w = d (ls - 32) book[c] is exact in fp32; products accumulate in fp32.
template <int TMAX, bool SWI>
__global__ void __launch_bounds__(kWarps * 32) gemv_iq4_kernel(const uint8_t* __restrict__ W,
                                                               const uint8_t* __restrict__ Wu, int n, int k,
                                                               const float* __restrict__ X, int T, float* Y, int ldy,
                                                               const float* R) {
  constexpr int NM = SWI ? 2 : 1;
  constexpr int RB = kq_rows(TMAX), NS = RB * NM;  // rows together; weight rows read (row r, weight m: r NM + m)
  constexpr int U = kq_unroll(TMAX) / RB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = k / 256;
  const size_t row_bytes = (size_t)nsb * 136;
  const uint32_t j = (uint32_t)lane >> 2, nsh = 4 * (((uint32_t)lane >> 1) & 1u);
  const uint32_t coff = 8 + 16 * j + 8 * ((uint32_t)lane & 1u);
  bool waited = false;
  for (int row0 = (blockIdx.x * kWarps + warp) * RB; row0 < n; row0 += gridDim.x * kWarps * RB) {
    float acc[NS][TMAX];
#pragma unroll
    for (int m = 0; m < NS; ++m)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[m][t] = 0.f;
    const uint8_t* base[NS];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const size_t rr = (size_t)min(row0 + r, n - 1);  // a row past n repeats the last one, unstored
      base[r * NM] = W + rr * row_bytes;
      if (SWI) base[r * NM + 1] = Wu + rr * row_bytes;
    }
    for (int sb0 = 0; sb0 < nsb; sb0 += U) {
      uint2 hd[U][NS], cw[U][NS];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int m = 0; m < NS; ++m)
          if (sb0 + u < nsb) {
            const uint8_t* sb = base[m] + (size_t)(sb0 + u) * 136;
            hd[u][m] = ldw_v2(sb);
            cw[u][m] = ldw_v2(sb + coff);
          }
      if (!waited) {
        grid_dependency_wait_inline();
        waited = true;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (sb0 + u >= nsb) break;
        float w[NS][8];
#pragma unroll
        for (int m = 0; m < NS; ++m) {
          const float a = __half2float(__ushort_as_half((unsigned short)(hd[u][m].x & 0xFFFFu))) *
                          (float)iq4_scale(hd[u][m].x, hd[u][m].y, j);
          // the lane's eight codes, one a byte, to book + 128
          const uint32_t b0 = iq4_bytes4((cw[u][m].x >> nsh) & 0x0F0F0F0Fu);
          const uint32_t b1 = iq4_bytes4((cw[u][m].y >> nsh) & 0x0F0F0F0Fu);
#pragma unroll
          for (int e = 0; e < 8; ++e)  // book[c] exactly: the float 2^23 + byte less 2^23 + 128
            w[m][e] = a * (__uint_as_float(__byte_perm(e < 4 ? b0 : b1, 0x4B000000u, 0x7440u + (e & 3))) -
                           8388736.0f);
        }
        const int col = (sb0 + u) * 256 + 8 * lane;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T) {
            const float4* xr = reinterpret_cast<const float4*>(X + (size_t)t * k + col);
            const float4 xa = __ldg(xr), xb = __ldg(xr + 1);
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int m = 0; m < NS; ++m) {
              float v = acc[m][t];
#pragma unroll
              for (int e = 0; e < 8; ++e) v = fmaf(w[m][e], xv[e], v);
              acc[m][t] = v;
            }
          }
        }
      }
    }
    kq_rows_out<TMAX, NM, RB, SWI>(acc, row0, n, T, lane, Y, ldy, R);
  }
  if (!waited) grid_dependency_wait_inline();  // a CTA without rows
}

template <int TMAX, bool SWI>
cudaError_t launch_iq4_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                         const float* R, cudaStream_t s) {
  const int rows = kWarps * kq_rows(TMAX);
  long blocks = (n + rows - 1) / rows;
  const long cap = (long)num_sms() * 2;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_iq4_kernel<TMAX, SWI>, static_cast<const uint8_t*>(W),
                            static_cast<const uint8_t*>(Wu), n, k, X, T, Y, ldy, R);
}

template <bool SWI>
cudaError_t launch_iq4(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                       const float* R, cudaStream_t s) {
  if (T <= 1) return launch_iq4_t<1, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 2) return launch_iq4_t<2, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 4) return launch_iq4_t<4, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (T <= 8) return launch_iq4_t<8, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return launch_iq4_t<16, SWI>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

}  // namespace

cudaError_t launch_gemv(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T,
                        float* Y, int ldy, const float* R, unsigned* status, cudaStream_t s) {
  const bool swi = Wu != nullptr;
  // one and two tokens: the integer-dot kernel; the whole-row kernel (one
  // token) needs no stride
  if (gemv_i8_fits(qtype, n, k, T, swi)) return launch_gemv_i8(qtype, W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (gemv_rows_fits(qtype, n, k, T, swi)) return launch_gemv_rows(qtype, W, Wu, n, k, X, T, Y, R, status, s);
  if (gemv_bulk_fits(qtype, k, T, swi)) return launch_gemv_bulk(qtype, W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (qtype == kQ4_K)
    return swi ? launch_q4k<kQ4_K, true>(W, Wu, n, k, X, T, Y, ldy, R, s)
               : launch_q4k<kQ4_K, false>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (qtype == kQ5_K)
    return swi ? launch_q4k<kQ5_K, true>(W, Wu, n, k, X, T, Y, ldy, R, s)
               : launch_q4k<kQ5_K, false>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (qtype == kQ6_K)
    return swi ? launch_q6k<true>(W, Wu, n, k, X, T, Y, ldy, R, s) : launch_q6k<false>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (qtype == kIQ4_XS)
    return swi ? launch_iq4<true>(W, Wu, n, k, X, T, Y, ldy, R, s) : launch_iq4<false>(W, Wu, n, k, X, T, Y, ldy, R, s);
  if (qtype == kF16) {
    if (k % 256 == 0)
      return swi ? launch_f16<true>(W, Wu, n, k, X, T, Y, ldy, R, s) : launch_f16<false>(W, Wu, n, k, X, T, Y, ldy, R, s);
    return swi ? launch_q<kF16, true>(W, Wu, n, k, X, T, Y, ldy, R, s)
               : launch_q<kF16, false>(W, Wu, n, k, X, T, Y, ldy, R, s);
  }
  if (qtype == kQ4_0)
    return swi ? launch_q<kQ4_0, true>(W, Wu, n, k, X, T, Y, ldy, R, s)
               : launch_q<kQ4_0, false>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return swi ? launch_q<kQ8_0, true>(W, Wu, n, k, X, T, Y, ldy, R, s)
             : launch_q<kQ8_0, false>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

}  // namespace apr
