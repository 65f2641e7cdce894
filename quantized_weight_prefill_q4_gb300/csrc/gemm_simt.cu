// Exact-fp32 GEMM over Q4_0 / Q8_0 blocks (or F16 weights) on the CUDA cores (FFMA).
//
// The f32 leg of aprender-serve 0.70.2 src/cuda/executor/gdn_prefill_ops.rs
// (qwen35_project_rows: fp32 in and out, no TF32, because these projections
// feed a recurrence that compounds low-precision error), without the f32
// dequant scratch: each 64-row x 32-column weight tile is decoded exactly
// (fp16 d times a code of at most 8 bits, or a half, is exact in fp32) straight into
// shared memory, next to a 64-token x 32-column tile of X, and 256 threads
// each accumulate a 4 x 4 block of outputs. Works for any k % 32 == 0.
//
// Epilogues: plain, + residual, or silu(g) * u with two weight tiles.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"

namespace apr {
namespace {

constexpr int BM = 64;  // W rows
constexpr int BN = 64;  // tokens
constexpr int BK = 32;  // one block per row
constexpr int PAD = 4;

template <int QT>
__device__ __forceinline__ void decode8(const uint8_t* __restrict__ blk, int part, float (&w)[8]) {
  // part 0..3 -> elements 8*part .. 8*part+7 of the block
  if constexpr (QT == kF16) {  // 32 halves, 2-byte aligned
    const __half* h = reinterpret_cast<const __half*>(blk) + part * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = __half2float(h[e]);
    return;
  }
  const uint16_t db = (uint16_t)blk[0] | ((uint16_t)blk[1] << 8);
  const float d = __half2float(__ushort_as_half(db));
  if (QT == kQ4_0) {
    const uint8_t* p = blk + 2 + (part & 1) * 8;  // bytes of elements 8(part&1) ..
    const int sh = (part >> 1) * 4;              // parts 2, 3 are the high nibbles
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = d * (float)((int)((p[e] >> sh) & 0xF) - 8);
  } else {
    const int8_t* p = reinterpret_cast<const int8_t*>(blk + 2 + part * 8);
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = d * (float)p[e];
  }
}

template <int QT, int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const uint8_t* __restrict__ W,
                                                        const uint8_t* __restrict__ Wu, int n, int k,
                                                        const float* __restrict__ X, int T,
                                                        float* Y, int ldy,
                                                        const float* R) {
  constexpr int BB = QT == kQ4_0 ? 18 : (QT == kQ8_0 ? 34 : 64);
  constexpr int NM = EPI == kEpiSwiGLU ? 2 : 1;
  __shared__ float Ws[NM][BK][BM + PAD];
  __shared__ float Xs[BK][BN + PAD];

  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int m0 = blockIdx.x * BM, t0 = blockIdx.y * BN;
  const size_t row_bytes = (size_t)(k / 32) * BB;

  float acc[NM][4][4];
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[m][i][j] = 0.f;

  const int lr = tid >> 2;     // row (or token) this thread loads
  const int part = tid & 3;    // which 8 elements of the 32

  for (int kb = 0; kb < k / 32; ++kb) {
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      float w[8];
      const int row = m0 + lr;
      if (row < n) {
        decode8<QT>((m ? Wu : W) + (size_t)row * row_bytes + (size_t)kb * BB, part, w);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = 0.f;
      }
      // element order inside the block: Q4_0 parts are 0..7, 8..15, 16..23, 24..31
#pragma unroll
      for (int e = 0; e < 8; ++e) Ws[m][part * 8 + e][lr] = w[e];
    }
    {
      const int tok = t0 + lr;
      float xv[8];
      if (tok < T) {
        const float* xr = X + (size_t)tok * k + (size_t)kb * 32 + part * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] = xr[e];
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) Xs[part * 8 + e][lr] = xv[e];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float b[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Xs[kk][tx * 4 + j];
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        float a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = Ws[m][kk][ty * 4 + i];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[m][i][j] = fmaf(a[i], b[j], acc[m][i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tok = t0 + tx * 4 + j;
    if (tok >= T) continue;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = m0 + ty * 4 + i;
      if (row >= n) continue;
      const size_t o = (size_t)tok * ldy + row;
      float v;
      if (EPI == kEpiSwiGLU) {
        const float g = acc[0][i][j], u = acc[NM - 1][i][j];
        v = g / (1.0f + expf(-g)) * u;
      } else if (EPI == kEpiResidual) {
        v = acc[0][i][j] + R[o];
      } else {
        v = acc[0][i][j];
      }
      Y[o] = v;
    }
  }
}

template <int QT>
cudaError_t launch_q(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                     const float* R, cudaStream_t s) {
  const dim3 grid((n + BM - 1) / BM, (T + BN - 1) / BN);
  const uint8_t* w = (const uint8_t*)W;
  const uint8_t* wu = (const uint8_t*)Wu;
  if (Wu)
    gemm_simt_kernel<QT, kEpiSwiGLU><<<grid, 256, 0, s>>>(w, wu, n, k, X, T, Y, ldy, R);
  else if (R)
    gemm_simt_kernel<QT, kEpiResidual><<<grid, 256, 0, s>>>(w, wu, n, k, X, T, Y, ldy, R);
  else
    gemm_simt_kernel<QT, kEpiPlain><<<grid, 256, 0, s>>>(w, wu, n, k, X, T, Y, ldy, R);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_simt(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T,
                             float* Y, int ldy, const float* R, cudaStream_t s) {
  if (qtype == kF16) return launch_q<kF16>(W, Wu, n, k, X, T, Y, ldy, R, s);
  return qtype == kQ4_0 ? launch_q<kQ4_0>(W, Wu, n, k, X, T, Y, ldy, R, s)
                        : launch_q<kQ8_0>(W, Wu, n, k, X, T, Y, ldy, R, s);
}

}  // namespace apr
