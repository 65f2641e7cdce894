// Row RMSNorm for the FFN sublayer, y = x / sqrt(mean(x^2) + eps) * w, written
// as fp16 (the input of the fp16-leg gate/up GEMM: the norm and the fp16
// conversion in one pass over X) or as fp32 (the GEMV and exact-leg inputs).
//
// The pages run this as the first step of the FFN sublayer (oxibonsai-kernels
// 0.1.4 src/gpu_backend/cuda_q_std_prefill.rs, encode_q_std_ffn_phase step 1,
// a batched RMSNorm with one CTA per row; aprender-serve
// src/gguf/cuda/forward_qwen35_cuda_prefill.rs, prefill_ffn_rows,
// batched_rmsnorm_into over hidden_dim with eps) and then convert to fp16 in a
// separate pass for their fp16 leg.
//
// One CTA of 256 threads per row: each thread sums the squares of its float4s
// in order, then warps and the CTA add in a fixed tree, so the result does not
// depend on timing; 1 / sqrt uses IEEE sqrt and division. HBM bound: 4 k bytes
// read and 2 k or 4 k written per row.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"

namespace apr {
namespace {

constexpr int RN_THREADS = 256;

template <bool F16>
__global__ void __launch_bounds__(RN_THREADS) rmsnorm_rows_kernel(const float* __restrict__ X,
                                                                  const float* __restrict__ w, float eps, int k,
                                                                  void* __restrict__ out) {
  // the GEMM after this kernel may launch at once: it reads only the weights
  // and what this kernel writes, after waiting for it
  grid_launch_dependents();
  const size_t row = blockIdx.x;
  const float4* x4 = reinterpret_cast<const float4*>(X + row * (size_t)k);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const int k4 = k / 4;
  float ss = 0.f;
  for (int i = threadIdx.x; i < k4; i += RN_THREADS) {
    const float4 v = x4[i];
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  __shared__ float wsum[RN_THREADS / 32];
  __shared__ float s_inv;
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < RN_THREADS / 32; ++i) t += wsum[i];
    s_inv = 1.0f / sqrtf(t / (float)k + eps);
  }
  __syncthreads();
  const float inv = s_inv;
  for (int i = threadIdx.x; i < k4; i += RN_THREADS) {
    const float4 v = x4[i], g = w4[i];
    const float y0 = v.x * inv * g.x, y1 = v.y * inv * g.y, y2 = v.z * inv * g.z, y3 = v.w * inv * g.w;
    if constexpr (F16) {
      const __half2 a = __floats2half2_rn(y0, y1), b = __floats2half2_rn(y2, y3);
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&a);
      o.y = *reinterpret_cast<const uint32_t*>(&b);
      reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + row * (size_t)k)[i] = o;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(out) + row * (size_t)k)[i] = make_float4(y0, y1, y2, y3);
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm_rows(const float* X, const float* w, float eps, int T, int k, void* out, bool f16,
                                cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (f16)
    rmsnorm_rows_kernel<true><<<T, RN_THREADS, 0, s>>>(X, w, eps, k, out);
  else
    rmsnorm_rows_kernel<false><<<T, RN_THREADS, 0, s>>>(X, w, eps, k, out);
  return cudaGetLastError();
}

}  // namespace apr
