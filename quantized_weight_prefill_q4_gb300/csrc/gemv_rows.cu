// Single-token GEMV (T = 1) over Q4_0 / Q8_0 blocks, exact fp32 arithmetic,
// streaming whole weight rows (the HBM-bound form of the single-token GEMVs
// gemv_q4_0_pf / gemv_q8_0_pf of oxibonsai-kernels 0.1.4
// src/gpu_backend/cuda_q_std_prefill.rs).
//
// Persistent CTAs, one per SM; CTA c takes rows [n c / grid, n (c + 1) / grid),
// which lie contiguously in memory. A producer warp streams them with one
// cp.async.bulk per stage: RS whole rows (RS = 16 KB / the bytes of a row, the
// W rows then the Wu rows for gate/up) into a ring of 8 stages.
//
// Consumers: a row has P = k / 64 block pairs and PW = P / 64 (rounded up)
// warps cover it, each lane two pairs (the exact fp32 decode takes about two
// instructions a product, so the SM is issue-bound: two independent pairs a
// lane and no CTA-wide barrier keep the issue slots busy). The 8 consumer warps
// form RG = 8 / PW row groups; thread (group g, warp wi of the group, lane l)
// holds the 128 X values of pairs wi 64 + l and wi 64 + 32 + l in registers for
// the whole kernel (from the X table, built in shared memory with coalesced
// loads and pre-scaled as gemv_decode.cuh describes) and takes those pairs of
// the CTA's rows r0 + g, r0 + g + RG, ... (whichever stage holds them, so
// every group has work even when a stage holds fewer rows than there are
// groups, and warps run ahead into later stages). A warp reduces its row partial with
// shuffles; with one warp a row it stores the result at once, otherwise the last
// of the row's warps to finish (a shared-memory counter) adds the PW partials
// in a fixed order, so the result does not depend on timing.
//
// Programmatic dependent launch: the producer streams W without waiting for
// the preceding kernel (so W must not be an output of the preceding call of
// this library on the stream); X, R and Y are read or written only after
// griddepcontrol.wait, and the kernel lets the next kernel of the stream
// launch only after that wait, so at most the one kernel before it runs
// beside it.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"
#include "gemv_decode.cuh"

namespace apr {
namespace {

using namespace gemv;

constexpr int RNCW = 8;                        // consumer warps
constexpr int RNTHREADS = 32 * (RNCW + 1);
constexpr int RSTAGE = 16384;                  // bytes of one stage
constexpr int RNS = 8;                         // stages
constexpr int RMAXROWS = 128;                  // rows a CTA may take (residual and row slots)

int rows_per_stage(int qtype, int k, bool swiglu) {
  const long row_bytes = (long)(k / 32) * block_bytes(qtype);
  return (int)(RSTAGE / ((swiglu ? 2 : 1) * row_bytes));
}

template <int QT, bool SWI>
__global__ void __launch_bounds__(RNTHREADS, 1)
    gemv_rows_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ Wu, int n, int k,
                     const float* __restrict__ X, float* Y, const float* R, unsigned* status, int rs) {
  constexpr int NM = SWI ? 2 : 1;
  constexpr int BB = QT == kQ4_0 ? 18 : 34;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte aligned base, by pointer arithmetic on the shared array so that
  // the compiler keeps the shared address space
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int npk = k / 64;  // block pairs per row
  const int PW = (npk + 63) / 64;  // warps per row
  float* part = reinterpret_cast<float*>(smem + RNS * RSTAGE);      // [row slot][NM][PW]
  float* rres = part + RMAXROWS * NM * 8;                             // residual of the CTA's rows
  unsigned* done = reinterpret_cast<unsigned*>(rres + RMAXROWS);      // warps finished, per row slot
  float* xt = reinterpret_cast<float*>(done + RMAXROWS);              // X table
  uint64_t* bars = reinterpret_cast<uint64_t*>(xt + npk * XPAIR);
  uint64_t* full = bars;
  uint64_t* empty = bars + RNS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * RNS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row_bytes = (size_t)(k / 32) * BB;
  const int r0 = (int)((long)n * blockIdx.x / gridDim.x);
  const int r1 = (int)((long)n * (blockIdx.x + 1) / gridDim.x);
  const int nst = (r1 - r0 + rs - 1) / rs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RNS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], RNCW);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < RMAXROWS; i += RNTHREADS) done[i] = 0;
  __syncthreads();

  if (warp == RNCW) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      int last[RNS];
      for (int i = 0; i < RNS; ++i) last[i] = -1;
      bool ok = true;
      for (int s = 0; s < nst && ok; ++s) {
        const int st = s % RNS;
        ok = mbar_wait(&empty[st], ((s / RNS) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        const int rb = r0 + s * rs, rows = min(rs, r1 - rb);
        const uint32_t bytes = (uint32_t)(rows * row_bytes);
        mbar_arrive_expect_tx(&full[st], bytes * NM);
        bulk_load_1d(smem + st * RSTAGE, W + (size_t)rb * row_bytes, bytes, &full[st]);
        if (SWI) bulk_load_1d(smem + st * RSTAGE + rs * row_bytes, Wu + (size_t)rb * row_bytes, bytes, &full[st]);
        last[st] = s;
      }
      if (!ok)  // let the copies in flight land before the CTA exits
        for (int i = 0; i < RNS; ++i)
          if (last[i] >= 0) mbar_wait(&full[i], (last[i] / RNS) & 1, abort_flag + 1, status);
    }
    return;
  }

  // ------------------------------------------------ consumers
  const int RG = RNCW / PW;          // row groups
  const int g = warp / PW, wi = warp % PW;
  const int pa = wi * 64 + lane, pb = pa + 32;  // this thread's block pairs
  const bool act_a = g < RG && pa < npk, act_b = g < RG && pb < npk;

  // X, R and Y may belong to the preceding kernel until it completes; once it
  // has, the next kernel may launch (so only this kernel runs beside it)
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  build_x_table<QT>(X, 1, k, xt, threadIdx.x, RNCW * 32);
  if (!SWI && R)
    for (int i = threadIdx.x; i < r1 - r0; i += RNCW * 32) rres[i] = R[r0 + i];
  named_sync(1, RNCW * 32);
  float xa[64], xb[64];
  if (act_a) load_x_pair(xt, pa, xa);
  if (act_b) load_x_pair(xt, pb, xb);

  bool ok = true;
  for (int s = 0; s < nst; ++s) {
    const int st = s % RNS;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (s / RNS) & 1, abort_flag, status));
    if (!ok) break;
    const int rb = r0 + s * rs, rows = min(rs, r1 - rb);
    if (g < RG) {
      // the stage's rows whose index within the CTA is g modulo RG
      for (int rr = ((g - (rb - r0)) % RG + RG) % RG; rr < rows; rr += RG) {
        float acc[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const uint8_t* rowp = smem + st * RSTAGE + (size_t)(m * rs + rr) * row_bytes;
          float a = 0.f, b = 0.f;
          if (act_a) pair_dot_regs<QT>(reinterpret_cast<const uint32_t*>(rowp + pa * 2 * BB), xa, a);
          if (act_b) pair_dot_regs<QT>(reinterpret_cast<const uint32_t*>(rowp + pb * 2 * BB), xb, b);
          a += b;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
          acc[m] = a;
        }
        const int slot = rb + rr - r0;  // the row's index within the CTA
        bool last = true;
        if (PW > 1) {
          // park the warp's partial; the last of the row's warps finishes the row
          if (lane == 0) {
#pragma unroll
            for (int m = 0; m < NM; ++m) part[(slot * NM + m) * 8 + wi] = acc[m];
            __threadfence_block();
            last = atomicAdd(&done[slot], 1u) == (unsigned)(PW - 1);
            if (last) {
              __threadfence_block();
#pragma unroll
              for (int m = 0; m < NM; ++m) {
                float v = 0.f;
                for (int w = 0; w < PW; ++w) v += part[(slot * NM + m) * 8 + w];
                acc[m] = v;
              }
            }
          }
        }
        if (lane == 0 && last) {
          float y;
          if (SWI) {
            y = acc[0] / (1.0f + expf(-acc[0])) * acc[NM - 1];
          } else {
            y = acc[0] + (R ? rres[slot] : 0.f);
          }
          Y[rb + rr] = y;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage's rows
  }
}

template <int QT, bool SWI>
cudaError_t launch_rows(const void* W, const void* Wu, int n, int k, const float* X, float* Y, const float* R,
                        unsigned* status, cudaStream_t s, int nsm) {
  const size_t smem = gemv_rows_smem(QT, k, 1);
  auto kern = gemv_rows_kernel<QT, SWI>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n < nsm ? n : nsm));
  cfg.blockDim = dim3(RNTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, (const uint8_t*)W, (const uint8_t*)Wu, n, k, X, Y, R, status,
                                     rows_per_stage(QT, k, SWI));
  if (e == cudaSuccess) e = cudaGetLastError();
  return e;
}

int device_sms() {
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return sms[dev] > 0 ? sms[dev] : 148;
}

}  // namespace

size_t gemv_rows_smem(int qtype, int k, int T) {
  (void)qtype;
  (void)T;
  return 128 + (size_t)RNS * RSTAGE + (size_t)RMAXROWS * (2 * 8 + 1 + 1) * 4 + (size_t)(k / 64) * XPAIR * 4 +
         2 * RNS * 8 + 16;
}

bool gemv_rows_fits(int qtype, int n, int k, int T, bool swiglu) {
  // block formats, one token; a row's warps within the consumer warps; whole rows in a
  // stage, each starting on a 16-byte boundary (k % 256 == 0); at most
  // RMAXROWS rows a CTA
  if (!block32_format(qtype) || T != 1 || k % 256 != 0 || (k / 64 + 63) / 64 > RNCW) return false;
  if ((n + device_sms() - 1) / device_sms() > RMAXROWS) return false;
  return rows_per_stage(qtype, k, swiglu) >= 1 && gemv_rows_smem(qtype, k, T) <= 232448;
}

cudaError_t launch_gemv_rows(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y,
                             const float* R, unsigned* status, cudaStream_t s) {
  (void)T;
  const bool swi = Wu != nullptr;
  const int nsm = device_sms();
  if (qtype == kQ4_0)
    return swi ? launch_rows<kQ4_0, true>(W, Wu, n, k, X, Y, R, status, s, nsm)
               : launch_rows<kQ4_0, false>(W, Wu, n, k, X, Y, R, status, s, nsm);
  return swi ? launch_rows<kQ8_0, true>(W, Wu, n, k, X, Y, R, status, s, nsm)
             : launch_rows<kQ8_0, false>(W, Wu, n, k, X, Y, R, status, s, nsm);
}

}  // namespace apr
