// Small-T GEMV over Q4_0 / Q8_0 blocks, exact fp32 arithmetic, streamed with
// 1-D bulk copies (the HBM-bound form of the single-token GEMVs gemv_q4_0_pf /
// gemv_q8_0_pf of oxibonsai-kernels 0.1.4 src/gpu_backend/cuda_q_std_prefill.rs).
//
// Persistent CTAs, one per SM: a producer warp streams groups of 16 weight
// rows, 2048 columns at a time (one contiguous run of blocks per row), into a
// ring of shared-memory stages with cp.async.bulk; 8 consumer warps each own 2
// of the 16 rows, and each lane one block pair (64 columns, 36 or 68 bytes,
// always 4-byte aligned) of those rows. This form takes rows of any length;
// rows that fit a stage of gemv_rows.cu go there instead. The decode is in
// gemv_decode.cuh.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"
#include "gemv_decode.cuh"

namespace apr {
namespace {

using namespace gemv;

constexpr int NCW = 8;                // consumer warps
constexpr int RW = 2;                 // rows per consumer warp
constexpr int G = NCW * RW;           // rows per group
constexpr int KC = 2048;              // columns per chunk: 32 lanes x one block pair
constexpr int NTHREADS = 32 * (NCW + 1);

// Ring depth: Q8_0 with eight tokens takes two stages, so that the ring and
// the X table of k = 4096 fit shared memory.
template <int QT, bool SWI, int TMAX>
struct BCfg {
  static constexpr int NM = SWI ? 2 : 1;
  static constexpr int BB = QT == kQ4_0 ? 18 : 34;
  static constexpr int CB = KC / 32 * BB;            // bytes of one row's chunk
  static constexpr int STAGE = NM * G * CB;
  static constexpr int NS = QT == kQ4_0 ? (SWI ? 3 : 4) : (SWI || TMAX == 8 ? 2 : 3);
  static constexpr int RING = NS * STAGE;
};

template <int QT, int TMAX, bool SWI>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemv_bulk_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ Wu, int n, int k,
                     const float* __restrict__ X, int T, float* Y, int ldy, const float* R, unsigned* status) {
  using C = BCfg<QT, SWI, TMAX>;
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
  build_x_table<QT>(X, T, k, xt, threadIdx.x, NCW * 32);
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
            pair_dot<QT, TMAX>(src, xp, T, npk * XPAIR, acc[m][r]);
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
          const size_t o = (size_t)t * ldy + row;
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
cudaError_t launch_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                     const float* R, unsigned* status, cudaStream_t s) {
  using C = BCfg<QT, SWI, TMAX>;
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
  kern<<<grid, NTHREADS, smem, s>>>((const uint8_t*)W, (const uint8_t*)Wu, n, k, X, T, Y, ldy, R, status);
  return cudaGetLastError();
}

template <int QT, bool SWI>
cudaError_t launch_q(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                     const float* R, unsigned* status, cudaStream_t s) {
  if (T <= 1) return launch_t<QT, 1, SWI>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (T <= 2) return launch_t<QT, 2, SWI>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (T <= 4) return launch_t<QT, 4, SWI>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  return launch_t<QT, 8, SWI>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
}

template <int QT, int TMAX>
size_t ring_bytes(bool swiglu) {
  return swiglu ? BCfg<QT, true, TMAX>::RING : BCfg<QT, false, TMAX>::RING;
}

template <int QT>
size_t ring_bytes_t(int T, bool swiglu) {  // the TMAX launch_q picks for T
  if (T <= 1) return ring_bytes<QT, 1>(swiglu);
  if (T <= 2) return ring_bytes<QT, 2>(swiglu);
  if (T <= 4) return ring_bytes<QT, 4>(swiglu);
  return ring_bytes<QT, 8>(swiglu);
}

}  // namespace

size_t gemv_bulk_smem(int qtype, int k, int T, bool swiglu) {
  const size_t ring = qtype == kQ4_0 ? ring_bytes_t<kQ4_0>(T, swiglu) : ring_bytes_t<kQ8_0>(T, swiglu);
  const size_t xt = ((size_t)T * (k / 64) * XPAIR * 4 + 15) & ~(size_t)15;
  return 1024 + ring + xt + 2 * 8 * 4 + 16;
}

bool gemv_bulk_fits(int qtype, int k, int T, bool swiglu) {
  if (!block32_format(qtype) || k % 256 != 0 || T < 1 || T > (swiglu ? 4 : 8)) return false;
  return gemv_bulk_smem(qtype, k, T, swiglu) <= 232448;
}

cudaError_t launch_gemv_bulk(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y,
                             int ldy, const float* R, unsigned* status, cudaStream_t s) {
  const bool swi = Wu != nullptr;
  if (qtype == kQ4_0)
    return swi ? launch_q<kQ4_0, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
               : launch_q<kQ4_0, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  return swi ? launch_q<kQ8_0, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
             : launch_q<kQ8_0, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
}

}  // namespace apr
