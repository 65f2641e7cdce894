// Causal prefill attention over a KV cache on the tensor cores, head_dim 256:
// for query row t of a chunk (position pos0 + t) and query head h,
//   out[t][h] = sum_{j <= pos0 + t} softmax_j(q[t][h] . k[j][g] / 16) v[j][g],
//   g = h / (num_heads / num_kv_heads),
// with q, k and v rounded to fp16 for the products, fp32 accumulation and an
// fp32 online softmax; no score matrix goes to memory. This is the fused form
// of aprender-serve 0.70.2 src/cuda/executor/gdn_prefill_ops.rs
// (qwen35_flash_prefill_attention: f16 tensor-core inputs, f32 accumulation and
// online softmax, head_dim 256), whose unfused twin (qwen35_prefill_attention /
// qwen35_attention_pass: scores GEMM, causal mask and softmax, value GEMM per
// KV group) fixes the layouts, the mask and the head grouping.
//
// One CTA per (128 query rows, query head); the CTAs of the last query rows,
// which see the most keys, are launched first. Keys go in tiles of 64:
//   warps 0-3   own the 128 query rows (one row per thread, TMEM lane = row):
//               they put fp16 Q into tensor memory once, then per key tile read
//               the 64 scores, update the running max and sum, write the fp16
//               weights P into tensor memory, and at the end scale O by 1 / sum
//   warps 4-11  convert K and V tiles from the f32 cache to fp16 in shared
//               memory, 128-byte swizzled and K-major for the MMAs (V
//               transposed), two tiles ahead in a ring of three; keys past the
//               chunk's last position are written as zeros, never read
//   warp 4      also issues the MMAs (one elected lane): S = Q . K^T (M = 128,
//               N = 64, 16 steps of K = 16 over the head dim) and O += P . V
//               (M = 128, N = 256, 4 steps of K = 16 over the keys), with Q
//               and P read from tensor memory
// Tensor memory (512 columns): O fp32 [0, 256), S fp32 [256, 320), P fp16
// pairs [320, 352), Q fp16 pairs [384, 512).
// The softmax works in base 2 (scores times log2(e) / 16). The weights are
// taken against a reference max m_ref that is moved (rescaling O and the sum)
// only when the running max exceeds it by more than 8, so a weight is at most
// 2^8 and O is rewritten only when the max jumps; the sum adds the weights
// as rounded to fp16, the values the MMA multiplies.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the device
// status word, the CTA leaves its loop at the next block-wide barrier, waits
// (bounded) for its MMAs in flight and frees its tensor memory.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"

namespace apr {
namespace {

constexpr int AD = 256;                          // head dim
constexpr int AQ = 128;                          // query rows per CTA (MMA M, TMEM lanes)
constexpr int AKEY = 64;                         // keys per tile
constexpr int ANBUF = 3;                         // K/V tile ring
constexpr int SOFT_WARPS = 4;
constexpr int LOAD_WARPS = 8;
constexpr int LOAD_THREADS = 32 * LOAD_WARPS;
constexpr int A_THREADS = 32 * (SOFT_WARPS + LOAD_WARPS);
constexpr int K_PANEL = AKEY * 128;              // [64 keys][64 dims] fp16, 8 KB
constexpr int K_BYTES = (AD / 64) * K_PANEL;     // four panels, 32 KB
constexpr int V_BYTES = AD * 128;                // [256 dims][64 keys] fp16, 32 KB
constexpr int BUF_BYTES = K_BYTES + V_BYTES;
constexpr int OFF_BAR = ANBUF * BUF_BYTES;
constexpr int A_SMEM = OFF_BAR + 64 + 1024;      // barriers, TMEM holder, flags; alignment slack
constexpr uint32_t COL_O = 0, COL_S = 256, COL_P = 320, COL_Q = 384;
constexpr uint32_t A_TMEM_COLS = 512;
constexpr float kRescaleAbove = 8.0f;            // log2 of the largest weight kept unscaled
static_assert(A_SMEM <= 232448, "shared memory budget");
static_assert(AKEY * (AD / 8) == 8 * LOAD_THREADS && AD * (AKEY / 8) == 8 * LOAD_THREADS, "8 chunks a thread");

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Keys [kb, kb + 64) of KV head g into a ring buffer. K: four panels [64 keys]
// [64 dims], one 128-byte row per key; V transposed: [256 dims][64 keys], one
// 128-byte row per dim; 16-byte chunk c of row r sits at chunk c ^ (r & 7)
// (the 128-byte swizzle). Keys >= nkeys are zeros.
__device__ __forceinline__ void load_kv_tile(const float* __restrict__ Kc, const float* __restrict__ Vc,
                                             size_t kv_dim, int g, int kb, int nkeys, uint8_t* buf, int ltid) {
  const float* kbase = Kc + (size_t)g * AD;
  const float* vbase = Vc + (size_t)g * AD;
#pragma unroll 4
  for (int i = 0; i < 8; ++i) {
    const int c = ltid + LOAD_THREADS * i;
    const int key = c >> 5, dc = c & 31;         // 32 chunks of 8 dims per key
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (kb + key < nkeys) {
      const float4* src = reinterpret_cast<const float4*>(kbase + (size_t)(kb + key) * kv_dim + dc * 8);
      const float4 a = __ldg(src), b = __ldg(src + 1);
      o = make_uint4(pack_half2(a.x, a.y), pack_half2(a.z, a.w), pack_half2(b.x, b.y), pack_half2(b.z, b.w));
    }
    *reinterpret_cast<uint4*>(buf + (dc >> 3) * K_PANEL + key * 128 + (((dc & 7) ^ (key & 7)) << 4)) = o;
  }
  uint8_t* vt = buf + K_BYTES;
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int c = ltid + LOAD_THREADS * i;
    const int d = c & (AD - 1), kg = c >> 8;     // dim d, keys 8 kg .. 8 kg + 7
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int key = kb + kg * 8 + e;
      x[e] = key < nkeys ? __ldg(vbase + (size_t)key * kv_dim + d) : 0.f;
    }
    *reinterpret_cast<uint4*>(vt + d * 128 + ((kg ^ (d & 7)) << 4)) =
        make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]), pack_half2(x[6], x[7]));
  }
}

__global__ void __launch_bounds__(A_THREADS, 1)
    prefill_attention_kernel(const float* __restrict__ Q, const float* __restrict__ Kc, const float* __restrict__ Vc,
                             float* __restrict__ O, int T, int pos0, int num_heads, int num_kv_heads,
                             unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* barS = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* barO = barS + 1;
  uint64_t* drain = barS + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(barS + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(barS + 4);

  const int warp = threadIdx.x >> 5;
  const int nqt = (T + AQ - 1) / AQ;
  const int h = blockIdx.x % num_heads;
  const int t0 = (nqt - 1 - (int)(blockIdx.x / num_heads)) * AQ;
  const int g = h / (num_heads / num_kv_heads);
  const size_t q_dim = (size_t)num_heads * AD, kv_dim = (size_t)num_kv_heads * AD;
  const int nkeys = pos0 + min(t0 + AQ, T);      // keys this CTA's rows see
  const int nkt = (nkeys + AKEY - 1) / AKEY;

  if (threadIdx.x == 0) {
    mbar_init(barS, 1);
    mbar_init(barO, 1);
    mbar_init(drain, 1);
    abort_flag[0] = 0;
    abort_flag[1] = 0;   // never set: the drain wait ignores the abort
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_holder, A_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // softmax rows: thread r = query row t0 + r = TMEM lane r
  const int r = threadIdx.x;
  const int t = t0 + r;
  const uint32_t lane_addr = tmem_base + ((uint32_t)(warp * 32) << 16);
  const int ltid = threadIdx.x - SOFT_WARPS * 32;

  // ---- prologue: Q into tensor memory, K/V tiles 0 and 1 into the ring
  if (warp < SOFT_WARPS) {
    const float* qrow = Q + (size_t)t * q_dim + (size_t)h * AD;
#pragma unroll 1
    for (int cb = 0; cb < AD / 64; ++cb) {
      uint32_t a[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < T) v = __ldg(reinterpret_cast<const float4*>(qrow + cb * 64) + i);
        a[2 * i] = pack_half2(v.x, v.y);
        a[2 * i + 1] = pack_half2(v.z, v.w);
      }
      tmem_st_32x32b_x32(lane_addr + COL_Q + cb * 32, a);
    }
    tmem_st_wait();
    tc_fence_before();
  } else {
    load_kv_tile(Kc, Vc, kv_dim, g, 0, nkeys, smem, ltid);
    if (nkt > 1) load_kv_tile(Kc, Vc, kv_dim, g, AKEY, nkeys, smem + BUF_BYTES, ltid);
    fence_proxy_async_smem();
  }
  __syncthreads();

  constexpr uint32_t IDESC_S = idesc_f16_f32(AQ, AKEY);
  constexpr uint32_t IDESC_O = idesc_f16_f32(AQ, AD);
  const float sl2 = 1.4426950408889634f / 16.0f;   // log2(e) / sqrt(256)
  const int plim = pos0 + min(t, T - 1);            // last key row t sees (rows past T: the last row's)
  float m_run = -INFINITY, m_ref = 0.f, l = 0.f;
  bool aborted = false;

#pragma unroll 1
  for (int j = 0; j < nkt; ++j) {
    uint8_t* buf = smem + (j % ANBUF) * BUF_BYTES;
    // (1) S = Q . K_j^T
    if (warp == SOFT_WARPS) {
      tc_fence_after();
      const uint64_t kdesc = smem_desc_sw128(buf);
#pragma unroll
      for (int kk = 0; kk < AD / 16; ++kk)
        mma_f16_ts_elect(tmem_base + COL_S, tmem_base + COL_Q + 8 * kk,
                         kdesc + (uint64_t)(((kk >> 2) * K_PANEL) >> 4) + 2 * (kk & 3), IDESC_S, kk != 0);
      mma_commit_elect(barS);
    }
    bool ok = true;
    if (warp < SOFT_WARPS) {
      // (2) softmax of tile j (its completion also means O += P . V_{j-1} is done)
      ok = __all_sync(0xffffffffu, mbar_wait(barS, (uint32_t)(j & 1), abort_flag, status));
      if (ok) {
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld_32x32b_x32(lane_addr + COL_S, sv);
        tmem_ld_32x32b_x32(lane_addr + COL_S + 32, sv + 32);
        tmem_ld_wait_regs(sv);
        regs_after_wait(sv + 32);
        const int kb = j * AKEY;
        float s[64];
        float m_tile = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] = kb + c <= plim ? __uint_as_float(sv[c]) * sl2 : -INFINITY;
          m_tile = fmaxf(m_tile, s[c]);
        }
        const float m_new = fmaxf(m_run, m_tile);
        if (j == 0) {
          m_ref = m_new;   // key 0 is visible to every row: finite
        } else if (__any_sync(0xffffffffu, m_new > m_ref + kRescaleAbove)) {
          // the whole warp moves its reference (tensor-memory access is per warp)
          const float f = exp2f(m_ref - m_new);
          l *= f;
#pragma unroll 1
          for (int cb = 0; cb < AD / 32; ++cb) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(lane_addr + COL_O + cb * 32, ov);
            tmem_ld_wait_regs(ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
            tmem_st_32x32b_x32(lane_addr + COL_O + cb * 32, ov);
          }
          m_ref = m_new;
        }
        m_run = m_new;
        uint32_t pv[32];
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const __half2 p = __floats2half2_rn(exp2f(s[2 * c] - m_ref), exp2f(s[2 * c + 1] - m_ref));
          const float2 pf = __half22float2(p);
          lsum += pf.x + pf.y;
          pv[c] = *reinterpret_cast<const uint32_t*>(&p);
        }
        l += lsum;
        tmem_st_32x32b_x32(lane_addr + COL_P, pv);
        tmem_st_wait();
        tc_fence_before();
      }
    } else if (j + 2 < nkt) {
      // (2') tile j + 2 into the buffer of tile j - 1, whose MMAs are done once S_j is
      ok = __all_sync(0xffffffffu, mbar_wait(barS, (uint32_t)(j & 1), abort_flag, status));
      if (ok) {
        load_kv_tile(Kc, Vc, kv_dim, g, (j + 2) * AKEY, nkeys, smem + ((j + 2) % ANBUF) * BUF_BYTES, ltid);
        fence_proxy_async_smem();
      }
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    // (3) O += P_j . V_j
    if (warp == SOFT_WARPS) {
      tc_fence_after();
      const uint64_t vdesc = smem_desc_sw128(buf + K_BYTES);
#pragma unroll
      for (int kk = 0; kk < AKEY / 16; ++kk)
        mma_f16_ts_elect(tmem_base + COL_O, tmem_base + COL_P + 8 * kk, vdesc + 2 * kk, IDESC_O, (j | kk) != 0);
      if (j == nkt - 1) mma_commit_elect(barO);
    }
  }

  // ---- epilogue: O / l to global memory
  if (!aborted && warp < SOFT_WARPS) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(barO, 0, abort_flag, status));
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l;
      float* orow = O + (size_t)t * q_dim + (size_t)h * AD;
#pragma unroll 1
      for (int cb = 0; cb < AD / 32; ++cb) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(lane_addr + COL_O + cb * 32, ov);
        tmem_ld_wait_regs(ov);
        if (t < T) {
          float4* dst = reinterpret_cast<float4*>(orow + cb * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                                 __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
        }
      }
    }
  }
  if (aborted && warp == SOFT_WARPS) {
    // wait until the MMAs already issued have finished
    mma_commit_elect(drain);
    __all_sync(0xffffffffu, mbar_wait(drain, 0, abort_flag + 1, status));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem_base, A_TMEM_COLS);
}

}  // namespace

cudaError_t launch_prefill_attention(const float* Q, const float* K, const float* V, float* O, int T, int pos0,
                                     int num_heads, int num_kv_heads, unsigned* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, A_SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  const long long grid = (long long)((T + AQ - 1) / AQ) * num_heads;
  prefill_attention_kernel<<<(unsigned)grid, A_THREADS, A_SMEM, s>>>(Q, K, V, O, T, pos0, num_heads, num_kv_heads,
                                                                     status);
  return cudaGetLastError();
}

}  // namespace apr
