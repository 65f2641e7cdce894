// fp16-input tensor-core GEMM over Q4_0 / Q8_0 blocks, sm_103a (tcgen05 + TMA).
//
//   D[W rows][tokens] = dequant(W)[128 x k] . fp16(X)[BN x k]^T   (fp32 in TMEM)
//   Y[t][i] = D[i][t]  (+ R[t][i])       or  silu(Dg[i][t]) * Du[i][t]
//
// This is the f16 leg of aprender-serve 0.70.2 src/cuda/executor/gdn_prefill_ops.rs
// (qwen35_project_rows_f16: fp16 inputs, fp32 accumulation and output on the
// tensor cores), but the weight is never written out as fp16 or f32: raw GGUF
// blocks stream into shared memory and are decoded in registers straight into
// tensor memory, where the MMA reads them as its A operand. The same page's f32
// path dequantizes every weight to an f32 scratch per chunk, and the chunked
// driver of src/gguf/cuda/forward_qwen35_cuda_prefill.rs reports that dequant
// as a large share of prefill time (module constants PREFILL_MAX_CHUNK_ROWS and
// UNIFIED_PREFILL_CHUNK_ROWS); here it costs no memory traffic at all.
//
// One CTA computes one 128-row x BN-token output tile. Warp roles:
//   warp 0       TMA producer of raw weight chunks: 128 rows x 256 k (8 blocks
//                per row: 144 B for Q4_0, 272 B for Q8_0, the smallest box whose
//                width is a multiple of 16 bytes for both formats) into a ring
//                of S_RAW slots, with L2 prefetches PF chunks ahead
//   warp 1       TMEM allocator and the single MMA-issuing thread
//   warp 2       TMA producer of X tiles: BN tokens x 64 k of the fp16 copy of X,
//                128-byte swizzled, into the B ring (S_B stages)
//   warp 3       idle
//   warps 4..    dequant warpgroups: each thread owns one of the 128 rows (its
//                TMEM lane), decodes 2 blocks (64 k) per stage from the raw slot
//                and stores them as 32 columns of fp16 pairs into an A stage in
//                TMEM (S_A stages); with one weight, two warpgroups take
//                alternate stages, with gate/up one warpgroup per weight. Then
//                the same warps read the accumulators out of TMEM and run the
//                epilogue.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the device
// status word and an abort flag in shared memory so that every role leaves its
// loop, drains its own TMA copies and MMAs, and the CTA frees its TMEM.

#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "apr_internal.h"
#include "dev_common.cuh"

namespace apr {
namespace {

constexpr int BM = 128;         // weight rows per tile (UMMA M)
constexpr int BK = 64;          // k per operand stage
constexpr int CHUNK = 256;      // k per raw TMA chunk
constexpr int SUBS = CHUNK / BK;
constexpr int A_COLS = BK / 2;  // TMEM columns of one A stage (two fp16 per column)
constexpr int PF = 4;           // raw chunks prefetched into L2 ahead of their TMA load

template <int QT, int EPI, int BN_, bool RTMA_ = false>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr int NM = EPI == kEpiSwiGLU ? 2 : 1;
  static constexpr int DQ = NM == 1 ? 2 : 1;           // warpgroups per weight (alternate stages)
  static constexpr int NWG = NM * DQ;                   // dequant / epilogue warpgroups
  // residual tile [BN tokens][128 rows] f32 fetched by TMA at kernel start
  static constexpr bool RTMA = RTMA_ && EPI == kEpiResidual;
  static constexpr int R_BYTES = RTMA ? BN * BM * 4 : 0;
  static constexpr int BB = QT == kQ4_0 ? 18 : 34;
  static constexpr int RAW_ROW = CHUNK / 32 * BB;     // 144 / 272 bytes
  static constexpr int RAW_BYTES = BM * RAW_ROW;      // one raw slot
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int S_A = 4;
  static constexpr int S_B = QT == kQ4_0 ? 6 : 5;
  static constexpr int S_RAW = NM == 1 ? (QT == kQ4_0 ? 3 : 2) : (QT == kQ4_0 ? 4 : 3);
  static constexpr int NTHREADS = 128 + 128 * NWG;
  static constexpr int ACC_COLS = NM * BN;
  static constexpr int A_COL0 = ACC_COLS;                       // first A column
  static constexpr int USED_COLS = ACC_COLS + NM * S_A * A_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 128 ? 128 : USED_COLS <= 256 ? 256 : 512;
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_B = 0;
  static constexpr int OFF_RAW = OFF_B + S_B * B_BYTES;
  static constexpr int OFF_R = OFF_RAW + S_RAW * RAW_BYTES;
  static constexpr int OFF_BAR = OFF_R + R_BYTES;
  static constexpr int NBAR = 2 * S_A + 2 * S_B + 2 * S_RAW + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;   // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(USED_COLS <= 512, "TMEM budget");
  static_assert(BN % (16 * NWG) == 0, "epilogue split");
};

// ---------------------------------------------------------------- dequant
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Q4_0 payload word p (bytes b0..b3 = elements e..e+3 low, e+16..e+19 high):
// out[0] = (w_e, w_e+1), out[1] = (w_e+2, w_e+3), out[2] = (w_e+16, w_e+17),
// out[3] = (w_e+18, w_e+19), each w = fp16(d * (nibble - 8)).
//   (0x6400 | n) is the fp16 1024 + n; minus 1032 gives n - 8 exactly.
//   (0x6400 | 16 n) is 1024 + 16 n; times 1/16 minus 72 gives n - 8 exactly.
__device__ __forceinline__ void q4_word(uint32_t p, __half2 d2, uint32_t (&out)[4]) {
  const uint32_t lo01 = __byte_perm(p, 0u, 0x4140);   // b0 . b1 .
  const uint32_t lo23 = __byte_perm(p, 0u, 0x4342);   // b2 . b3 .
  const __half2 k1032 = u32_as_h2(0x64086408u);        // 1032, 1032
  const __half2 k16th = u32_as_h2(0x2C002C00u);        // 1/16
  const __half2 km72 = u32_as_h2(0xD480D480u);         // -72
  const __half2 a = __hsub2(u32_as_h2((lo01 & 0x000F000Fu) | 0x64006400u), k1032);
  const __half2 b = __hsub2(u32_as_h2((lo23 & 0x000F000Fu) | 0x64006400u), k1032);
  const __half2 c = __hfma2(u32_as_h2((lo01 & 0x00F000F0u) | 0x64006400u), k16th, km72);
  const __half2 e = __hfma2(u32_as_h2((lo23 & 0x00F000F0u) | 0x64006400u), k16th, km72);
  out[0] = h2_as_u32(__hmul2_rn(a, d2));
  out[1] = h2_as_u32(__hmul2_rn(b, d2));
  out[2] = h2_as_u32(__hmul2_rn(c, d2));
  out[3] = h2_as_u32(__hmul2_rn(e, d2));
}

// Q8_0 payload word q (4 int8, elements e..e+3):
// out[0] = (w_e, w_e+1), out[1] = (w_e+2, w_e+3), w = fp16(d * q).
//   (0x6400 | (b ^ 0x80)) is 1024 + b + 128; minus 1152 gives b exactly.
__device__ __forceinline__ void q8_word(uint32_t q, __half2 d2, uint32_t (&out)[2]) {
  const uint32_t x = q ^ 0x80808080u;
  const __half2 k1152 = u32_as_h2(0x64806480u);  // 1152, 1152
  const __half2 a = __hsub2(u32_as_h2(__byte_perm(x, 0x64646464u, 0x5140)), k1152);
  const __half2 b = __hsub2(u32_as_h2(__byte_perm(x, 0x64646464u, 0x7362)), k1152);
  out[0] = h2_as_u32(__hmul2_rn(a, d2));
  out[1] = h2_as_u32(__hmul2_rn(b, d2));
}

__device__ __forceinline__ __half2 scale2(uint32_t dbits) {
  return u32_as_h2((dbits & 0xFFFFu) | (dbits << 16));
}

// Decodes one row's two blocks (64 k) at `src` (4-byte aligned) into 32 fp16
// pairs in k order: a[j] = (w_2j, w_2j+1), j = 0..31.
template <int QT>
__device__ __forceinline__ void dequant_row_stage(const uint8_t* src, uint32_t (&a)[32]) {
  const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src);
  if constexpr (QT == kQ4_0) {
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = s32[i];
    // block 0: d in bytes 0-1, payload in bytes 2..17; block 1: d in 18-19, payload 20..35
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __byte_perm(w[i], w[i + 1], 0x5432);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[4 + i] = w[5 + i];
    const __half2 d0 = scale2(w[0] & 0xFFFFu);
    const __half2 d1 = scale2(w[4] >> 16);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t o[4];
        q4_word(p[blk * 4 + i], blk ? d1 : d0, o);
        a[16 * blk + 2 * i] = o[0];          // elements 4i, 4i+1
        a[16 * blk + 2 * i + 1] = o[1];      // 4i+2, 4i+3
        a[16 * blk + 8 + 2 * i] = o[2];      // 16+4i, 16+4i+1
        a[16 * blk + 8 + 2 * i + 1] = o[3];  // 16+4i+2, 16+4i+3
      }
    }
  } else {
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) w[i] = s32[i];
    // block 0: d in bytes 0-1, payload 2..33; block 1: d in 34-35, payload 36..67
    const __half2 d0 = scale2(w[0] & 0xFFFFu);
    const __half2 d1 = scale2(w[8] >> 16);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t p = c < 8 ? __byte_perm(w[c], w[c + 1], 0x5432) : w[1 + c];
      uint32_t o[2];
      q8_word(p, c < 8 ? d0 : d1, o);
      a[2 * c] = o[0];
      a[2 * c + 1] = o[1];
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int QT, int EPI, int BN, bool RTMA>
__global__ void __launch_bounds__(Cfg<QT, EPI, BN, RTMA>::NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWu,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmR, int n, int k,
                   int T, float* Y, const float* R, unsigned* status) {
  using C = Cfg<QT, EPI, BN, RTMA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sRaw = smem + C::OFF_RAW;
  const float* sR = reinterpret_cast<const float*>(smem + C::OFF_R);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* fullA = bars;
  uint64_t* emptyA = fullA + C::S_A;
  uint64_t* fullB = emptyA + C::S_A;
  uint64_t* emptyB = fullB + C::S_B;
  uint64_t* rawFull = emptyB + C::S_B;
  uint64_t* rawEmpty = rawFull + C::S_RAW;
  uint64_t* accFull = rawEmpty + C::S_RAW;
  uint64_t* drain = accFull + 1;
  uint64_t* rFull = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM;
  const int t0 = blockIdx.y * BN;
  const int nk = k / BK;
  const int nchunks = k / CHUNK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S_A; ++i) {
      mbar_init(&fullA[i], 4 * C::NM);
      mbar_init(&emptyA[i], 1);
    }
    for (int i = 0; i < C::S_B; ++i) {
      mbar_init(&fullB[i], 1);
      mbar_init(&emptyB[i], 1);
    }
    for (int i = 0; i < C::S_RAW; ++i) {
      mbar_init(&rawFull[i], 1);
      mbar_init(&rawEmpty[i], 4 * C::DQ);
    }
    mbar_init(accFull, 1);
    mbar_init(drain, 1);
    mbar_init(rFull, 1);
    abort_flag[0] = 0;   // set by a wait that gives up
    abort_flag[1] = 0;   // never set: drain waits ignore the abort
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------ raw weight producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      if (C::NM == 2) tma_prefetch_desc(&tmWu);
      if (C::RTMA) {  // the residual tile is needed only by the epilogue: fetch it first
        mbar_arrive_expect_tx(rFull, C::R_BYTES);
        tma_load_2d(smem + C::OFF_R, &tmR, m0, t0, rFull);
      }
      for (int c = 0; c < PF && c < nchunks; ++c)
        for (int m = 0; m < C::NM; ++m)
          tma_prefetch_l2_2d(m ? (const void*)&tmWu : (const void*)&tmW, c * (C::RAW_ROW / 2), m0);
      int last_issued[C::S_RAW];
      for (int i = 0; i < C::S_RAW; ++i) last_issued[i] = -1;
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        for (int m = 0; m < C::NM && ok; ++m) {
          const int j = c * C::NM + m;
          const int slot = j % C::S_RAW;
          ok = mbar_wait(&rawEmpty[slot], ((j / C::S_RAW) & 1) ^ 1, abort_flag, status);
          if (!ok) break;
          const void* map = m ? (const void*)&tmWu : (const void*)&tmW;
          mbar_arrive_expect_tx(&rawFull[slot], C::RAW_BYTES);
          tma_load_2d(sRaw + slot * C::RAW_BYTES, map, c * (C::RAW_ROW / 2), m0, &rawFull[slot]);
          if (c + PF < nchunks) tma_prefetch_l2_2d(map, (c + PF) * (C::RAW_ROW / 2), m0);
          last_issued[slot] = j;
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (int i = 0; i < C::S_RAW; ++i)
          if (last_issued[i] >= 0) mbar_wait(&rawFull[i], (last_issued[i] / C::S_RAW) & 1, abort_flag + 1, status);
        if (C::RTMA) mbar_wait(rFull, 0, abort_flag + 1, status);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ activation producer
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      int last_issued[C::S_B];
      for (int i = 0; i < C::S_B; ++i) last_issued[i] = -1;
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int sb = i % C::S_B;
        ok = mbar_wait(&emptyB[sb], ((i / C::S_B) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        mbar_arrive_expect_tx(&fullB[sb], C::B_BYTES);
        tma_load_2d(sB + sb * C::B_BYTES, &tmX, i * BK, t0, &fullB[sb]);
        last_issued[sb] = i;
      }
      if (!ok) {
        for (int i = 0; i < C::S_B; ++i)
          if (last_issued[i] >= 0) mbar_wait(&fullB[i], (last_issued[i] / C::S_B) & 1, abort_flag + 1, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      bool ok = true;
      for (int i = 0; i < nk && ok; ++i) {
        const int sa = i % C::S_A, sb = i % C::S_B;
        ok = mbar_wait(&fullA[sa], (i / C::S_A) & 1, abort_flag, status) &&
             mbar_wait(&fullB[sb], (i / C::S_B) & 1, abort_flag, status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bdesc = smem_desc_sw128(sB + sb * C::B_BYTES);
#pragma unroll
        for (int m = 0; m < C::NM; ++m) {
          const uint32_t a_tmem = tmem_base + C::A_COL0 + (m * C::S_A + sa) * A_COLS;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // 16 k = 8 TMEM columns of A, +32 bytes of B inside its swizzle atom
            mma_f16_ts(tmem_base + m * BN, a_tmem + kk * 8, bdesc + 2 * kk, idesc, (i | kk) != 0);
          }
        }
        mma_commit(&emptyA[sa]);
        mma_commit(&emptyB[sb]);
      }
      if (ok) {
        mma_commit(accFull);
      } else {  // wait until the MMAs already issued have finished
        mma_commit(drain);
        mbar_wait(drain, 0, abort_flag + 1, status);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ dequant, then epilogue
    const int wg = (warp - 4) >> 2;                  // dequant warpgroup
    const int g = wg % C::NM;                        // which weight (0: W / gate, 1: up)
    const int par = wg / C::NM;                      // which stages: i % DQ == par
    const uint32_t q = (uint32_t)(warp & 3);         // lane quarter of TMEM this warp may access
    const uint32_t r = q * 32 + lane;                // tile row == TMEM lane
    const uint32_t lane_base = tmem_base + ((q * 32u) << 16);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int j = c * C::NM + g;
      const int slot = j % C::S_RAW;
      ok = __all_sync(0xffffffffu, mbar_wait(&rawFull[slot], (j / C::S_RAW) & 1, abort_flag, status));
      if (!ok) break;
      const uint8_t* raw_row = sRaw + slot * C::RAW_BYTES + r * C::RAW_ROW;
      for (int s = par; s < SUBS; s += C::DQ) {
        const int i = c * SUBS + s;
        const int sa = i % C::S_A;
        uint32_t a[32];
        dequant_row_stage<QT>(raw_row + s * 2 * C::BB, a);  // overlaps the wait below
        ok = __all_sync(0xffffffffu, mbar_wait(&emptyA[sa], ((i / C::S_A) & 1) ^ 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        tmem_st_32x32b_x32(lane_base + C::A_COL0 + (g * C::S_A + sa) * A_COLS, a);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&fullA[sa]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rawEmpty[slot]);
    }
    // epilogue: the warpgroups split the BN token columns
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(accFull, 0, abort_flag, status));
    if (ok && C::RTMA) ok = __all_sync(0xffffffffu, mbar_wait(rFull, 0, abort_flag, status));
    if (ok) {
      tc_fence_after();
      const int row = m0 + (int)r;
      constexpr int COLS_PER_WG = BN / C::NWG;
      for (int cb = wg * COLS_PER_WG; cb < (wg + 1) * COLS_PER_WG; cb += 16) {
        // residual without the shared tile: issue all 16 loads before any store
        // (Y may be R itself, so a load may not move past an earlier store)
        float rv[16];
        if (EPI == kEpiResidual && !C::RTMA) {
#pragma unroll
          for (int j2 = 0; j2 < 16; ++j2) {
            const int t = t0 + cb + j2;
            rv[j2] = (row < n && t < T) ? R[(size_t)t * n + row] : 0.f;
          }
        }
        uint32_t v[16];
        tmem_ld_32x32b_x16(lane_base + cb, v);
        uint32_t u[16];
        if (C::NM == 2) tmem_ld_32x32b_x16(lane_base + BN + cb, u);
        tmem_ld_wait();
        if (row < n) {
#pragma unroll
          for (int j2 = 0; j2 < 16; ++j2) {
            const int t = t0 + cb + j2;
            if (t < T) {
              const size_t o = (size_t)t * n + row;
              const float acc = __uint_as_float(v[j2]);
              float y;
              if (EPI == kEpiSwiGLU) {
                const float up = __uint_as_float(u[j2]);
                y = acc / (1.0f + expf(-acc)) * up;
              } else if (EPI == kEpiResidual) {
                y = acc + (C::RTMA ? sR[(cb + j2) * BM + (int)r] : rv[j2]);
              } else {
                y = acc;
              }
              Y[o] = y;
            }
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- X -> fp16
__global__ void __launch_bounds__(256) x_to_f16_kernel(const float* __restrict__ X, uint16_t* __restrict__ X16,
                                                       size_t count) {
  const size_t n8 = count / 8;
  const float4* X4 = reinterpret_cast<const float4*>(X);
  uint4* Y4 = reinterpret_cast<uint4*>(X16);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (size_t i = tid; i < n8; i += stride) {
    const float4 a = X4[2 * i], b = X4[2 * i + 1];
    const __half2 h0 = __floats2half2_rn(a.x, a.y), h1 = __floats2half2_rn(a.z, a.w);
    const __half2 h2 = __floats2half2_rn(b.x, b.y), h3 = __floats2half2_rn(b.z, b.w);
    Y4[i] = make_uint4(h2_as_u32(h0), h2_as_u32(h1), h2_as_u32(h2), h2_as_u32(h3));
  }
  for (size_t i = n8 * 8 + tid; i < count; i += stride) X16[i] = __half_as_ushort(__float2half_rn(X[i]));
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char* msg, size_t msg_len) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn) snprintf(msg, msg_len, "cuTensorMapEncodeTiled is not available from the driver");
  return fn;
}

bool make_map_2d(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* map, CUtensorMapDataType dt,
                 const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                 uint32_t box_outer, CUtensorMapSwizzle swz, char* msg, size_t msg_len) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return false;
  }
  return true;
}

template <int QT, int EPI, int BN, bool RTMA>
int launch_cfg(const void* W, const void* Wu, int n, int k, const uint16_t* X16, int T, float* Y,
               const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  using C = Cfg<QT, EPI, BN, RTMA>;
  auto fn = encode_fn(msg, msg_len);
  if (!fn) return -1;
  CUtensorMap mW, mWu, mX;
  const uint64_t row_bytes = (uint64_t)(k / 32) * C::BB;
  if (!make_map_2d(fn, &mW, CU_TENSOR_MAP_DATA_TYPE_UINT16, W, row_bytes / 2, (uint64_t)n, row_bytes,
                   C::RAW_ROW / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE, msg, msg_len))
    return -1;
  if (C::NM == 2) {
    if (!make_map_2d(fn, &mWu, CU_TENSOR_MAP_DATA_TYPE_UINT16, Wu, row_bytes / 2, (uint64_t)n, row_bytes,
                     C::RAW_ROW / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE, msg, msg_len))
      return -1;
  } else {
    mWu = mW;
  }
  if (!make_map_2d(fn, &mX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X16, (uint64_t)k, (uint64_t)T, (uint64_t)k * 2, BK,
                   BN, CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len))
    return -1;
  CUtensorMap mR = mX;
  if (C::RTMA) {  // residual [T][n] f32, box 128 rows x BN tokens
    if (!make_map_2d(fn, &mR, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, R, (uint64_t)n, (uint64_t)T, (uint64_t)n * 4, BM, BN,
                     CU_TENSOR_MAP_SWIZZLE_NONE, msg, msg_len))
      return -1;
  }

  auto kern = gemm_tc_kernel<QT, EPI, BN, RTMA>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) {
      snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return -1;
    }
    attr_set[dev] = 1;
  }
  const dim3 grid((n + BM - 1) / BM, (T + BN - 1) / BN);
  kern<<<grid, C::NTHREADS, C::SMEM, s>>>(mW, mWu, mX, mR, n, k, T, Y, R, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, msg_len, "gemm_tc launch: %s", cudaGetErrorString(e));
    return -1;
  }
  return 0;
}

}  // namespace

cudaError_t launch_x_to_f16(const float* X, uint16_t* X16, size_t count, cudaStream_t s) {
  size_t blocks = (count / 8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) blocks = 1;
  x_to_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(X, X16, count);
  return cudaGetLastError();
}

int launch_gemm_tc(int qtype, const void* W, const void* Wu, int n, int k, const uint16_t* X16, int T, float* Y,
                   const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  constexpr int BN = 128;
  // The residual tile goes through TMA when a row of R is a multiple of 16 bytes.
  const bool rtma = R && (n % 4) == 0;
  if (qtype == kQ4_0) {
    if (Wu) return launch_cfg<kQ4_0, kEpiSwiGLU, BN, false>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
    if (rtma) return launch_cfg<kQ4_0, kEpiResidual, BN, true>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
    if (R) return launch_cfg<kQ4_0, kEpiResidual, BN, false>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
    return launch_cfg<kQ4_0, kEpiPlain, BN, false>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
  }
  if (Wu) return launch_cfg<kQ8_0, kEpiSwiGLU, BN, false>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
  if (rtma) return launch_cfg<kQ8_0, kEpiResidual, BN, true>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
  if (R) return launch_cfg<kQ8_0, kEpiResidual, BN, false>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
  return launch_cfg<kQ8_0, kEpiPlain, BN, false>(W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len);
}

}  // namespace apr
