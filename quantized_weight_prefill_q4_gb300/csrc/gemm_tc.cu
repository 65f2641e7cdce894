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
//                128-byte swizzled, into the B ring
//   warp 3       idle
//   warps 4..    dequant warpgroups: each thread owns one of the 128 rows (its
//                TMEM lane), decodes 2 blocks (64 k) per stage from the raw slot
//                and stores them as 32 columns of fp16 pairs into an A stage in
//                TMEM; A and B stages advance together (S of them); with one weight, two warpgroups take
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
#include <atomic>
#include <mutex>

#include "apr_internal.h"
#include "dev_common.cuh"

namespace apr {
namespace {

constexpr int BM = 128;         // weight rows per tile (UMMA M)
constexpr int CHUNK = 256;      // k per raw TMA chunk
constexpr int PF = 4;           // raw chunks prefetched into L2 ahead of their TMA load

// Residual handling: kRNone (no residual, or loads straight from R), kREarly
// (the residual tile is fetched by TMA into its own shared buffer at kernel
// start), kRLate (prefetched into L2 at kernel start, then fetched by TMA into
// the operand ring once the mainloop has finished with it).
enum RMode { kRNone = 0, kREarly = 1, kRLate = 2 };

// Two arithmetic legs share the kernel:
//   f16 leg:   a stage is 64 k; A = fp16(d * q') (two per TMEM column), B = fp16(X);
//              kind::f16, four K = 16 MMAs per stage.
//   exact leg: a stage is one 32-k block; A = d * q' exactly in fp32, split into
//              tf32 hi + lo (the product has at most 19 significant bits, so hi
//              + lo is exact), one per TMEM column (32 hi columns, 32 lo); B = X
//              split the same way (hi has the top 11 bits, lo the rest); per
//              K = 8 step three kind::tf32 MMAs accumulate hi.hi + hi.lo + lo.hi.
template <int QT, int EPI, int BN_, int RM_ = kRNone, bool EX_ = false>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr bool EX = EX_;
  static constexpr int BK = EX ? 32 : 64;               // k per operand stage (128 B of B per row)
  static constexpr int SUBS = CHUNK / BK;               // stages per raw chunk
  static constexpr int A_COLS = EX ? 64 : 32;           // TMEM columns of one A stage of one weight
  static constexpr int B_TILE = BN * 128;               // one 128-B-swizzled B tile
  static constexpr int NB = EX ? 2 : 1;                 // B tiles per stage (hi, lo)
  static constexpr int NM = EPI == kEpiSwiGLU ? 2 : 1;
  static constexpr int DQ = NM == 1 ? 2 : 1;           // warpgroups per weight (alternate stages)
  static constexpr int NWG = NM * DQ;                   // dequant / epilogue warpgroups
  static constexpr int RM = EPI == kEpiResidual ? RM_ : kRNone;
  static constexpr int BB = QT == kQ4_0 ? 18 : 34;
  static constexpr int RAW_ROW = CHUNK / 32 * BB;     // 144 / 272 bytes
  static constexpr int RAW_BYTES = BM * RAW_ROW;      // one raw slot
  static constexpr int B_BYTES = NB * B_TILE;
  static constexpr int R_BYTES = BN * BM * 4;          // residual tile
  // operand stages (A in TMEM and B in shared memory advance together)
  static constexpr int S = EX ? (NM == 2 ? 2 : 4) : (NM == 2 ? 4 : (BN == 256 ? 4 : (QT == kQ4_0 ? 6 : 5)));
  static constexpr int S_RAW = NM == 1 ? (QT == kQ4_0 ? 3 : 2) : (QT == kQ4_0 ? 4 : 3);
  static constexpr int NTHREADS = 128 + 128 * NWG;
  static constexpr int ACC_COLS = NM * BN;
  static constexpr int A_COL0 = ACC_COLS;                       // first A column
  static constexpr int USED_COLS = ACC_COLS + NM * S * A_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 128 ? 128 : USED_COLS <= 256 ? 256 : 512;
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_B = 0;
  static constexpr int OFF_RAW = OFF_B + S * B_BYTES;
  static constexpr int OFF_R = OFF_RAW + S_RAW * RAW_BYTES;
  static constexpr int OFF_BAR = OFF_R + (RM == kREarly ? R_BYTES : 0);
  static constexpr int NBAR = 2 * S + 2 * S_RAW + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;   // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(USED_COLS <= 512, "TMEM budget");
  static_assert(BN % (16 * NWG) == 0, "epilogue split");
  static_assert(RM != kRLate || R_BYTES <= S * B_BYTES, "late residual tile fits the operand ring");
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

// Exact leg: decodes one row's block b of the raw chunk at `chunk_row` (the
// row's 144 / 272 bytes, 4-byte aligned; the block starts 2 bytes off a word
// boundary when b is odd) into w = d * q' in fp32, split into tf32 hi (top 11
// significant bits: 13 low mantissa bits cleared) and lo = w - hi, element j in
// column j.
template <int QT>
__device__ __forceinline__ void dequant_block_exact(const uint8_t* chunk_row, int b, uint32_t (&hi)[32],
                                                    uint32_t (&lo)[32]) {
  constexpr int BB = QT == kQ4_0 ? 18 : 34;
  constexpr int NW = QT == kQ4_0 ? 5 : 9;  // words covering the block from its aligned start
  const int off = b * BB;
  const uint32_t* s32 = reinterpret_cast<const uint32_t*>(chunk_row + (off & ~3));
  uint32_t w[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) w[i] = s32[i];
  const bool odd = (off & 3) != 0;  // block starts at byte 2 of w[0]
  // realigned block words: x[i] = bytes 4i..4i+3 of the block (the last one
  // only partly inside the block)
  const uint32_t sel = odd ? 0x5432u : 0x3210u;
  uint32_t x[NW];
#pragma unroll
  for (int i = 0; i < NW - 1; ++i) x[i] = __byte_perm(w[i], w[i + 1], sel);
  x[NW - 1] = __byte_perm(w[NW - 1], 0u, sel);
  const float d = __half2float(__ushort_as_half((unsigned short)(x[0] & 0xFFFFu)));
  // payload words: bytes 2..BB-1 of the block
  float v[32];
  if constexpr (QT == kQ4_0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t p = __byte_perm(x[i], x[i + 1], 0x5432);  // payload bytes 4i..4i+3
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t byte = (p >> (8 * m)) & 0xFFu;
        v[4 * i + m] = __uint_as_float(0x4B000000u | (byte & 0xFu)) - 8388616.0f;          // low nibble
        v[16 + 4 * i + m] = __uint_as_float(0x4B000000u | (byte >> 4)) - 8388616.0f;       // high nibble
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t q = __byte_perm(x[i], x[i + 1], 0x5432) ^ 0x80808080u;  // int8 + 128
#pragma unroll
      for (int m = 0; m < 4; ++m)
        v[4 * i + m] = __uint_as_float(__byte_perm(q, 0x4B000000u, 0x7540 + m)) - 8388736.0f;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float wv = v[j] * d;  // exact: <= 8 x 11 significant bits
    const uint32_t h = __float_as_uint(wv) & 0xFFFFE000u;
    hi[j] = h;
    lo[j] = __float_as_uint(wv - __uint_as_float(h));  // exact
  }
}

// ---------------------------------------------------------------- kernel
template <int QT, int EPI, int BN, int RM, bool EX>
__global__ void __launch_bounds__(Cfg<QT, EPI, BN, RM, EX>::NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWu,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmX2,
                   const __grid_constant__ CUtensorMap tmR, int n, int k, int T, float* Y, const float* R,
                   unsigned* status, float* ws, unsigned long long* tickets, unsigned epoch) {
  using C = Cfg<QT, EPI, BN, RM, EX>;
  constexpr int BK = C::BK, SUBS = C::SUBS, A_COLS = C::A_COLS;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the shared array so that
  // the compiler keeps the shared address space (shared loads, not generic)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sRaw = smem + C::OFF_RAW;
  const float* sR = reinterpret_cast<const float*>(smem + (C::RM == kRLate ? C::OFF_B : C::OFF_R));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;              // stage ready: B landed and every A writer arrived
  uint64_t* empty = full + C::S;      // stage free: its MMAs completed
  uint64_t* rawFull = empty + C::S;
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
  // split-K: CTA z of gridDim.z takes raw chunks [c0, c1); ring indices are local
  const int nchunks_all = k / CHUNK;
  const int nsplit = gridDim.z, z = blockIdx.z;
  const int c0 = (int)((long)z * nchunks_all / nsplit), c1 = (int)((long)(z + 1) * nchunks_all / nsplit);
  const int nchunks = c1 - c0;
  const int nk = nchunks * SUBS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; ++i) {
      mbar_init(&full[i], 1 + 4 * C::NM);
      mbar_init(&empty[i], 1);
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
    *reinterpret_cast<unsigned*>(smem + C::OFF_MISC + 16) = 0;  // split-K epilogue arrivals
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
      if (C::RM == kREarly) {  // the residual tile is needed only by the epilogue: fetch it first
        mbar_arrive_expect_tx(rFull, C::R_BYTES);
        tma_load_2d(smem + C::OFF_R, &tmR, m0, t0, rFull);
      } else if (C::RM == kRLate) {
        tma_prefetch_l2_2d(&tmR, m0, t0);
      }
      for (int c = 0; c < PF && c < nchunks; ++c)
        for (int m = 0; m < C::NM; ++m)
          tma_prefetch_l2_2d(m ? (const void*)&tmWu : (const void*)&tmW, (c0 + c) * (C::RAW_ROW / 2), m0);
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
          tma_load_2d(sRaw + slot * C::RAW_BYTES, map, (c0 + c) * (C::RAW_ROW / 2), m0, &rawFull[slot]);
          if (c + PF < nchunks) tma_prefetch_l2_2d(map, (c0 + c + PF) * (C::RAW_ROW / 2), m0);
          last_issued[slot] = j;
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (int i = 0; i < C::S_RAW; ++i)
          if (last_issued[i] >= 0) mbar_wait(&rawFull[i], (last_issued[i] / C::S_RAW) & 1, abort_flag + 1, status);
        if (C::RM == kREarly) mbar_wait(rFull, 0, abort_flag + 1, status);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ activation producer
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      if (C::EX) tma_prefetch_desc(&tmX2);
      // X (fp16 or split) is written by the conversion kernel that may still be
      // running when this grid starts (programmatic dependent launch); nothing
      // else this kernel reads or writes is touched by that kernel
      grid_dependency_wait();
      bool ok = true;
      int last = -1;
      for (int i = 0; i < nk; ++i) {
        const int st = i % C::S;
        ok = mbar_wait(&empty[st], ((i / C::S) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[st], C::B_BYTES);
        const int kx = (c0 * SUBS + i) * BK;
        tma_load_2d(sB + st * C::B_BYTES, &tmX, kx, t0, &full[st]);
        if (C::EX) tma_load_2d(sB + st * C::B_BYTES + C::B_TILE, &tmX2, kx, t0, &full[st]);
        last = i;
      }
      // After a give-up, wait (bounded) on the last stage issued: its phase
      // also needs the dequant warps, so it may never complete, but by the
      // time the bounded wait ends every copy issued has landed.
      if (!ok && last >= 0) mbar_wait(&full[last % C::S], (last / C::S) & 1, abort_flag + 1, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = C::EX ? idesc_tf32_f32(BM, BN) : idesc_f16_f32(BM, BN);
      const uint64_t bdesc0 = smem_desc_sw128(sB);
      bool ok = true;
      int st = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nk && ok; ++i) {
        ok = mbar_wait(&full[st], ph, abort_flag, status);
        if (!ok) break;
        tc_fence_after();
        // stage st of B starts st * B_BYTES later: (B_BYTES >> 4) descriptor units
        const uint64_t bdesc = bdesc0 + (uint64_t)((st * C::B_BYTES) >> 4);
#pragma unroll
        for (int m = 0; m < C::NM; ++m) {
          const uint32_t a_tmem = tmem_base + C::A_COL0 + (m * C::S + st) * A_COLS;
          if constexpr (C::EX) {
            constexpr uint64_t lo_b = (uint64_t)(C::B_TILE >> 4);  // X lo tile follows X hi
#pragma unroll
            for (int kk = 0; kk < BK / 8; ++kk) {
              // 8 k = 8 TMEM columns of A (hi at +0, lo at +32), +32 bytes of B
              const uint32_t ah = a_tmem + kk * 8, al = ah + 32;
              const uint64_t bh = bdesc + 2 * kk, bl = bh + lo_b;
              mma_tf32_ts(tmem_base + m * BN, ah, bh, idesc, (i | kk) != 0);
              mma_tf32_ts(tmem_base + m * BN, ah, bl, idesc, 1);
              mma_tf32_ts(tmem_base + m * BN, al, bh, idesc, 1);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // 16 k = 8 TMEM columns of A, +32 bytes of B inside its swizzle atom
              mma_f16_ts(tmem_base + m * BN, a_tmem + kk * 8, bdesc + 2 * kk, idesc, (i | kk) != 0);
            }
          }
        }
        mma_commit(&empty[st]);
        if (++st == C::S) {
          st = 0;
          ph ^= 1u;
        }
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
        const int st = i % C::S;
        uint32_t a[32], a_lo[32];
        if constexpr (C::EX)
          dequant_block_exact<QT>(raw_row, s, a, a_lo);          // overlaps the wait below
        else
          dequant_row_stage<QT>(raw_row + s * 2 * C::BB, a);     // overlaps the wait below
        ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((i / C::S) & 1) ^ 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        tmem_st_32x32b_x32(lane_base + C::A_COL0 + (g * C::S + st) * A_COLS, a);
        if constexpr (C::EX) tmem_st_32x32b_x32(lane_base + C::A_COL0 + (g * C::S + st) * A_COLS + 32, a_lo);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rawEmpty[slot]);
    }
    // epilogue: the warpgroups split the BN token columns
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(accFull, 0, abort_flag, status));
    const int row = m0 + (int)r;
    constexpr int COLS_PER_WG = BN / C::NWG;
    const int cb0 = wg * COLS_PER_WG, cb1 = cb0 + COLS_PER_WG;
    const size_t tile = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
    float* partial = ws + tile * (size_t)(BN * BM);  // [BN tokens][128 rows]
    bool writer = true;  // this CTA writes Y
    if (nsplit == 2) {
      // split-K over two CTAs: the first to get here parks its fp32 partial in
      // the workspace and raises the tile's flag; the second waits for the
      // flag (the first is already in its epilogue), then writes Y = p0 + p1
      // (+ R) in split order, whichever CTA got here first
      // tile word: (epoch << 32) | arrivals this call; flag: epoch once the
      // partial is parked. Workspace memory is not cleared between calls: a
      // word from an earlier call (another epoch) counts as no arrival yet.
      volatile int* role = abort_flag + 2;
      unsigned* epi_done = reinterpret_cast<unsigned*>(smem + C::OFF_MISC + 16);  // zeroed at start
      unsigned long long* ticket = tickets + 2 * tile;
      unsigned* flag = reinterpret_cast<unsigned*>(tickets + 2 * tile + 1);
      if (threadIdx.x == 128) {
        int got = -1;
        if (ok) {
          unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ticket);
          for (;;) {
            const unsigned long long next =
                (unsigned)(old >> 32) == epoch ? old + 1 : ((unsigned long long)epoch << 32) | 1ull;
            const unsigned long long seen = atomicCAS(ticket, old, next);
            if (seen == old) {
              got = (int)(next & 0xFFFFFFFFull) - 1;
              break;
            }
            old = seen;
          }
        }
        *role = got;
      }
      named_sync(1, 128 * C::NWG);
      const int my_role = *role;
      writer = my_role == 1;
      if (my_role == 0) {
        if (ok) {
          tc_fence_after();
          for (int cb = cb0; cb < cb1; cb += 16) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(lane_base + cb, v);
            tmem_ld_wait();
#pragma unroll
            for (int j2 = 0; j2 < 16; ++j2) partial[(cb + j2) * BM + (int)r] = __uint_as_float(v[j2]);
          }
        }
        // no barrier here (a warp that gave up must not be waited for): each
        // warp counts itself in, the last one publishes the partial
        __threadfence();
        __syncwarp();
        if (lane == 0 && atomicAdd(epi_done, 1u) == 4u * C::NWG - 1u) atomicExch(flag, epoch);
      } else if (my_role == 1 && ok) {
        // bounded wait for the first CTA's partial
        if (lane == 0) {
          const unsigned long long t_start = global_ns();
          while (atomicAdd(flag, 0u) != epoch) {
            if (global_ns() - t_start > kWaitLimitNs) {
              atomicOr(status, kStatusTimeout);
              abort_flag[0] = 1;
              break;
            }
            __nanosleep(64);
          }
        }
        __syncwarp();
        ok = abort_flag[0] == 0;
        __threadfence();
      } else {
        writer = false;
      }
    }
    if (ok && writer && C::RM == kRLate && threadIdx.x == 128) {
      // every MMA has completed, so the operand ring is free: fetch the
      // residual tile (prefetched into L2 at kernel start) into it
      mbar_arrive_expect_tx(rFull, C::R_BYTES);
      tma_load_2d(smem + C::OFF_B, &tmR, m0, t0, rFull);
    }
    if (ok && writer && C::RM != kRNone) ok = __all_sync(0xffffffffu, mbar_wait(rFull, 0, abort_flag, status));
    if (ok && writer) {
      tc_fence_after();
      const bool first_is_z0 = z == 1;  // with a split, the parked partial belongs to the other CTA
      constexpr int CB_BATCH = COLS_PER_WG < 64 ? COLS_PER_WG : 64;
      for (int cbb = cb0; cbb < cb1; cbb += CB_BATCH) {
        // the other CTA's parked partial: all CB_BATCH loads in flight at once
        float other[CB_BATCH];
        if (nsplit == 2) {
#pragma unroll
          for (int q2 = 0; q2 < CB_BATCH; ++q2) other[q2] = __ldcg(partial + (cbb + q2) * BM + (int)r);
        }
#pragma unroll
        for (int sub = 0; sub < CB_BATCH; sub += 16) {
          const int cb = cbb + sub;
          // residual without the shared tile: issue all 16 loads before any store
          // (Y may be R itself, so a load may not move past an earlier store)
          float rv[16];
          if (EPI == kEpiResidual && C::RM == kRNone) {
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
                float acc = __uint_as_float(v[j2]);
                if (nsplit == 2) acc = first_is_z0 ? other[sub + j2] + acc : acc + other[sub + j2];  // p0 + p1
                float y;
                if (EPI == kEpiSwiGLU) {
                  const float up = __uint_as_float(u[j2]);
                  y = acc / (1.0f + expf(-acc)) * up;
                } else if (EPI == kEpiResidual) {
                  y = acc + (C::RM != kRNone ? sR[(cb + j2) * BM + (int)r] : rv[j2]);
                } else {
                  y = acc;
                }
                Y[o] = y;
              }
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
  grid_launch_dependents();
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

// ---------------------------------------------------------------- X -> tf32 hi, lo
// hi = x with its 13 low mantissa bits cleared, lo = x - hi (exact).
__global__ void __launch_bounds__(256) x_split_kernel(const float* __restrict__ X, float* __restrict__ hi,
                                                      float* __restrict__ lo, size_t count) {
  grid_launch_dependents();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const float x = X[i];
    const float h = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    hi[i] = h;
    lo[i] = x - h;
  }
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

template <int QT, int EPI, int BN, int RM, bool EX = false>
int launch_cfg(const void* W, const void* Wu, int n, int k, const void* Xa, const void* Xb, int T, float* Y,
               const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len, int nsplit = 1,
               float* ws = nullptr, unsigned long long* tickets = nullptr, unsigned epoch = 0) {
  using C = Cfg<QT, EPI, BN, RM, EX>;
  auto fn = encode_fn(msg, msg_len);
  if (!fn) return -1;
  CUtensorMap mW, mWu;
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
  // B operand: fp16 X (f16 leg) or the fp32 hi and lo parts of X (exact leg),
  // 128-byte rows of a BK-column stage, swizzled
  CUtensorMap mX, mX2;
  const CUtensorMapDataType xt = C::EX ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t xrow = (uint64_t)k * (C::EX ? 4 : 2);
  if (!make_map_2d(fn, &mX, xt, Xa, (uint64_t)k, (uint64_t)T, xrow, C::BK, BN, CU_TENSOR_MAP_SWIZZLE_128B, msg,
                   msg_len))
    return -1;
  mX2 = mX;
  if (C::EX && !make_map_2d(fn, &mX2, xt, Xb, (uint64_t)k, (uint64_t)T, xrow, C::BK, BN, CU_TENSOR_MAP_SWIZZLE_128B,
                            msg, msg_len))
    return -1;
  CUtensorMap mR = mX;
  if (C::RM != kRNone) {  // residual [T][n] f32, box 128 rows x BN tokens
    if (!make_map_2d(fn, &mR, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, R, (uint64_t)n, (uint64_t)T, (uint64_t)n * 4, BM, BN,
                     CU_TENSOR_MAP_SWIZZLE_NONE, msg, msg_len))
      return -1;
  }

  auto kern = gemm_tc_kernel<QT, EPI, BN, RM, EX>;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + BM - 1) / BM, (T + BN - 1) / BN, nsplit);
  cfg.blockDim = dim3(C::NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  // may start while the preceding kernel (the conversion of X) finishes; only
  // the X producer waits for it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mW, mWu, mX, mX2, mR, n, k, T, Y, R, status, ws, tickets, epoch);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, msg_len, "gemm_tc launch: %s", cudaGetErrorString(e));
    return -1;
  }
  return 0;
}

int num_sms() {
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return sms[dev] > 0 ? sms[dev] : 148;
}

template <int QT>
int launch_q(const GemmPlan& pl, const void* W, const void* Wu, int n, int k, const uint16_t* X16, int T, float* Y,
             const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len, float* ws,
             unsigned long long* tickets, unsigned epoch) {
  if (Wu) return launch_cfg<QT, kEpiSwiGLU, 128, kRNone>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len);
  // The residual tile goes through TMA when a row of R is a multiple of 16 bytes.
  const bool rtma = R && (n % 4) == 0;
  if (pl.bn == 256) {
    if (rtma)
      return launch_cfg<QT, kEpiResidual, 256, kRLate>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len,
                                                       pl.nsplit, ws, tickets, epoch);
    if (R)
      return launch_cfg<QT, kEpiResidual, 256, kRNone>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len,
                                                       pl.nsplit, ws, tickets, epoch);
    return launch_cfg<QT, kEpiPlain, 256, kRNone>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len,
                                                  pl.nsplit, ws, tickets, epoch);
  }
  if (rtma) return launch_cfg<QT, kEpiResidual, 128, kREarly>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len);
  if (R) return launch_cfg<QT, kEpiResidual, 128, kRNone>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len);
  return launch_cfg<QT, kEpiPlain, 128, kRNone>(W, Wu, n, k, X16, nullptr, T, Y, R, status, s, msg, msg_len);
}

}  // namespace

cudaError_t launch_x_to_f16(const float* X, uint16_t* X16, size_t count, cudaStream_t s) {
  size_t blocks = (count / 8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) blocks = 1;
  x_to_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(X, X16, count);
  return cudaGetLastError();
}

template <int QT>
int launch_q_exact(const void* W, const void* Wu, int n, int k, const float* Xhi, const float* Xlo, int T, float* Y,
                   const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  if (Wu)
    return launch_cfg<QT, kEpiSwiGLU, 128, kRNone, true>(W, Wu, n, k, Xhi, Xlo, T, Y, R, status, s, msg, msg_len);
  if (R && (n % 4) == 0)
    return launch_cfg<QT, kEpiResidual, 128, kRLate, true>(W, Wu, n, k, Xhi, Xlo, T, Y, R, status, s, msg, msg_len);
  if (R) return launch_cfg<QT, kEpiResidual, 128, kRNone, true>(W, Wu, n, k, Xhi, Xlo, T, Y, R, status, s, msg, msg_len);
  return launch_cfg<QT, kEpiPlain, 128, kRNone, true>(W, Wu, n, k, Xhi, Xlo, T, Y, R, status, s, msg, msg_len);
}

GemmPlan plan_gemm_tc(int n, int k, int T, bool swiglu, bool allow_split) {
  GemmPlan pl;
  if (swiglu) return pl;  // 128-token tiles, two accumulators fill TMEM
  const int sms = num_sms();
  const long tiles256 = (long)((n + BM - 1) / BM) * ((T + 255) / 256);
  // 256-token tiles halve the MMA instructions per flop (the single issuing
  // thread, not the tensor core, limits 128-token tiles): taken when they
  // still keep most SMs busy, or, split over k in two, fit in one wave
  if (10 * tiles256 >= 6L * sms) {
    pl.bn = 256;
  } else if (allow_split && 2 * tiles256 <= sms && k / CHUNK >= 2) {
    pl.bn = 256;
    pl.nsplit = 2;
    // fp32 partial tiles, then per tile a ticket word and a ready flag
    pl.ws_bytes = (size_t)tiles256 * 256 * BM * 4 + (size_t)tiles256 * 16;
  }
  return pl;
}

int launch_gemm_tc(const GemmPlan& pl, int qtype, const void* W, const void* Wu, int n, int k, const uint16_t* X16,
                   int T, float* Y, const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len,
                   void* ws) {
  static std::atomic<unsigned> next_epoch{1};
  unsigned epoch = 0;
  float* partials = nullptr;
  unsigned long long* tickets = nullptr;
  if (pl.nsplit > 1) {
    if (!ws) {
      snprintf(msg, msg_len, "split-K GEMM without a workspace");
      return -1;
    }
    epoch = next_epoch.fetch_add(1);
    if (epoch == 0) epoch = next_epoch.fetch_add(1);
    const size_t ntiles = pl.ws_bytes / ((size_t)pl.bn * BM * 4 + 16);
    partials = static_cast<float*>(ws);
    tickets = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + ntiles * (size_t)pl.bn * BM * 4);
  }
  return qtype == kQ4_0
             ? launch_q<kQ4_0>(pl, W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len, partials, tickets, epoch)
             : launch_q<kQ8_0>(pl, W, Wu, n, k, X16, T, Y, R, status, s, msg, msg_len, partials, tickets, epoch);
}

int launch_gemm_tc_exact(int qtype, const void* W, const void* Wu, int n, int k, const float* Xhi, const float* Xlo,
                         int T, float* Y, const float* R, unsigned* status, cudaStream_t s, char* msg,
                         size_t msg_len) {
  return qtype == kQ4_0 ? launch_q_exact<kQ4_0>(W, Wu, n, k, Xhi, Xlo, T, Y, R, status, s, msg, msg_len)
                        : launch_q_exact<kQ8_0>(W, Wu, n, k, Xhi, Xlo, T, Y, R, status, s, msg, msg_len);
}

cudaError_t launch_x_split(const float* X, float* hi, float* lo, size_t count, cudaStream_t s) {
  size_t blocks = (count + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) blocks = 1;
  x_split_kernel<<<(unsigned)blocks, 256, 0, s>>>(X, hi, lo, count);
  return cudaGetLastError();
}

}  // namespace apr
