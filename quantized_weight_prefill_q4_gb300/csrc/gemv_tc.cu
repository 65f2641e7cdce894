// Small-T GEMV (2 <= T <= 4 tokens) over Q4_0 / Q8_0 blocks on the tensor cores,
// exact to fp32 level, sm_103a (tcgen05 + TMA).
//
//   Y[t][i] = sum_b d[i][b] * sum_{j in block b} q[i][j] * X[t][j]   (+ R[t][i])
//
// This computes what the single-token GEMVs gemv_q4_0_pf / gemv_q8_0_pf of
// oxibonsai-kernels 0.1.4 (src/gpu_backend/cuda_q_std_prefill.rs) compute,
// and what the CUDA-core GEMV kernels of this library compute with FFMA, but
// with the per-element work cut to the decode: every product runs on the
// tensor cores, and none of them is rounded.
//
// * A operand (TMEM): the block codes as fp16 integers, q = nibble - 8 (Q4_0)
//   or the int8 (Q8_0). Both are exact in fp16. The fp16 scale d is not
//   applied here; it is applied in fp32 after the MMA, block by block.
// * B operand (shared memory): X split into three fp16 pieces, hi + mid + lo =
//   x * 2^s with hi = fp16(x 2^s), mid = fp16(x 2^s - hi), lo = fp16(x 2^s -
//   hi - mid). The power of two 2^s is chosen per token and 64-column group
//   so that the group's largest |x 2^s| lies in [2^14, 2^15): the pieces then
//   carry 33 significant bits, which covers the 24 of an fp32 x (only
//   elements more than 2^6 below the group's largest lose bits, all below
//   2^-39 of it). Each product q * piece has at most 15 significant bits:
//   exact in the fp32 accumulator. The B builder and the readback each find
//   the group's largest |x| from the same 64 values, so they agree on 2^s.
// * One MMA per 16 columns (M = 128 weight rows, N = 16, K = 16). The rows of
//   B are laid out so that each 32-column block b lands in its own TMEM
//   accumulator columns: row (b mod G) * RB + 3 t + c of B holds piece c of
//   token t in the columns of blocks b' with b' mod G = b mod G and zero in
//   the others, so the G blocks that share one MMA's 16 accumulator columns
//   never mix. The accumulators hold one block partial P[b][t][c] each; the
//   tensor core adds at most 2 G products of 16 terms per partial.
// * Readback (fp32, FFMA): y[t] += 2^-s * sum_b d[b] * ((P[b][t][0] +
//   P[b][t][1]) + P[b][t][2]), b over the group's two blocks.
//
// Cost: each chunk takes 16 MMAs whose A tile (128 x 256 fp16) is read from
// TMEM once; measured on GB300 that is about 800 cycles a chunk, which a Q4_0
// weight streams in about 850. Against the CUDA-core GEMV (gemv_rows.cu /
// gemv_bulk.cu, whose FFMA work grows with T) this kernel wins for T >= 3,
// and for T = 2 on large weights; the dispatch (gemv_tc_takes) says which.
//
// Work split: the weight is cut into 128-row tiles x 256-column chunks; the
// grid (one CTA per SM) takes the chunks in tile-major order, each CTA a
// contiguous range, so that every SM streams the same number of bytes. A tile
// whose chunks span several CTAs is finished by whichever of its contributors
// arrives last at the tile's ticket counter: each contributor writes its
// partial sums to a workspace and takes a ticket; the last one adds the
// partials in a fixed order (by contributor), so the result does not depend
// on arrival order, and clears the counter for the next call. Nothing ever
// waits on another CTA.
//
// Warp roles (640 threads):
//   warp 0   TMA producer of raw weight chunks (128 rows x 256 columns: 144 /
//            272 bytes a row) into a ring, with L2 prefetches ahead
//   warp 1   TMEM allocator and MMA issuer (whole warp, one elected lane)
//   warp 2   B builder: X's pieces for each chunk (X fetched three chunks
//            ahead with cp.async), written into a ring of 128-byte-swizzled
//            B tiles (16 rows x 256 columns of fp16)
//   warp 3   publisher: at the end of each of the CTA's shares of a tile it
//            adds the warpgroups' sums, publishes them, takes the ticket and
//            finishes the tile if it is the last contributor
//   warps 4..19  four decode warpgroups: warpgroup w owns blocks 2w, 2w + 1
//            of every chunk; each thread one weight row (its TMEM lane). It
//            decodes chunk j + 2 into an A slot while the MMAs of chunk j + 1
//            run and chunk j's partials come out of TMEM, then accumulates
//            chunk j. At the end of a share it hands its sums to the
//            publisher through shared memory and goes on.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the device
// status word and an abort flag so that every role leaves its loop, drains its
// copies and MMAs, and the CTA frees its TMEM.
//
// Programmatic dependent launch: the kernel streams W at once (W must not be
// written by the kernel before it, which may still be running); every other
// access to global memory (X, R, Y, the counters and partial sums) waits for
// griddepcontrol.wait. Each CTA lets the next kernel launch only after that
// wait, so at most the one kernel before runs alongside.

#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"
#include "host_common.h"

namespace apr {
namespace {

constexpr int BM = 128;                   // weight rows per tile (MMA M)
constexpr int CHUNK = 256;                // columns per raw chunk
constexpr int NB = CHUNK / 32;            // blocks per chunk
constexpr int NDQ = 4;                    // decode warpgroups, two blocks each
constexpr int BROWS = 16;                 // rows of a B tile (MMA N)
constexpr int B_SUB = BROWS * 128;        // one 64-column swizzled sub-tile
constexpr int B_BYTES = 4 * B_SUB;        // B for one chunk
constexpr int A_COLS = CHUNK / 2;         // TMEM columns of one chunk of A
constexpr int NTHREADS = 128 + 128 * NDQ;
constexpr int PF = 4;                     // raw chunks prefetched into L2 ahead

template <int QT, int TMAX>
struct VCfg {
  static constexpr int BB = QT == kQ4_0 ? 18 : 34;
  static constexpr int RAW_ROW = NB * BB;
  static constexpr int RAW_BYTES = BM * RAW_ROW;
  // B rows per block (3 pieces a token, rounded up to a power of two) and
  // the blocks G that share one MMA's 16 accumulator columns
  static constexpr int RB = 3 * TMAX <= 4 ? 4 : (3 * TMAX <= 8 ? 8 : 16);
  static constexpr int G = BROWS / RB;
  static constexpr int D_COLS = NB * RB;                 // accumulator columns of one chunk
  static constexpr int SLOT_COLS = A_COLS + D_COLS;      // one A + D slot in TMEM
  static constexpr int S = 512 / SLOT_COLS >= 3 ? 3 : 2;
  static constexpr int S_RAW = QT == kQ4_0 ? 6 : 4;
  static constexpr int S_B = 4;
  static constexpr int S_X = 4;                          // chunks of X the builder fetches ahead
  static constexpr int OFF_RAW = 0;
  static constexpr int OFF_B = OFF_RAW + S_RAW * RAW_BYTES;
  static constexpr int OFF_RED = OFF_B + S_B * B_BYTES;        // warpgroup sums, [NDQ][TMAX][128]
  static constexpr int OFF_X = OFF_RED + NDQ * TMAX * BM * 4;   // X ring of the builder, [S_X][TMAX][256]
  static constexpr int OFF_BAR = OFF_X + S_X * TMAX * CHUNK * 4;
  static constexpr int NBAR = 2 * S_RAW + 2 * S_B + 3 * S + 1 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;      // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(S * SLOT_COLS <= 512, "TMEM budget");
  static_assert(3 * TMAX <= RB && NB % G == 0, "B row layout");
  static_assert(RAW_BYTES % 1024 == 0 && OFF_B % 1024 == 0, "swizzled B tiles start on 1024 bytes");
};

// ---------------------------------------------------------------- decode
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Q4_0 payload word p (bytes b0..b3: low nibbles = elements e..e+3, high
// nibbles = e+16..e+19) -> four fp16 pairs of (nibble - 8), in k order:
// o[0] = (e, e+1), o[1] = (e+2, e+3), o[2] = (e+16, e+17), o[3] = (e+18, e+19).
//   (0x6400 | n) is the fp16 1024 + n; minus 1032 gives n - 8 exactly.
//   (0x6400 | 16 n) is 1024 + 16 n; times 1/16 minus 72 gives n - 8 exactly.
__device__ __forceinline__ void q4_codes(uint32_t p, uint32_t (&o)[4]) {
  const uint32_t lo01 = __byte_perm(p, 0u, 0x4140);
  const uint32_t lo23 = __byte_perm(p, 0u, 0x4342);
  const __half2 k1032 = bits_h2(0x64086408u);
  const __half2 k16th = bits_h2(0x2C002C00u);
  const __half2 km72 = bits_h2(0xD480D480u);
  o[0] = h2_bits(__hsub2(bits_h2((lo01 & 0x000F000Fu) | 0x64006400u), k1032));
  o[1] = h2_bits(__hsub2(bits_h2((lo23 & 0x000F000Fu) | 0x64006400u), k1032));
  o[2] = h2_bits(__hfma2(bits_h2((lo01 & 0x00F000F0u) | 0x64006400u), k16th, km72));
  o[3] = h2_bits(__hfma2(bits_h2((lo23 & 0x00F000F0u) | 0x64006400u), k16th, km72));
}

// Q8_0 payload word q (4 int8, elements e..e+3) -> fp16 pairs (e, e+1),
// (e+2, e+3) of the int8 values: (0x6400 | (b ^ 0x80)) is 1024 + b + 128.
__device__ __forceinline__ void q8_codes(uint32_t q, uint32_t (&o)[2]) {
  const uint32_t x = q ^ 0x80808080u;
  const __half2 k1152 = bits_h2(0x64806480u);
  o[0] = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x5140)), k1152));
  o[1] = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x7362)), k1152));
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)w)); }
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// Two Q4_0 blocks (36 bytes) starting at word O of v: a[0..31] = fp16 pairs of
// codes in k order (block 0 then block 1), d[] = the blocks' scales.
template <int O>
__device__ __forceinline__ void decode_q4(const uint32_t (&v)[12], uint32_t (&a)[32], float (&d)[2]) {
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __byte_perm(v[O + i], v[O + i + 1], 0x5432);  // payload of block 0
#pragma unroll
  for (int i = 0; i < 4; ++i) p[4 + i] = v[O + 5 + i];                              // payload of block 1
  d[0] = half_lo(v[O]);
  d[1] = half_hi(v[O + 4]);
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t o[4];
      q4_codes(p[blk * 4 + i], o);
      a[16 * blk + 2 * i] = o[0];
      a[16 * blk + 2 * i + 1] = o[1];
      a[16 * blk + 8 + 2 * i] = o[2];
      a[16 * blk + 8 + 2 * i + 1] = o[3];
    }
  }
}

// Two Q8_0 blocks (68 bytes) starting at word O of v.
template <int O>
__device__ __forceinline__ void decode_q8(const uint32_t (&v)[20], uint32_t (&a)[32], float (&d)[2]) {
  d[0] = half_lo(v[O]);
  d[1] = half_hi(v[O + 8]);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t p = c < 8 ? __byte_perm(v[O + c], v[O + c + 1], 0x5432) : v[O + 1 + c];
    uint32_t o[2];
    q8_codes(p, o);
    a[2 * c] = o[0];
    a[2 * c + 1] = o[1];
  }
}

// Warpgroup w's two blocks of this thread's row of a raw chunk. The row
// starts on 16 bytes; the blocks start 36 w (Q4_0) or 68 w (Q8_0) bytes in,
// i.e. w words past the 16-byte boundary below them, which is read with
// 16-byte loads (conflict-free: rows are 144 / 272 bytes apart).
template <int QT>
__device__ __forceinline__ void decode_pair(const uint8_t* row, int w, uint32_t (&a)[32], float (&d)[2]) {
  if constexpr (QT == kQ4_0) {
    const uint4* s = reinterpret_cast<const uint4*>(row + ((36 * w) & ~15));
    uint32_t v[12];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint4 u = s[i];
      v[4 * i] = u.x;
      v[4 * i + 1] = u.y;
      v[4 * i + 2] = u.z;
      v[4 * i + 3] = u.w;
    }
    switch (w) {
      case 0: decode_q4<0>(v, a, d); break;
      case 1: decode_q4<1>(v, a, d); break;
      case 2: decode_q4<2>(v, a, d); break;
      default: decode_q4<3>(v, a, d); break;
    }
  } else {
    const uint4* s = reinterpret_cast<const uint4*>(row + ((68 * w) & ~15));
    uint32_t v[20];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const uint4 u = s[i];
      v[4 * i] = u.x;
      v[4 * i + 1] = u.y;
      v[4 * i + 2] = u.z;
      v[4 * i + 3] = u.w;
    }
    switch (w) {
      case 0: decode_q8<0>(v, a, d); break;
      case 1: decode_q8<1>(v, a, d); break;
      case 2: decode_q8<2>(v, a, d); break;
      default: decode_q8<3>(v, a, d); break;
    }
  }
}

// 32 lanes x NC consecutive 32-bit TMEM columns into v (valid after the wait).
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[NC]) {
  static_assert(NC == 8 || NC == 16 || NC == 32, "load width");
  if constexpr (NC == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (NC == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
  } else {
    tmem_ld_32x32b_x32(taddr, v);
  }
}

// Waits for this thread's TMEM loads, tying the NC registers to the wait.
template <int NC>
__device__ __forceinline__ void tmem_ld_wait_cols(uint32_t (&v)[NC]) {
  if constexpr (NC == 32) {
    tmem_ld_wait_regs(v);
  } else {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < NC; ++i) asm volatile("" : "+r"(v[i]) : : "memory");
  }
}

// The power of two that X's pieces of one 64-column group are scaled by: 2^e
// with the group's largest |x| times 2^e in [2^14, 2^15) (for a subnormal
// largest |x|, 2^100), or 1 for an all-zero or non-finite group (NaN and Inf
// then propagate). `inverse` gives 2^-e. The
// B builder and the readback compute it from the same 64 values.
__device__ __forceinline__ float group_scale(float m, bool inverse) {
  int e = 0;
  if (m > 0.f && m <= 3.402823466e38f) {
    e = 14 - (((__float_as_int(m) >> 23) & 0xFF) - 127);  // floor(log2 m) for a normal m
    e = e < -100 ? -100 : (e > 100 ? 100 : e);
  }
  return __int_as_float((127 + (inverse ? -e : e)) << 23);
}

// Ticket: atomic add with acquire-release semantics at GPU scope. With the
// warp barrier before it, the partial sums the warp wrote are visible to
// whichever warp draws the last ticket; with the barrier after it, that warp
// sees every other contributor's.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// CTA that owns chunk u when `total` chunks are cut into G contiguous ranges
// [floor(g total / G), floor((g + 1) total / G)).
__device__ __forceinline__ int chunk_owner(long u, long total, int G) {
  return (int)(((u + 1) * G + total - 1) / total) - 1;
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only) and its
// group bookkeeping.
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- kernel
template <int QT, int TMAX>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmW, int n, int k, const float* __restrict__ X, int T,
                   float* Y, int ldy, const float* R, float* ws, unsigned* cnt, unsigned* status) {
  using C = VCfg<QT, TMAX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sRaw = smem + C::OFF_RAW;
  uint8_t* sB = smem + C::OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* rawFull = bars;
  uint64_t* rawEmpty = rawFull + C::S_RAW;
  uint64_t* bFull = rawEmpty + C::S_RAW;
  uint64_t* bEmpty = bFull + C::S_B;
  uint64_t* aFull = bEmpty + C::S_B;   // A slot written by every decode warp
  uint64_t* dFull = aFull + C::S;      // the slot's MMAs completed
  uint64_t* dFree = dFull + C::S;      // the slot's accumulators read back
  uint64_t* drain = dFree + C::S;
  uint64_t* redFull = drain + 1;       // a tile's partial sums of every warpgroup written
  uint64_t* redFree = redFull + 1;     // ... and read by the publisher
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cpt = k / CHUNK;                       // chunks per tile
  const long total = (long)((n + BM - 1) / BM) * cpt;
  const int G = gridDim.x, g = blockIdx.x;
  const long ua = (long)g * total / G;
  const int nu = (int)((long)(g + 1) * total / G - ua);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S_RAW; ++i) {
      mbar_init(&rawFull[i], 1);
      mbar_init(&rawEmpty[i], 4 * NDQ);
    }
    for (int i = 0; i < C::S_B; ++i) {
      mbar_init(&bFull[i], 1);
      mbar_init(&bEmpty[i], 1);
    }
    for (int i = 0; i < C::S; ++i) {
      mbar_init(&aFull[i], 4 * NDQ);
      mbar_init(&dFull[i], 1);
      mbar_init(&dFree[i], 4 * NDQ);
    }
    mbar_init(drain, 1);
    mbar_init(redFull, 4 * NDQ);
    mbar_init(redFree, 1);
    abort_flag[0] = 0;   // set by a wait that gives up
    abort_flag[1] = 0;   // never set: drain waits ignore the abort
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------ raw weight producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      for (int i = 0; i < PF && i < nu; ++i) {
        const long u = ua + i;
        tma_prefetch_l2_2d(&tmW, (int)(u % cpt) * (C::RAW_ROW / 2), (int)(u / cpt) * BM);
      }
      int last[C::S_RAW];
      for (int i = 0; i < C::S_RAW; ++i) last[i] = -1;
      bool ok = true;
      for (int i = 0; i < nu; ++i) {
        const int slot = i % C::S_RAW;
        ok = mbar_wait(&rawEmpty[slot], ((i / C::S_RAW) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        const long u = ua + i;
        mbar_arrive_expect_tx(&rawFull[slot], C::RAW_BYTES);
        tma_load_2d(sRaw + slot * C::RAW_BYTES, &tmW, (int)(u % cpt) * (C::RAW_ROW / 2), (int)(u / cpt) * BM,
                    &rawFull[slot]);
        if (i + PF < nu)
          tma_prefetch_l2_2d(&tmW, (int)((u + PF) % cpt) * (C::RAW_ROW / 2), (int)((u + PF) / cpt) * BM);
        last[slot] = i;
      }
      if (!ok)  // let the copies in flight land before the CTA exits
        for (int i = 0; i < C::S_RAW; ++i)
          if (last[i] >= 0) mbar_wait(&rawFull[i], (last[i] / C::S_RAW) & 1, abort_flag + 1, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ B builder (whole warp)
    // Lane L takes columns 8 L .. 8 L + 7 of the chunk (block L / 4, 16 bytes
    // of one 128-byte row of sub-tile L / 8) and writes its pieces into rows
    // (block mod G) * RB + 3 t + c. Every other element of the ring is zero
    // and stays zero. Lanes 8 j .. 8 j + 7 hold the 64-column group j whose
    // largest |x| sets the group's power of two.
    for (int o = lane * 16; o < C::S_B * B_BYTES; o += 32 * 16)
      *reinterpret_cast<uint4*>(sB + o) = make_uint4(0u, 0u, 0u, 0u);
    grid_dependency_wait();                  // X may be written by the kernel before
    if (lane == 0) grid_launch_dependents();
    const int blk = lane >> 2, sub = lane >> 3, c16 = lane & 7;
    const int hh = blk % C::G;
    // each lane fetches its own 8 columns of every token S_X - 1 chunks ahead
    // (cp.async into the X ring; a lane reads only what it fetched itself)
    float* xring = reinterpret_cast<float*>(smem + C::OFF_X);
    auto fetch = [&](int i) {
      if (i < nu) {
        const int col = (int)((ua + i) % cpt) * CHUNK + 8 * lane;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t >= T) continue;
          float* dst = xring + ((i % C::S_X) * TMAX + t) * CHUNK + 8 * lane;
          cp_async_16(dst, X + (size_t)t * k + col);
          cp_async_16(dst + 4, X + (size_t)t * k + col + 4);
        }
      }
      cp_async_commit();
    };
    for (int i = 0; i < C::S_X - 1; ++i) fetch(i);
    bool ok = true;
    for (int i = 0; i < nu; ++i) {
      fetch(i + C::S_X - 1);
      cp_async_wait<C::S_X - 1>();  // chunk i's columns have landed
      const int sb = i % C::S_B;
      ok = __all_sync(0xffffffffu, mbar_wait(&bEmpty[sb], ((i / C::S_B) & 1) ^ 1, abort_flag, status));
      if (!ok) break;
      uint8_t* tile = sB + sb * B_BYTES + sub * B_SUB;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t >= T) continue;
        const float4* x4 = reinterpret_cast<const float4*>(xring + ((i % C::S_X) * TMAX + t) * CHUNK + 8 * lane);
        const float4 v0 = x4[0], v1 = x4[1];
        const float xs[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(xs[e]));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float sc = group_scale(m, false);
        uint32_t pw[3][4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          float hv[2], mv[2], lv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float x = xs[e + u] * sc;
            const float h = __half2float(__float2half_rn(x));
            const float r1 = x - h;
            const float md = __half2float(__float2half_rn(r1));
            hv[u] = h;
            mv[u] = md;
            lv[u] = r1 - md;
          }
          pw[0][e / 2] = h2_bits(__floats2half2_rn(hv[0], hv[1]));
          pw[1][e / 2] = h2_bits(__floats2half2_rn(mv[0], mv[1]));
          pw[2][e / 2] = h2_bits(__floats2half2_rn(lv[0], lv[1]));
        }
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const int row = hh * C::RB + 3 * t + c;
          *reinterpret_cast<uint4*>(tile + row * 128 + ((c16 ^ (row & 7)) << 4)) =
              make_uint4(pw[c][0], pw[c][1], pw[c][2], pw[c][3]);
        }
      }
      fence_proxy_async_smem();  // the tensor core reads B through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&bFull[sb]);
    }
    cp_async_wait<0>();  // no copy into shared memory outlives the loop
  } else if (warp == 3) {
    // ------------------------------------------------ publisher (whole warp)
    // At the end of each of this CTA's shares of a tile: add the warpgroups'
    // sums (lane L takes rows L, L + 32, L + 64, L + 96), write the share to
    // the workspace, take the tile's ticket, and if it is the last one, add
    // every contributor's share in contributor order and write Y.
    grid_dependency_wait();  // the workspace, counters, R and Y may be in use before
    int f = 0;
    for (int j = 0; j < nu; ++j) {
      const long u = ua + j;
      if ((u + 1) % cpt != 0 && j + 1 != nu) continue;
      const int m = (int)(u / cpt);
      if (!__all_sync(0xffffffffu, mbar_wait(redFull, f & 1, abort_flag, status))) break;
      float* mine = ws + (size_t)(m + g) * TMAX * BM;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int row = rr * 32 + lane;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < NDQ; ++w) v += red[(w * TMAX + t) * BM + row];
          __stcg(mine + t * BM + row, v);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(redFree);
      unsigned prev = 0;
      if (lane == 0) prev = atomic_add_acq_rel(&cnt[m], 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      __syncwarp();
      const int g0 = chunk_owner((long)m * cpt, total, G), g1 = chunk_owner((long)m * cpt + cpt - 1, total, G);
      if (prev == (unsigned)(g1 - g0)) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int r = rr * 32 + lane;
          float y[TMAX];
#pragma unroll
          for (int t = 0; t < TMAX; ++t) y[t] = 0.f;
          for (int gb = g0; gb <= g1; gb += 8) {
            float pv[8][TMAX];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
#pragma unroll
              for (int t = 0; t < TMAX; ++t)
                pv[jj][t] = gb + jj <= g1 ? __ldcg(ws + ((size_t)(m + gb + jj) * TMAX + t) * BM + r) : 0.f;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
#pragma unroll
              for (int t = 0; t < TMAX; ++t)
                if (gb + jj <= g1) y[t] += pv[jj][t];
          }
          const int row = m * BM + r;
          if (row < n) {
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              if (t < T) {
                const size_t o = (size_t)t * ldy + row;
                Y[o] = R ? y[t] + R[o] : y[t];
              }
            }
          }
        }
        // every contributor has drawn its ticket: clear the counter for the
        // next call on this scratch
        if (lane == 0) cnt[m] = 0u;
      }
      ++f;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t idesc = idesc_f16_f32(BM, BROWS);
    bool ok = true;
    for (int i = 0; i < nu; ++i) {
      const int sa = i % C::S, sb = i % C::S_B;
      ok = __all_sync(0xffffffffu, mbar_wait(&aFull[sa], (i / C::S) & 1, abort_flag, status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bFull[sb], (i / C::S_B) & 1, abort_flag, status));
      // the slot's accumulators of chunk i - S have been read back
      if (ok && i >= C::S)
        ok = __all_sync(0xffffffffu, mbar_wait(&dFree[sa], ((i / C::S) - 1) & 1, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      const uint64_t bdesc0 = smem_desc_sw128(sB + sb * B_BYTES);
      const uint32_t a0 = tmem_base + sa * C::SLOT_COLS;
      const uint32_t d0 = a0 + A_COLS;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // block b, columns 16 h.. of it: sub-tile b / 2 of B, 32 bytes per
          // 16 columns inside the swizzle atom; 8 TMEM columns of A
          const uint64_t bdesc = bdesc0 + (uint64_t)(((b >> 1) * B_SUB + ((b & 1) * 2 + h) * 32) >> 4);
          mma_f16_ts_elect(d0 + (b / C::G) * BROWS, a0 + b * 16 + h * 8, bdesc, idesc,
                           (b % C::G != 0 || h != 0) ? 1u : 0u);
        }
      }
      mma_commit_elect(&bEmpty[sb]);
      mma_commit_elect(&dFull[sa]);
    }
    if (!ok) {  // wait until the MMAs already issued have finished
      mma_commit_elect(drain);
      __all_sync(0xffffffffu, mbar_wait(drain, 0, abort_flag + 1, status));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ decode, readback, finish
    const int wg = (warp - 4) >> 2;                  // blocks 2 wg, 2 wg + 1 of every chunk
    const uint32_t q = (uint32_t)(warp & 3);         // lane quarter of TMEM this warp may access
    const uint32_t r = q * 32 + lane;                // tile row == TMEM lane
    const uint32_t lane_base = tmem_base + ((q * 32u) << 16);
    constexpr int NC = 2 * C::RB;                    // accumulator columns of this warpgroup's two blocks
    bool ok = true;

    // decode chunk i into A slot i % S (free: the MMAs of chunk i - S have
    // completed, which this warp has seen)
    auto produce = [&](int i, float (&d)[2]) -> bool {
      const int slot = i % C::S_RAW;
      if (!__all_sync(0xffffffffu, mbar_wait(&rawFull[slot], (i / C::S_RAW) & 1, abort_flag, status)))
        return false;
      uint32_t a[32];
      decode_pair<QT>(sRaw + slot * C::RAW_BYTES + r * C::RAW_ROW, wg, a, d);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rawEmpty[slot]);
      tc_fence_after();
      tmem_st_32x32b_x32(lane_base + (i % C::S) * C::SLOT_COLS + 32 * wg, a);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aFull[i % C::S]);
      return true;
    };

    float acc[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
    // block scales of chunks j, j + 1, j + 2; this warpgroup's 64 columns of
    // X in chunks j and j + 1 (two per lane), whose largest |x| gives the
    // power of two the builder scaled them by
    float dA[2] = {0.f, 0.f}, dB[2] = {0.f, 0.f}, dC[2] = {0.f, 0.f};
    float2 xA[TMAX], xB[TMAX];
    auto load_x = [&](int j, float2 (&xv)[TMAX]) {
      const int col = (int)((ua + j) % cpt) * CHUNK + 64 * wg + 2 * lane;
#pragma unroll
      for (int t = 0; t < TMAX; ++t)
        xv[t] = t < T ? __ldcg(reinterpret_cast<const float2*>(X + (size_t)t * k + col)) : make_float2(0.f, 0.f);
    };
    int nflush = 0;
    if (nu > 0) ok = produce(0, dA);
    if (ok && nu > 1) ok = produce(1, dB);
    // Iteration j reads back chunk j and decodes chunk j + 2: the TMEM load
    // of chunk j is issued first and awaited after the decode, and the MMAs
    // of chunk j + 1 run meanwhile. (The load's registers stay untouched in
    // between: nothing else in the iteration assigns them.)
    for (int j = 0; j < nu && ok; ++j) {
      const int sa = j % C::S;
      ok = __all_sync(0xffffffffu, mbar_wait(&dFull[sa], (j / C::S) & 1, abort_flag, status));
      if (!ok) break;
      if (j == 0) {
        grid_dependency_wait();  // X may be written by the kernel before
        load_x(0, xA);
      }
      if (j + 1 < nu) load_x(j + 1, xB);
      tc_fence_after();
      uint32_t v[NC];
      tmem_ld_cols<NC>(lane_base + sa * C::SLOT_COLS + A_COLS + 2 * wg * C::RB, v);
      if (j + 2 < nu) ok = produce(j + 2, dC);
      tmem_ld_wait_cols<NC>(v);
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dFree[sa]);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        float mx = fmaxf(fabsf(xA[t].x), fabsf(xA[t].y));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float part = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c0 = h * C::RB + 3 * t;
          const float p = (__uint_as_float(v[c0]) + __uint_as_float(v[c0 + 1])) + __uint_as_float(v[c0 + 2]);
          part = fmaf(dA[h], p, part);
        }
        acc[t] = fmaf(part, group_scale(mx, true), acc[t]);
        xA[t] = xB[t];
      }
      dA[0] = dB[0];
      dA[1] = dB[1];
      dB[0] = dC[0];
      dB[1] = dC[1];

      const long u = ua + j;
      if ((u + 1) % cpt != 0 && j + 1 != nu) continue;
      // this CTA's share of a tile is complete: hand the warpgroup's sums to
      // the publisher (once it has read the previous share)
      if (nflush > 0) ok = __all_sync(0xffffffffu, mbar_wait(redFree, (nflush - 1) & 1, abort_flag, status));
      if (!ok) break;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        red[(wg * TMAX + t) * BM + r] = acc[t];
        acc[t] = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(redFull);
      ++nflush;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------- host side
// Scratch of a call: a fixed region of ticket counters (one per tile, at most
// kCounters; zero before the first call, and every completed call leaves
// them zero) followed by the partial sums (one slot per (tile, contributor)
// pair: tile m and CTA g use slot m + g, which is unique because a tile's
// contributors are consecutive CTAs and a later tile never starts before an
// earlier tile's last contributor). The counters never move, so calls of any
// shape can share the scratch.
constexpr int kCounters = 16384;

int grid_size(int n, int k) {
  const long total = (long)((n + BM - 1) / BM) * (k / CHUNK);
  const int sms = num_sms();
  return total < sms ? (int)total : sms;
}

size_t scratch_bytes(int n, int k, int tmax) {
  return (size_t)kCounters * 4 + (size_t)((n + BM - 1) / BM + grid_size(n, k)) * tmax * BM * 4;
}

int tmax_of(int T) { return T <= 2 ? 2 : 4; }

template <int QT, int TMAX>
int launch_t(const void* W, int n, int k, const float* X, int T, float* Y, int ldy, const float* R, void* scratch,
             unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  using C = VCfg<QT, TMAX>;
  unsigned* cnt = static_cast<unsigned*>(scratch);
  float* ws = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + (size_t)kCounters * 4);
  auto fn = encode_fn(msg, msg_len);
  if (!fn) return -1;
  CUtensorMap mW;
  const uint64_t row_bytes = (uint64_t)(k / 32) * C::BB;
  if (!make_map_2d(fn, &mW, CU_TENSOR_MAP_DATA_TYPE_UINT16, W, row_bytes / 2, (uint64_t)n, row_bytes,
                   C::RAW_ROW / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE, msg, msg_len))
    return -1;
  auto kern = gemv_tc_kernel<QT, TMAX>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) {
      snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return -1;
    }
    attr_set[dev] = 1;
  }
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_size(n, k));
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mW, n, k, X, T, Y, ldy, R, ws, cnt, status);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, msg_len, "gemv_tc launch: %s", cudaGetErrorString(e));
    return -1;
  }
  return 0;
}

template <int QT>
int launch_q(const void* W, int n, int k, const float* X, int T, float* Y, int ldy, const float* R, void* scratch,
             unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  if (tmax_of(T) == 2) return launch_t<QT, 2>(W, n, k, X, T, Y, ldy, R, scratch, status, s, msg, msg_len);
  return launch_t<QT, 4>(W, n, k, X, T, Y, ldy, R, scratch, status, s, msg, msg_len);
}

}  // namespace

bool gemv_tc_takes(int n, int k, int T, bool swiglu) {
  if (swiglu || n <= 0 || (n + BM - 1) / BM > kCounters || k % CHUNK != 0 || T > kGemvTcMaxT) return false;
  // measured on GB300 (Q4_0 and Q8_0, 4096 x 4096 and 12288 x 4096): the
  // CUDA-core kernels are faster at T = 1, and at T = 2 on weights below
  // 2^25 elements
  return T >= 3 || (T == 2 && (long)n * k >= (1L << 25));
}

size_t gemv_tc_scratch_bytes(int n, int k, int T) { return scratch_bytes(n, k, tmax_of(T)); }

int launch_gemv_tc(int qtype, const void* W, int n, int k, const float* X, int T, float* Y, int ldy, const float* R,
                   void* scratch, unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  return qtype == kQ4_0 ? launch_q<kQ4_0>(W, n, k, X, T, Y, ldy, R, scratch, status, s, msg, msg_len)
                        : launch_q<kQ8_0>(W, n, k, X, T, Y, ldy, R, scratch, status, s, msg, msg_len);
}

}  // namespace apr
