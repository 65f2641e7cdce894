// Tensor-core GEMM over Q4_0 / Q8_0 blocks and F16 weights, sm_103a (tcgen05 + TMA):
// the fp16-input leg and, on the same skeleton, the exact-fp32 leg (XS below).
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
// One CTA computes one 128-row x BN-token output tile (BN = 128 or 256), or,
// split over k, half of the k range of one 256-token tile. Warp roles:
//   warp 0       TMA producer of raw weight chunks: 128 rows x 256 k (8 blocks
//                per row: 144 B for Q4_0, 272 B for Q8_0, the smallest box whose
//                width is a multiple of 16 bytes for both formats; F16 rows as
//                four 64-k boxes of [128 rows][128 B], 128-byte swizzled, half
//                a chunk per slot for a gate/up pair) into a ring of S_RAW
//                slots, with L2 prefetches PF slots ahead
//   warp 1       TMEM allocator and MMA issuer: the whole warp runs the loop,
//                one elected lane issues (four K = 16 MMAs per 64-k stage)
//   warp 2       TMA producer of X tiles: BN tokens x 64 k of the fp16 copy of X,
//                128-byte swizzled, into the B ring; a few stages before the
//                end it prefetches the residual pieces the CTA finalizes into L2
//   warp 3       idle
//   warps 4..    dequant warpgroups: each thread owns one of the 128 rows (its
//                TMEM lane), decodes 2 blocks (64 k) per stage from the raw slot
//                (F16: copies its 128 bytes) and stores them as 32 columns of
//                fp16 pairs into an A stage in TMEM; A and B stages advance
//                together (S of them); with one
//                weight, two warpgroups take alternate stages, with gate/up one
//                warpgroup per weight. Then the same warps run the epilogue.
// Epilogue: the tile's token columns go out in pieces of 64. A warpgroup reads
// a piece's accumulators out of TMEM (two 32-column loads, one wait), adds the
// residual (or applies the SiLU gate) in registers and stores Y straight from
// registers: thread r owns weight row r, so each store of a warp writes 32
// consecutive floats of one token's row. The residual of the warpgroup's
// first piece is loaded into registers while the last chunks are still in the
// MMA pipe (after the X producer prefetched it into L2). Nothing of the
// epilogue passes through shared memory except the split partner's half: the
// shared-memory round trips of a TMA residual load and a TMA store of Y cost
// more (the SM's shared-memory bandwidth) than the stores they replace.
// Split over k (two CTAs per tile, blockIdx.z = 0, 1, launched as a cluster
// (1, 1, 2)): CTA z finalizes token columns [128 z, 128 z + 128) of the tile.
// Its weight producer tells the partner when the raw ring is free (the last
// chunk decoded, a little before the last MMAs finish); after its MMAs each
// thread writes its row of the half the partner keeps straight from registers
// into the partner's raw ring (distributed shared memory stores) and arrives
// on the partner's barrier with release semantics; each CTA then adds p0 + p1
// in split order, so the result does not depend on which CTA finishes first.
// A cluster barrier at the end keeps both CTAs resident until neither touches
// the other's shared memory.
// Gate/up as a pair (kEpiGluPair, 256-token tiles): the same cluster of two,
// but CTA z streams and decodes one weight over the whole of k (z = 0 the
// gate, z = 1 the up weight) into its own accumulator, so that each decoded
// weight serves 256 tokens (a single CTA holding both accumulators has TMEM
// for 128 tokens only). The halves are exchanged as above and CTA z computes
// silu(gate) * up for token columns [128 z, 128 z + 128).
// Exact leg (XS): the pages' f32 leg (fp32 products, no reduced-precision
// input) on the same skeleton; see the comment above Cfg.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the device
// status word and an abort flag in shared memory so that every role leaves its
// loop, drains its own TMA copies and MMAs, and the CTA frees its TMEM.
// Programmatic dependent launch: the kernel lets the next kernel of the stream
// launch early. X16, Y and the residual are touched only after
// griddepcontrol.wait. The weights are read before it (`early` != kEarlyNone):
// the library's weights are never the output of the kernel just before (the
// header's stream-order rule), so the first weight chunks stream and decode
// while the preceding kernel finishes. With kEarlyNone everything waits.

#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "apr_internal.h"
#include "dev_common.cuh"
#include "host_common.h"
#include "iq4.cuh"
#include "q4k.cuh"

namespace apr {
namespace {

constexpr int BM = 128;         // weight rows per tile (UMMA M)
constexpr int CHUNK = 256;      // k per raw TMA chunk
constexpr int BK = 64;          // k per operand stage (128 B of fp16 B per token row)
constexpr int SUBS = CHUNK / BK;
constexpr int PF = 4;           // raw chunks prefetched into L2 ahead of their TMA load
constexpr int PIECE = 64;                      // token columns per epilogue piece
constexpr int PIECE_BYTES = PIECE * BM * 4;    // one fp32 piece, [64 tokens][128 rows]

// XS: the exact leg. The weight is split W = W1 + W2 and X = X1 + X2 into
// fp16 pieces (scaled by powers of two per weight row and per token), and
// each 16-k step runs three MMAs, W1.X1 + W1.X2 + W2.X1: NP = 2 pieces of A
// and of B per stage. The tensor core's fp32 accumulator loses about 2e-8 of
// its magnitude per update (measured: 1.35e-5 relative after the 768 updates
// of k = 4096), so each 256-k chunk accumulates afresh, alternately into two
// accumulators, and a decode warpgroup adds every finished chunk into a
// running sum in TMEM with fp32 round-to-nearest additions (acc0, acc1 and
// the sum: three accumulator regions).
template <int QT, int EPI, int BN_, bool XS_ = false>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr bool XS = XS_;
  static constexpr int NP = XS ? 2 : 1;                 // operand pieces
  static constexpr int A_COLS = 32;                     // TMEM columns of one A piece of one stage of one weight
  static constexpr int B_BYTES = BN * 128;              // one 128-B-swizzled B piece of a stage
  static constexpr int NM = EPI == kEpiSwiGLU ? 2 : 1;
  static constexpr int DQ = NM == 1 ? 2 : 1;           // warpgroups per weight (alternate stages)
  static constexpr int NWG = NM * DQ;                   // dequant / epilogue warpgroups
  static constexpr bool F16W = QT == kF16;
  static constexpr bool IQ4 = QT == kIQ4_XS;
  // ring depths of the short-row formats
  static constexpr bool Q4W = QT == kQ4_0 || QT == kQ4_K || QT == kQ5_K || IQ4;
  static constexpr bool Q6K = QT == kQ6_K;
  static constexpr int BB =
      QT == kQ4_0 || QT == kQ4_K ? 18 : (QT == kQ8_0 ? 34 : (QT == kQ5_K ? 22 : (IQ4 ? 17 : 64)));
  // words a decode thread reads per stage: two blocks, or for Q4_K / Q5_K the
  // superblock's header and scales (4 words), Q5_K's fifth-bit bytes (8
  // words) and the stage's 32 code bytes (8 words); for Q6_K the aligned
  // words over the stage's 64 low-nibble bytes, 32 high-bit bytes and 4
  // scales (each one word more: the superblock may start 2 bytes into a
  // word) and the word holding d; for IQ4_XS the header's two words (d and
  // the high scale bits, the low scale nibbles) and the stage's 32 code bytes
  static constexpr int NWORDS = QT == kQ4_K ? 12 : (QT == kQ5_K ? 20 : (Q6K ? 29 : (IQ4 ? 10 : 2 * BB / 4)));
  // k per raw slot: a chunk, or half of one for F16 gate/up (four slots of
  // 32 KB keep each weight double-buffered; a CTA pair's two 32 KB slots
  // beside its 256-token B ring)
  static constexpr int RAW_K = F16W && (NM == 2 || BN == 256) ? CHUNK / 2 : CHUNK;
  static constexpr int RAW_SUBS = RAW_K / BK;         // operand stages per raw slot
  // 144 / 272 / 512 (or 256) bytes; Q6_K: a 224-byte box from the 16-byte
  // boundary at or below the 210-byte superblock; IQ4_XS: a 144-byte box from
  // the 16-byte boundary at or below the 136-byte superblock (8 bytes below
  // every other one)
  static constexpr int RAW_ROW = Q6K ? 224 : (IQ4 ? 144 : RAW_K / 32 * BB);
  static constexpr int RAW_BYTES = BM * RAW_ROW;      // one raw slot
  // F16 rows arrive as 64-column boxes of [128 rows][128 B], 128-byte
  // swizzled (conflict-free row reads); block formats as one unswizzled box
  static constexpr int RAW_LOADS = F16W ? RAW_SUBS : 1;
  static constexpr int RAW_BOX = F16W ? BK : RAW_ROW / 2;  // 16-bit elements across a box
  static constexpr int NPIECE = BN / PIECE;
  // operand stages (A in TMEM and B in shared memory advance together)
  static constexpr int S = XS ? 2 : (NM == 2 ? 4 : (BN == 256 ? 4 : (Q4W ? 6 : (F16W ? 4 : 5))));
  static_assert(!Q6K || RAW_K == 256, "a Q6_K raw slot is one superblock");
  static_assert(!IQ4 || RAW_K == 256, "an IQ4_XS raw slot is one superblock");
  // (with 256-token tiles the raw ring also receives the partner's half of a
  // split). With gate/up the chunks of the two weights alternate through the
  // ring, chunk j in slot j % S_RAW; S_RAW must be even so that a slot always
  // holds the same weight: each slot's phases are then awaited in order by one
  // warpgroup. With an odd ring a warpgroup would wait on phase p + 2 of a slot
  // whose phase p + 1 belongs to the other warpgroup, and a parity wait cannot
  // tell phase p + 2 from phase p.
  static constexpr int S_RAW = NM == 1 ? (Q4W ? (BN == 256 ? 4 : 3) : (Q6K ? 3 : 2)) : 4;
  static_assert(!XS || RAW_K == CHUNK, "the exact leg folds one raw slot per accumulation chunk");
  static_assert(!F16W || BN == 128 || EPI == kEpiGluPair, "F16 tiles take 128 tokens, except a gate/up pair's");
  static constexpr int NTHREADS = 128 + 128 * NWG;
  static constexpr int ACC_COLS = (XS ? 3 : NM) * BN;
  static constexpr int A_COL0 = ACC_COLS;                       // first A column
  static constexpr int USED_COLS = ACC_COLS + NM * S * NP * A_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 128 ? 128 : USED_COLS <= 256 ? 256 : 512;
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_B = 0;
  static constexpr int OFF_RAW = OFF_B + S * NP * B_BYTES;
  static constexpr int OFF_BAR = OFF_RAW + S_RAW * RAW_BYTES;
  static constexpr int NBAR = 2 * S + 2 * S_RAW + 2 + 1 + 2 + 4;  // + accFull, drain, peerFree, 2 xferFull, 4 chunk
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;   // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NM == 1 || S_RAW % 2 == 0, "gate/up: each raw slot keeps one weight");
  static_assert(USED_COLS <= 512, "TMEM budget");
  static_assert(BN % PIECE == 0 && NPIECE >= NWG, "epilogue pieces (of 64 tokens) per warpgroup");
  static_assert(BN != 256 || S_RAW * RAW_BYTES >= 2 * PIECE_BYTES, "split: the raw ring holds the partner's two pieces");
  static_assert(!XS || (BN == 128 && NM == 1), "the exact leg takes 128-token tiles of one weight");
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

// Decodes one row's two blocks (64 k), held as the words w[0 .. 2 BB / 4),
// into 32 fp16 pairs in k order: a[j] = (w_2j, w_2j+1), j = 0..31.
template <int QT>
__device__ __forceinline__ void dequant_row_stage(const uint32_t* w, uint32_t (&a)[32]) {
  if constexpr (QT == kQ4_0) {
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


// F16: the 64 k of one row in one 128-byte-swizzled box row: 16-byte unit u
// of row r sits at unit u ^ (r mod 8) (the box starts 1024-byte aligned).
__device__ __forceinline__ void f16_row_stage(const uint8_t* box, uint32_t r, uint32_t (&a)[32]) {
  const uint8_t* row = box + r * 128u;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + ((u ^ (r & 7u)) << 4));
    a[4 * u] = v.x;
    a[4 * u + 1] = v.y;
    a[4 * u + 2] = v.z;
    a[4 * u + 3] = v.w;
  }
}

// Exact leg: one row's two blocks (64 k), words w[0 .. 2 BB / 4), into the
// fp16 pieces of W * 2^e: a1[j] = fp16(v_2j, v_2j+1) and a2[j] = fp16 of the
// remainders, v = d * q' * 2^e computed exactly in fp32 (an fp16 scale times a
// code of at most 8 bits, times a power of two). sw = 2^e.
//   code to float: a code c at bit offset 0 of a word OR-ed into the exponent
//   of 2^23 is the float 2^23 + c; minus 2^23 + 8 (Q4_0) or 2^23 + 128 (Q8_0,
//   the byte XOR 0x80) leaves q' exactly.
__device__ __forceinline__ void split2(float x, float y, uint32_t& h1, uint32_t& h2) {
  const __half2 a = __floats2half2_rn(x, y);
  const float2 b = __half22float2(a);
  const __half2 c = __floats2half2_rn(x - b.x, y - b.y);
  h1 = h2_as_u32(a);
  h2 = h2_as_u32(c);
}

template <int QT>
__device__ __forceinline__ void dequant_row_stage_xs(const uint32_t* w, float sw, uint32_t (&a1)[32],
                                                     uint32_t (&a2)[32]) {
  if constexpr (QT == kF16) {
    // w holds the 64 halves themselves (f16_row_stage); v = w * 2^e is exact
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float2 f = __half22float2(u32_as_h2(w[j]));
      split2(f.x * sw, f.y * sw, a1[j], a2[j]);
    }
  } else if constexpr (QT == kQ4_0) {
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __byte_perm(w[i], w[i + 1], 0x5432);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[4 + i] = w[5 + i];
    const float d0 = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu))) * sw;
    const float d1 = __half2float(__ushort_as_half((unsigned short)(w[4] >> 16))) * sw;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const float d = blk ? d1 : d0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = p[blk * 4 + i];  // bytes m = 0..3: elements 4i + m (low), 16 + 4i + m (high)
        // the nibbles four at a time; byte m under exponent 0x4B is 2^23 + n
        const uint32_t xl = x & 0x0F0F0F0Fu, xh = (x >> 4) & 0x0F0F0F0Fu;
        float lo[4], hi[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          lo[m] = (__uint_as_float(__byte_perm(xl, 0x4B000000u, 0x7440u + m)) - 8388616.0f) * d;
          hi[m] = (__uint_as_float(__byte_perm(xh, 0x4B000000u, 0x7440u + m)) - 8388616.0f) * d;
        }
        split2(lo[0], lo[1], a1[16 * blk + 2 * i], a2[16 * blk + 2 * i]);
        split2(lo[2], lo[3], a1[16 * blk + 2 * i + 1], a2[16 * blk + 2 * i + 1]);
        split2(hi[0], hi[1], a1[16 * blk + 8 + 2 * i], a2[16 * blk + 8 + 2 * i]);
        split2(hi[2], hi[3], a1[16 * blk + 8 + 2 * i + 1], a2[16 * blk + 8 + 2 * i + 1]);
      }
    }
  } else {
    const float d0 = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu))) * sw;
    const float d1 = __half2float(__ushort_as_half((unsigned short)(w[8] >> 16))) * sw;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t x = (c < 8 ? __byte_perm(w[c], w[c + 1], 0x5432) : w[1 + c]) ^ 0x80808080u;
      const float d = c < 8 ? d0 : d1;
      float v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)  // byte m under exponent 0x4B: 2^23 + 128 + q
        v[m] = (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u + m)) - 8388736.0f) * d;
      split2(v[0], v[1], a1[2 * c], a2[2 * c]);
      split2(v[2], v[3], a1[2 * c + 1], a2[2 * c + 1]);
    }
  }
}

// Q4_K / Q5_K: stage g (64 k) of one row's superblock, words w[0] = d | dmin
// << 16, w[1..3] = the packed scales, then (Q5_K) w[4..11] the fifth-bit
// bytes 0 .. 31, then the code bytes 32 g .. 32 g + 31 (8 words):
// a[j] for j < 16 the low nibbles (sub-block 2 g, elements 2j, 2j + 1), for
// j >= 16 the high nibbles (sub-block 2 g + 1). Each weight d sc q - dmin m is
// one fma of two exact products, rounded to fp32, then to fp16 (xs = false),
// or times sw = 2^e and split into two fp16 pieces (xs = true).
template <bool XSP, bool FIVE>
__device__ __forceinline__ void q4k_row_stage(const uint32_t* w, uint32_t g, float sw, uint32_t (&a1)[32],
                                              uint32_t (&a2)[32]) {
  const float d = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half((unsigned short)(w[0] >> 16)));
  float A[2], B[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t sc, m;
    q4k_scale_min_w(w + 1, 2 * g + h, sc, m);
    A[h] = d * (float)sc;
    B[h] = -(dmin * (float)m);
  }
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint32_t x = w[(FIVE ? 12 : 4) + v];
    const uint32_t f = FIVE ? w[4 + v] : 0u;  // fifth bits of elements 4 v .. 4 v + 3 (and + 32)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // the four codes of sub-block 2 g + h, one a byte (the fifth bit, bit
      // 2 g + h of each fifth-bit byte, worth 16)
      uint32_t qw = (x >> (4 * h)) & 0x0F0F0F0Fu;
      if (FIVE) qw |= ((f >> (2 * g + h)) & 0x01010101u) << 4;
      float q[4];
#pragma unroll
      for (int b = 0; b < 4; ++b)  // q exactly: the float 2^23 + q (byte b under exponent 0x4B) less 2^23
        q[b] = fmaf(A[h], __uint_as_float(__byte_perm(qw, 0x4B000000u, 0x7440u + b)) - 8388608.0f, B[h]);
      const int j = 16 * h + 2 * v;
      if constexpr (XSP) {
        split2(q[0] * sw, q[1] * sw, a1[j], a2[j]);
        split2(q[2] * sw, q[3] * sw, a1[j + 1], a2[j + 1]);
      } else {
        a1[j] = h2_as_u32(__floats2half2_rn(q[0], q[1]));
        a1[j + 1] = h2_as_u32(__floats2half2_rn(q[2], q[3]));
      }
    }
  }
}

// Q6_K: stage g (64 k) of one row's superblock, from shared-memory words that
// start at the word holding the superblock's first byte, sh bytes (0 or 2)
// into it: w[0..16] over the low-nibble bytes 64 h .. 64 h + 63 (h = g / 2),
// w[17..25] over the high-bit bytes 128 + 32 h .. 128 + 32 h + 31, w[26..27]
// over the scale bytes 192 + 4 g .. 192 + 4 g + 3, w[28] the word holding d.
// Element i of the stage takes nibble g % 2 of low byte i, bits 2 c of high
// byte i % 32 (c = 2 (g % 2) + i / 32) and scale 4 g + i / 16; d sc (q - 32)
// has at most 23 significant bits, so it is exact in fp32, then rounded once
// to fp16 (xs = false) or scaled by sw = 2^e and split (xs = true).
template <bool XSP>
__device__ __forceinline__ void q6k_row_stage(const uint32_t* w, uint32_t g, uint32_t sh, float sw,
                                              uint32_t (&a1)[32], uint32_t (&a2)[32]) {
  const uint32_t s8 = 8 * sh;
  auto at = [&](int m) { return __funnelshift_r(w[m], w[m + 1], s8); };
  const float d = __half2float(__ushort_as_half((unsigned short)((w[28] >> s8) & 0xFFFFu)));
  const uint32_t scw = at(26);
  float A[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) A[j] = d * (float)((int)(scw << (24 - 8 * j)) >> 24);  // int8 scale j
  const uint32_t nib = 4 * (g & 1u), hb = 4 * (g & 1u);
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    const uint32_t x = at(v);                       // low bytes of elements 4 v .. 4 v + 3
    const uint32_t y = at(17 + (v & 7));            // their high-bit bytes (element % 32)
    const uint32_t hs = hb + 2 * (uint32_t)(v >> 3);  // 2 c
    // the four 6-bit codes, one a byte
    const uint32_t qw = ((x >> nib) & 0x0F0F0F0Fu) | (((y >> hs) & 0x03030303u) << 4);
    float q[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)  // q - 32 exactly: the float 2^23 + q (byte b under exponent 0x4B) less 2^23 + 32
      q[b] = A[v >> 2] * (__uint_as_float(__byte_perm(qw, 0x4B000000u, 0x7440u + b)) - 8388640.0f);
    if constexpr (XSP) {
      split2(q[0] * sw, q[1] * sw, a1[2 * v], a2[2 * v]);
      split2(q[2] * sw, q[3] * sw, a1[2 * v + 1], a2[2 * v + 1]);
    } else {
      a1[2 * v] = h2_as_u32(__floats2half2_rn(q[0], q[1]));
      a1[2 * v + 1] = h2_as_u32(__floats2half2_rn(q[2], q[3]));
    }
  }
}

// IQ4_XS: stage g (64 k: sub-blocks 2 g and 2 g + 1) of one row's superblock,
// words w[0] = d | high scale bits << 16, w[1] = the low scale nibbles, then
// the stage's code bytes, w[2..5] for sub-block 2 g and w[6..9] for 2 g + 1.
// Word v of a sub-block holds elements 4 v .. 4 v + 3 in its low nibbles and
// 16 + 4 v .. in its high ones; the book lookup turns it into (A0, B0, A1, B1)
// and (A2, B2, A3, B3) as bytes book + 128. d (ls - 32) book[c] has at most
// 23 significant bits, so it is exact in fp32, then rounded once to fp16
// (xs = false) or scaled by sw = 2^e and split (xs = true).
template <bool XSP>
__device__ __forceinline__ void iq4xs_row_stage(const uint32_t* w, uint32_t g, float sw, uint32_t (&a1)[32],
                                                uint32_t (&a2)[32]) {
  const float d = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float D = d * (float)iq4_scale(w[0], w[1], 2 * g + h);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t u[2];
      iq4_word(w[2 + 4 * h + v], u[0], u[1]);
      // element 4 v + m is byte 2 (m % 2) of u[m / 2], 16 + 4 v + m the byte after
      float A[4], B[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {  // book[c] exactly: the float 2^23 + byte less 2^23 + 128
        A[m] = (__uint_as_float(__byte_perm(u[m >> 1], 0x4B000000u, 0x7440u + 2 * (m & 1))) - 8388736.0f) * D;
        B[m] = (__uint_as_float(__byte_perm(u[m >> 1], 0x4B000000u, 0x7441u + 2 * (m & 1))) - 8388736.0f) * D;
      }
      const int j = 16 * h + 2 * v;
      if constexpr (XSP) {
        split2(A[0] * sw, A[1] * sw, a1[j], a2[j]);
        split2(A[2] * sw, A[3] * sw, a1[j + 1], a2[j + 1]);
        split2(B[0] * sw, B[1] * sw, a1[j + 8], a2[j + 8]);
        split2(B[2] * sw, B[3] * sw, a1[j + 9], a2[j + 9]);
      } else {
        a1[j] = h2_as_u32(__floats2half2_rn(A[0], A[1]));
        a1[j + 1] = h2_as_u32(__floats2half2_rn(A[2], A[3]));
        a1[j + 8] = h2_as_u32(__floats2half2_rn(B[0], B[1]));
        a1[j + 9] = h2_as_u32(__floats2half2_rn(B[2], B[3]));
      }
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int QT, int EPI, int BN, bool XS>
__global__ void __launch_bounds__(Cfg<QT, EPI, BN, XS>::NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWu,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmX2,
                   const __grid_constant__ CUtensorMap tmR, int n, int k, int T, float* Y, int ldy, const float* R,
                   const int* erow, const int* etok, unsigned* status, int early, OutRegions reg) {
  // early: bits 0-3 what may be read before the dependency wait (kEarly*),
  // bit 4 set when tmR describes the residual (L2 prefetches of it), bit 5
  // independent k splits (below), bit 6 (kOutF16) an fp16 gate/up output.
  // Exact leg (XS): X and X2 are the two fp16 pieces of X * 2^etok[t];
  // erow[i] (erow[n + i] for the up weight) is the exponent e of the
  // row's scale 2^e (computed before the launch, see row_exp_kernel).
  using C = Cfg<QT, EPI, BN, XS>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the shared array so that
  // the compiler keeps the shared address space (shared loads, not generic)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sRaw = smem + C::OFF_RAW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;              // stage ready: B landed and every A writer arrived
  uint64_t* empty = full + C::S;      // stage free: its MMAs completed
  uint64_t* rawFull = empty + C::S;
  uint64_t* rawEmpty = rawFull + C::S_RAW;
  uint64_t* accFull = rawEmpty + C::S_RAW;
  uint64_t* drain = accFull + 1;
  uint64_t* peerFree = drain + 1;     // split: the partner's raw ring is free to receive
  uint64_t* xferFull = peerFree + 1;  // split: [wg] the partner's piece for warpgroup wg has landed
  uint64_t* chunkFull = xferFull + 2;   // exact leg: [b] the chunk in accumulator b is complete
  uint64_t* chunkEmpty = chunkFull + 2; // exact leg: [b] accumulator b has been added into the sum
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM;
  const int t0 = blockIdx.y * BN;
  // split-K: CTA z of gridDim.z takes raw chunks [c0, c1); ring indices are
  // local. A gate/up pair: CTA z takes all of k for weight z.
  constexpr bool pair = EPI == kEpiGluPair;
  const int nchunks_all = k / CHUNK;
  const int nsplit = gridDim.z, z = blockIdx.z;
  const int c0 = pair ? 0 : (int)((long)z * nchunks_all / nsplit);
  const int c1 = pair ? nchunks_all : (int)((long)(z + 1) * nchunks_all / nsplit);
  const CUtensorMap* wmap0 = pair && z ? &tmWu : &tmW;  // the weight of m = 0
  // k split: a cluster pair that exchanges halves (two splits), or, with bit
  // 5 of `early`, independent splits each writing its own partial output (Y +
  // z T ldy), added by a second kernel
  const bool indep = (early & 32) != 0;
  const bool clus = nsplit == 2 && !indep;
  if (indep) Y += (size_t)z * (size_t)T * (size_t)ldy;
  const int nchunks = c1 - c0;
  const int nk = nchunks * SUBS;
  const int nunits = nk / C::RAW_SUBS;  // raw slots' worth of k
  // piece p (token columns t0 + 64 p ..) holds a token; with a split, CTA z
  // (its rank in the cluster) writes pieces 2 z and 2 z + 1
  auto live = [&](int p) { return t0 + p * PIECE < T; };
  auto kept = [&](int p) { return !clus || (p >> 1) == z; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; ++i) {
      mbar_init(&full[i], 1 + 4 * C::NM);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::S_RAW; ++i) {
      mbar_init(&rawFull[i], 1);
      mbar_init(&rawEmpty[i], 4 * C::DQ);  // every warpgroup of the weight reads the chunk
    }
    mbar_init(accFull, 1);
    mbar_init(drain, 1);
    mbar_init(peerFree, 1);
    // one arrival per thread of the partner's sending warpgroup
    for (int w = 0; w < 2; ++w) mbar_init(&xferFull[w], 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&chunkFull[b], 1);
      mbar_init(&chunkEmpty[b], 4);  // the warps of the summing warpgroup
    }
    abort_flag[0] = 0;   // set by a wait that gives up
    abort_flag[1] = 0;   // never set: drain waits ignore the abort
    fence_mbar_init();
    grid_launch_dependents();
  }
  // split: the partner's barriers must be initialized before the first remote
  // access (the matching wait comes just before it); a thread arrives at the
  // closing barrier once it touches the partner's shared memory no more
  bool cl_started = false, cl_done = false;
  if (clus) cluster_arrive_relaxed();
  if (warp == 1) tmem_alloc(tmem_holder, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------ raw weight producer
    if (lane == 0) {
      tma_prefetch_desc(wmap0);
      if (C::NM == 2) tma_prefetch_desc(&tmWu);
      // x of box b of raw slot u (16-bit elements): the raw row bytes of block
      // formats, the k index itself for F16
      auto raw_x = [&](int u, int b) {
        if constexpr (C::Q6K) return (((c0 + u) * 210) & ~15) / 2;  // 16-byte aligned; the decode skips the rest
        if constexpr (C::IQ4) return (((c0 + u) * 136) & ~15) / 2;
        return C::F16W ? c0 * CHUNK + u * C::RAW_K + b * BK : (c0 + u) * (C::RAW_ROW / 2);
      };
      // an L2 prefetch changes no data, so it may run before the wait
      for (int u = 0; u < PF && u < nunits; ++u)
        for (int m = 0; m < C::NM; ++m)
          for (int b = 0; b < C::RAW_LOADS; ++b)
            tma_prefetch_l2_2d(m ? (const void*)&tmWu : (const void*)wmap0, raw_x(u, b), m0);
      if ((early & 15) == kEarlyNone) grid_dependency_wait();
      int last_issued[C::S_RAW];
      for (int i = 0; i < C::S_RAW; ++i) last_issued[i] = -1;
      bool ok = true;
      for (int u = 0; u < nunits && ok; ++u) {
        for (int m = 0; m < C::NM && ok; ++m) {
          const int j = u * C::NM + m;
          const int slot = j % C::S_RAW;
          ok = mbar_wait(&rawEmpty[slot], ((j / C::S_RAW) & 1) ^ 1, abort_flag, status);
          if (!ok) break;
          const void* map = m ? (const void*)&tmWu : (const void*)wmap0;
          mbar_arrive_expect_tx(&rawFull[slot], C::RAW_BYTES);
          for (int b = 0; b < C::RAW_LOADS; ++b)
            tma_load_2d(sRaw + slot * C::RAW_BYTES + b * (C::RAW_BYTES / C::RAW_LOADS), map, raw_x(u, b), m0,
                        &rawFull[slot]);
          if (u + PF < nunits)
            for (int b = 0; b < C::RAW_LOADS; ++b) tma_prefetch_l2_2d(map, raw_x(u + PF, b), m0);
          last_issued[slot] = j;
        }
      }
      if (ok && clus) {
        // every raw slot read for the last time: the partner may send into the ring
        const int total = nunits * C::NM;
        for (int v = total; v < total + C::S_RAW && ok; ++v)
          ok = mbar_wait(&rawEmpty[v % C::S_RAW], ((v / C::S_RAW) & 1) ^ 1, abort_flag, status);
        cluster_wait();
        cl_started = true;
        if (ok) mbar_arrive_remote(mapa_shared(smem_u32(peerFree), (uint32_t)(1 - z)));
        cluster_arrive();
        cl_done = true;
      }
      if (!ok)  // let the copies in flight land before the CTA exits
        for (int i = 0; i < C::S_RAW; ++i)
          if (last_issued[i] >= 0) mbar_wait(&rawFull[i], (last_issued[i] / C::S_RAW) & 1, abort_flag + 1, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ activation producer
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      if (XS) tma_prefetch_desc(&tmX2);
      // X is written by the conversion kernel, which may still be running
      grid_dependency_wait();
      bool ok = true;
      int last = -1;
      for (int i = 0; i < nk; ++i) {
        const int st = i % C::S;
        ok = mbar_wait(&empty[st], ((i / C::S) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[st], C::NP * C::B_BYTES);
        tma_load_2d(sB + st * C::NP * C::B_BYTES, &tmX, (c0 * SUBS + i) * BK, t0, &full[st]);
        if (XS) tma_load_2d(sB + (st * C::NP + 1) * C::B_BYTES, &tmX2, (c0 * SUBS + i) * BK, t0, &full[st]);
        last = i;
        // the residual pieces this CTA finalizes, into L2 a few stages before
        // the end (the epilogue threads load them into registers)
        if (EPI == kEpiResidual && (early & 16) && i == (nk > 2 * C::S ? nk - 2 * C::S : 0))
          for (int p = 0; p < C::NPIECE; ++p)
            if (kept(p) && live(p)) tma_prefetch_l2_2d(&tmR, m0, t0 + p * PIECE);
      }
      // After a give-up, wait (bounded) on the last stage issued: its phase
      // also needs the dequant warps, so it may never complete, but by the time
      // the bounded wait ends every copy issued has landed.
      if (!ok && last >= 0) mbar_wait(&full[last % C::S], (last / C::S) & 1, abort_flag + 1, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
    const uint64_t bdesc0 = smem_desc_sw128(sB);
    bool ok = true;
    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nk; ++i) {
      const int cc = i / SUBS, ss = i % SUBS;  // local chunk, stage within it
      if (XS && ss == 0 && cc >= 2) {  // accumulator cc & 1 has been added into the sum
        ok = __all_sync(0xffffffffu, mbar_wait(&chunkEmpty[cc & 1], ((cc - 2) >> 1) & 1, abort_flag, status));
        if (!ok) break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      // stage st of B starts st * NP * B_BYTES later: (bytes >> 4) descriptor units
      const uint64_t bdesc = bdesc0 + (uint64_t)((st * C::NP * C::B_BYTES) >> 4);
#pragma unroll
      for (int m = 0; m < C::NM; ++m) {
        const uint32_t a_tmem = tmem_base + C::A_COL0 + (m * C::S + st) * C::NP * C::A_COLS;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // 16 k = 8 TMEM columns of A, +32 bytes of B inside its swizzle atom
          if (XS) {  // W1 . X1 + W1 . X2 + W2 . X1 into the chunk's accumulator
            const uint32_t d = tmem_base + (uint32_t)(cc & 1) * BN;
            mma_f16_ts_elect(d, a_tmem + kk * 8, bdesc + 2 * kk, idesc, (ss | kk) != 0);
            mma_f16_ts_elect(d, a_tmem + kk * 8, bdesc + (C::B_BYTES >> 4) + 2 * kk, idesc, 1);
            mma_f16_ts_elect(d, a_tmem + C::A_COLS + kk * 8, bdesc + 2 * kk, idesc, 1);
          } else {
            mma_f16_ts_elect(tmem_base + m * BN, a_tmem + kk * 8, bdesc + 2 * kk, idesc, (i | kk) != 0);
          }
        }
      }
      mma_commit_elect(&empty[st]);
      if (XS && ss == SUBS - 1) mma_commit_elect(&chunkFull[cc & 1]);
      if (++st == C::S) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (ok) {
      mma_commit_elect(accFull);
    } else {  // wait until the MMAs already issued have finished
      mma_commit_elect(drain);
      __all_sync(0xffffffffu, mbar_wait(drain, 0, abort_flag + 1, status));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ dequant, then epilogue
    const int wg = (warp - 4) >> 2;                  // dequant warpgroup
    const int g = wg % C::NM;                        // which weight (0: W / gate, 1: up)
    const int par = wg / C::NM;                      // which stages: i % DQ == par
    const uint32_t q = (uint32_t)(warp & 3);         // lane quarter of TMEM this warp may access
    const uint32_t r = q * 32 + lane;                // tile row == TMEM lane
    const uint32_t lane_base = tmem_base + ((q * 32u) << 16);
    // exact leg: 2^e of this thread's weight row (erow is written by a kernel
    // launched in plain stream order before this one)
    float sw = 1.f;
    if (XS) {
      grid_dependency_wait();
      const int ri = m0 + (int)r;
      sw = __int_as_float((127 + (ri < n ? erow[(size_t)g * n + ri] : 0)) << 23);
    }
    bool ok = true;
    // exact leg: add the finished chunk cs in accumulator cs & 1 into the sum
    // (chunk 0 starts it); warpgroup 0, 128 token columns a thread
    auto fold = [&](int cs) {
      bool okf = __all_sync(0xffffffffu, mbar_wait(&chunkFull[cs & 1], (cs >> 1) & 1, abort_flag, status));
      if (okf) {
        tc_fence_after();
        const uint32_t src = lane_base + (uint32_t)(cs & 1) * BN, sum = lane_base + 2 * BN;
#pragma unroll 1
        for (int cb = 0; cb < BN / 32; ++cb) {
          uint32_t va[32], vs[32];
          tmem_ld_32x32b_x32(src + cb * 32, va);
          if (cs > 0) tmem_ld_32x32b_x32(sum + cb * 32, vs);
          tmem_ld_wait_regs(va);
          if (cs > 0) {
            regs_after_wait(vs);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) vs[jj] = __float_as_uint(__uint_as_float(vs[jj]) + __uint_as_float(va[jj]));
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) vs[jj] = va[jj];
          }
          tmem_st_32x32b_x32(sum + cb * 32, vs);
          tmem_st_wait();
        }
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&chunkEmpty[cs & 1]);
      return okf;
    };
    for (int c = 0; c < nunits && ok; ++c) {
      if (XS && par == 0 && c >= 2) ok = fold(c - 2);  // exact leg: a raw slot is a chunk
      if (!ok) break;
      const int j = c * C::NM + g;
      const int slot = j % C::S_RAW;
      ok = __all_sync(0xffffffffu, mbar_wait(&rawFull[slot], (j / C::S_RAW) & 1, abort_flag, status));
      if (!ok) break;
      const uint8_t* raw_slot = sRaw + slot * C::RAW_BYTES;
      const uint32_t* raw_row = reinterpret_cast<const uint32_t*>(raw_slot + r * C::RAW_ROW);
      for (int s = par; s < C::RAW_SUBS; s += C::DQ) {
        const int i = c * C::RAW_SUBS + s;
        const int st = i % C::S;
        uint32_t w[C::NWORDS], a[32], a2[32];
        if constexpr (C::F16W) {
          f16_row_stage(raw_slot + s * (C::RAW_BYTES / C::RAW_LOADS), r, w);
        } else if constexpr (C::Q6K) {
          // the superblock starts rem = 210 c mod 16 bytes into the box row
          const uint32_t* sbw = raw_row + ((((c0 + c) * 2) & 15) >> 2);
          const int h = s >> 1;
#pragma unroll
          for (int v = 0; v < 17; ++v) w[v] = sbw[16 * h + v];
#pragma unroll
          for (int v = 0; v < 9; ++v) w[17 + v] = sbw[32 + 8 * h + v];
          w[26] = sbw[48 + s];
          w[27] = sbw[49 + s];
          w[28] = sbw[52];
        } else if constexpr (C::IQ4) {
          // the superblock starts 8 bytes into the box row when its index is odd
          const uint32_t* sbw = raw_row + 2 * ((c0 + c) & 1);
          w[0] = sbw[0];
          w[1] = sbw[1];
#pragma unroll
          for (int v = 0; v < 8; ++v) w[2 + v] = sbw[2 + 8 * s + v];
        } else if constexpr (QT == kQ4_K || QT == kQ5_K) {
          constexpr int H = QT == kQ5_K ? 12 : 4;  // words before the code bytes
#pragma unroll
          for (int v = 0; v < H; ++v) w[v] = raw_row[v];
#pragma unroll
          for (int v = 0; v < 8; ++v) w[H + v] = raw_row[H + 8 * s + v];
        } else {
#pragma unroll
          for (int v = 0; v < C::NWORDS; ++v) w[v] = raw_row[s * C::NWORDS + v];
        }
        if constexpr (C::Q6K)
          q6k_row_stage<XS>(w, (uint32_t)s, (uint32_t)((c0 + c) * 2) & 2u, sw, a, a2);  // overlaps the wait below
        else if constexpr (C::IQ4)
          iq4xs_row_stage<XS>(w, (uint32_t)s, sw, a, a2);
        else if constexpr (QT == kQ4_K || QT == kQ5_K)
          q4k_row_stage<XS, QT == kQ5_K>(w, (uint32_t)s, sw, a, a2);
        else if constexpr (XS)
          dequant_row_stage_xs<QT>(w, sw, a, a2);  // overlaps the wait below
        else if constexpr (C::F16W)
#pragma unroll
          for (int v = 0; v < 32; ++v) a[v] = w[v];  // already the fp16 operand
        else
          dequant_row_stage<QT>(w, a);
        ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((i / C::S) & 1) ^ 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        // tcgen05.st reads its source registers asynchronously: a[] stays
        // untouched until the wait
        const uint32_t acol = lane_base + C::A_COL0 + (g * C::S + st) * C::NP * C::A_COLS;
        tmem_st_32x32b_x32(acol, a);
        if constexpr (XS) tmem_st_32x32b_x32(acol + C::A_COLS, a2);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rawEmpty[slot]);
    }

    // ---------------------------------------------- epilogue
    // Y and R may still be in use by the preceding kernel
    grid_dependency_wait();
    const int row = m0 + (int)r;
    // pieces wg, wg + NWG, ... (a 192-token tile: two for warpgroup 0, one for 1)
    const int npw = clus ? 1 : (C::NPIECE - wg + C::NWG - 1) / C::NWG;
    // the pieces this warpgroup finalizes: all of the tile's pieces split
    // evenly, or with a split piece 2 z + wg
    auto piece = [&](int pp) { return clus ? 2 * z + wg : wg + pp * C::NWG; };
    // residual of piece p into registers (coalesced: the warp's lanes read 32
    // consecutive floats of one token's row)
    float rv[PIECE];
    auto load_r = [&](int p) {
#pragma unroll
      for (int j = 0; j < PIECE; ++j) {
        const int t = t0 + p * PIECE + j;
        rv[j] = (EPI == kEpiResidual && t < T && row < n) ? R[(size_t)t * ldy + row] : 0.f;
      }
    };
    if (EPI == kEpiResidual && ok && live(piece(0))) load_r(piece(0));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(accFull, 0, abort_flag, status));
    tc_fence_after();
    if (XS) {  // warpgroup 0's last fold is in TMEM before either reads the sum
      tc_fence_before();
      named_sync(3, 256);
      tc_fence_after();
    }

    if (clus) {
      // the piece the partner keeps, pg, goes from registers straight into the
      // partner's raw ring at 32 KB x wg ([64 tokens][128 rows]); the
      // partner's copy of piece pk lands in this raw ring the same way
      const uint32_t peer = (uint32_t)(1 - z);
      const int pg = 2 * (1 - z) + wg;
      cluster_wait();  // the partner has started: its barriers exist
      cl_started = true;
      if (ok && live(pg)) {
        uint32_t v[64];
        tmem_ld_32x32b_x32(lane_base + pg * PIECE, v);
        tmem_ld_32x32b_x32(lane_base + pg * PIECE + 32, v + 32);
        tmem_ld_wait_regs(v);
        regs_after_wait(v + 32);
        // the partner's raw ring is free once it has decoded its last chunk
        bool go = __all_sync(0xffffffffu, mbar_wait_cluster(peerFree, 0, abort_flag, status));
        if (go) {
          const uint32_t dst = mapa_shared(smem_u32(sRaw + wg * PIECE_BYTES), peer) + r * 4;
#pragma unroll
          for (int j = 0; j < PIECE; ++j) st_cluster_f32(dst + (uint32_t)(j * BM * 4), __uint_as_float(v[j]));
          // release: the stores above before the arrival the partner waits on
          mbar_arrive_remote(mapa_shared(smem_u32(&xferFull[wg]), peer));
        }
      }
      // this CTA no longer touches the partner's shared memory
      cluster_arrive();
      cl_done = true;
    }

    for (int pp = 0; pp < npw; ++pp) {
      const int p = piece(pp);
      if (!live(p)) continue;  // the same for the whole warpgroup
      if (pp > 0 && EPI == kEpiResidual && ok) load_r(p);
      uint32_t v[64];
      if (ok && clus)  // the partner's half of this piece has landed
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(&xferFull[wg], 0, abort_flag, status));
      if (!ok) continue;
      if constexpr (XS) {
        // y = ((sum + acc of chunk nc - 2) + acc of chunk nc - 1), the sum
        // holding chunks 0 .. nc - 3
        const int nc = nchunks;
        bool first = true;
        for (int part = 0; part < 3; ++part) {
          uint32_t col;
          if (part == 0) {
            if (nc < 3) continue;
            col = 2 * BN;
          } else {
            const int cs = nc - 3 + part;  // nc - 2, nc - 1
            if (cs < 0) continue;
            col = (uint32_t)(cs & 1) * BN;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t t[32];
            tmem_ld_32x32b_x32(lane_base + col + p * PIECE + 32 * h, t);
            tmem_ld_wait_regs(t);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              v[32 * h + jj] = first ? t[jj] : __float_as_uint(__uint_as_float(v[32 * h + jj]) + __uint_as_float(t[jj]));
          }
          first = false;
        }
      } else {
        tmem_ld_32x32b_x32(lane_base + p * PIECE, v);
        tmem_ld_32x32b_x32(lane_base + p * PIECE + 32, v + 32);
        tmem_ld_wait_regs(v);
        regs_after_wait(v + 32);
      }
      if (C::NM == 2 && !XS) {  // y = silu(gate) * up
        uint32_t u[64];
        tmem_ld_32x32b_x32(lane_base + BN + p * PIECE, u);
        tmem_ld_32x32b_x32(lane_base + BN + p * PIECE + 32, u + 32);
        tmem_ld_wait_regs(u);
        regs_after_wait(u + 32);
#pragma unroll
        for (int j = 0; j < PIECE; ++j) {
          const float gt = __uint_as_float(v[j]);
          v[j] = __float_as_uint(gt / (1.0f + expf(-gt)) * __uint_as_float(u[j]));
        }
      }
      if (clus) {  // p0 + p1, in split order; a gate/up pair: silu(gate) * up
        const float* src = reinterpret_cast<const float*>(sRaw + wg * PIECE_BYTES) + r;
#pragma unroll
        for (int j = 0; j < PIECE; ++j) {
          const float o = src[j * BM];
          const float mine = __uint_as_float(v[j]);
          if constexpr (pair) {
            const float gt = z == 0 ? mine : o, up = z == 0 ? o : mine;
            v[j] = __float_as_uint(gt / (1.0f + expf(-gt)) * up);
          } else {
            v[j] = __float_as_uint(z == 0 ? mine + o : o + mine);
          }
        }
      }
      if constexpr (XS) {
        // undo the scales: y = acc * 2^-erow * 2^-etok (exact, two steps)
        const float sr = __int_as_float((127 - erow[row < n ? row : 0]) << 23);
#pragma unroll
        for (int j = 0; j < PIECE; ++j) {
          const int t = t0 + p * PIECE + j;
          const float stk = __int_as_float((127 - etok[t < T ? t : 0]) << 23);
          v[j] = __float_as_uint(__uint_as_float(v[j]) * sr * stk);
        }
      }
      if constexpr (EPI == kEpiSwiGLU || pair) {
        if (row < n && (early & kOutF16)) {
          // fp16 output, the next GEMM's operand (Y holds uint16, ldy in them)
          uint16_t* Y16 = reinterpret_cast<uint16_t*>(Y);
#pragma unroll
          for (int j = 0; j < PIECE; ++j) {
            const int t = t0 + p * PIECE + j;
            if (t < T) Y16[(size_t)t * ldy + row] = __half_as_ushort(__float2half_rn(__uint_as_float(v[j])));
          }
          continue;
        }
      }
      if (row < n) {
        // this row's place: Y, or (a plain GEMM) the region its row falls in
        float* yb = Y;
        int ld = ldy, rr = row;
        if constexpr (EPI == kEpiPlain) {
          if (reg.y1 && row >= reg.r1) {
            const bool second = reg.y2 && row >= reg.r2;
            yb = second ? reg.y2 : reg.y1;
            ld = second ? reg.ld2 : reg.ld1;
            rr = row - (second ? reg.r2 : reg.r1);
          }
        }
        // R row t was read before Y row t is written (Y may be R), by this thread
#pragma unroll
        for (int j = 0; j < PIECE; ++j) {
          const int t = t0 + p * PIECE + j;
          float y = __uint_as_float(v[j]);
          if (EPI == kEpiResidual) y += rv[j];
          if (t < T) yb[(size_t)t * ld + rr] = y;
        }
      }
    }
    tc_fence_before();
  }

  // split: neither CTA exits while the other may still access its shared memory
  if (clus) {
    if (!cl_started) cluster_wait();
    if (!cl_done) cluster_arrive();
    cluster_wait();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- X -> fp16
// Launched in plain stream order (its griddepcontrol.wait then returns at
// once); it lets the GEMM after it launch as soon as it starts. One
// CTA per SM, at most 64 registers a thread (so that a GEMM CTA of up to 128
// registers a thread fits beside it); each thread converts four groups of 8
// per pass, all loads issued before the stores.
__global__ void __launch_bounds__(256, 4) x_to_f16_kernel(const float* __restrict__ X, uint16_t* __restrict__ X16,
                                                       size_t count) {
  grid_dependency_wait();
  grid_launch_dependents();
  const size_t n8 = count / 8;
  const float4* X4 = reinterpret_cast<const float4*>(X);
  uint4* Y4 = reinterpret_cast<uint4*>(X16);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (size_t i0 = tid; i0 < n8; i0 += 4 * stride) {
    float4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t i = i0 + u * stride;
      if (i < n8) {
        a[u] = X4[2 * i];
        b[u] = X4[2 * i + 1];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t i = i0 + u * stride;
      if (i < n8) {
        const __half2 h0 = __floats2half2_rn(a[u].x, a[u].y), h1 = __floats2half2_rn(a[u].z, a[u].w);
        const __half2 h2 = __floats2half2_rn(b[u].x, b[u].y), h3 = __floats2half2_rn(b[u].z, b[u].w);
        Y4[i] = make_uint4(h2_as_u32(h0), h2_as_u32(h1), h2_as_u32(h2), h2_as_u32(h3));
      }
    }
  }
  for (size_t i = n8 * 8 + tid; i < count; i += stride) X16[i] = __half_as_ushort(__float2half_rn(X[i]));
}

// ---------------------------------------------------------------- host side
template <int QT, int EPI, int BN, bool XS = false>
int launch_cfg(const void* W, const void* Wu, int n, int k, const uint16_t* X16, int T, float* Y, int ldy,
               const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len, int nsplit, int early,
               int x_rows, const uint16_t* X16b = nullptr, const int* erow = nullptr, const int* etok = nullptr,
               OutRegions reg = OutRegions{nullptr, nullptr, 0, 0, 0, 0}) {
  using C = Cfg<QT, EPI, BN, XS>;
  auto fn = encode_fn(msg, msg_len);
  if (!fn) return -1;
  CUtensorMap mW, mWu;
  const uint64_t row_bytes = C::Q6K ? (uint64_t)(k / 256) * 210 : (uint64_t)(k / 32) * C::BB;
  const CUtensorMapSwizzle wswz = C::F16W ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (!make_map_2d(fn, &mW, CU_TENSOR_MAP_DATA_TYPE_UINT16, W, row_bytes / 2, (uint64_t)n, row_bytes, C::RAW_BOX,
                   BM, wswz, msg, msg_len))
    return -1;
  if (C::NM == 2 || EPI == kEpiGluPair) {
    if (!make_map_2d(fn, &mWu, CU_TENSOR_MAP_DATA_TYPE_UINT16, Wu, row_bytes / 2, (uint64_t)n, row_bytes, C::RAW_BOX,
                     BM, wswz, msg, msg_len))
      return -1;
  } else {
    mWu = mW;
  }
  // B operand: fp16 X, 128-byte rows of a 64-column stage, swizzled
  const uint64_t xr = (uint64_t)(x_rows > T ? x_rows : T);
  CUtensorMap mX;
  if (!make_map_2d(fn, &mX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X16, (uint64_t)k, xr, (uint64_t)k * 2, BK, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len))
    return -1;
  CUtensorMap mX2 = mX;
  if (XS && !make_map_2d(fn, &mX2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X16b, (uint64_t)k, xr, (uint64_t)k * 2, BK, BN,
                         CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len))
    return -1;
  // the residual, [T] rows of n fp32 ldy apart, only for L2 prefetches of
  // 128-row x 64-token boxes: a row stride that is not a multiple of 16
  // bytes cannot be described, and then nothing is prefetched
  CUtensorMap mR = mX;
  int r_pf = 0;
  if (EPI == kEpiResidual && (ldy % 4) == 0 && ((uintptr_t)R & 15) == 0) {
    if (!make_map_2d(fn, &mR, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, R, (uint64_t)n, (uint64_t)T, (uint64_t)ldy * 4, BM,
                     PIECE, CU_TENSOR_MAP_SWIZZLE_NONE, msg, msg_len))
      return -1;
    r_pf = 1;
  }

  auto kern = gemm_tc_kernel<QT, EPI, BN, XS>;
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
  cudaLaunchAttribute attr[2] = {pdl_attr(), pdl_attr()};
  cfg.numAttrs = 1;
  if (nsplit == 2 && !(early & 32)) {  // the two k halves (or gate/up CTAs) of a tile form a cluster
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 2;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, mW, mWu, mX, mX2, mR, n, k, T, Y, ldy, R, erow, etok, status, early | (r_pf << 4),
                         reg);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, msg_len, "gemm_tc launch: %s", cudaGetErrorString(e));
    return -1;
  }
  return 0;
}

template <int QT>
int launch_q(const GemmPlan& pl, const void* W, const void* Wu, int n, int k, const uint16_t* X16, int T, float* Y,
             int ldy, const float* R, unsigned* status, cudaStream_t s, char* msg, size_t msg_len, int w, int xr,
             const OutRegions& reg) {
  if (Wu && pl.pair)
    return launch_cfg<QT, kEpiGluPair, 256>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, 2, w, xr);
  if (Wu) return launch_cfg<QT, kEpiSwiGLU, 128>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, 1, w, xr);
  if constexpr (QT == kF16) {
    // an F16 raw slot is four times a Q4_0 one: 256-token tiles do not fit
    (void)pl;
  } else if (pl.bn == 256) {
    if (R)
      return launch_cfg<QT, kEpiResidual, 256>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, pl.nsplit, w,
                                               xr);
    return launch_cfg<QT, kEpiPlain, 256>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, pl.nsplit, w, xr,
                                          nullptr, nullptr, nullptr, reg);
  } else if (pl.bn == 192) {
    if (R) return launch_cfg<QT, kEpiResidual, 192>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, 1, w, xr);
    return launch_cfg<QT, kEpiPlain, 192>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, 1, w, xr, nullptr,
                                          nullptr, nullptr, reg);
  }
  if (R) return launch_cfg<QT, kEpiResidual, 128>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, 1, w, xr);
  return launch_cfg<QT, kEpiPlain, 128>(W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, 1, w, xr, nullptr,
                                        nullptr, nullptr, reg);
}

// ---------------------------------------------------------------- exact-leg splits
// Per weight row: the exponent e with max_b |d_b| * qmax * 2^e in [2^14, 2^15)
// (qmax = 8 for Q4_0, 128 for Q8_0, the largest |q'|), so that every d * q' of
// the row times 2^e lies below 2^15 and its remainder after fp16 rounding
// stays an fp16 normal number unless it is far below the row's largest. One
// warp per row; 0 for a row of zero scales.
__global__ void row_exp_kernel(const uint8_t* __restrict__ W, int n, int nblk, int bb, float qmax,
                               int* __restrict__ erow) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;
  const uint8_t* base = W + (size_t)row * nblk * bb;
  float m = 0.f;
  for (int b = lane; b < nblk; b += 32) {
    const unsigned short bits = *reinterpret_cast<const unsigned short*>(base + (size_t)b * bb);
    m = fmaxf(m, fabsf(__half2float(__ushort_as_half(bits))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) {
    int e = 0;
    if (m > 0.f) e = 14 - ((int)((__float_as_uint(m * qmax) >> 23) & 0xFFu) - 127);
    erow[row] = e;
  }
}

// F16: the same exponent from the row's largest |w| (qmax = 1): every w * 2^e
// is again an fp16 value while it stays above 2^-14, so W2 is zero there.
// One warp per row, 16-byte loads (k % 256 == 0); the largest magnitude is
// the largest of the bit patterns with the sign cleared (finite halves).
__global__ void row_exp_f16_kernel(const uint16_t* __restrict__ W, int n, int k, int* __restrict__ erow) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;
  const uint4* base = reinterpret_cast<const uint4*>(W + (size_t)row * k);
  uint32_t m = 0;
  for (int i = lane; i < k / 8; i += 32) {
    const uint4 v = base[i];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, max(w4[q] & 0x7FFFu, (w4[q] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) {
    int e = 0;
    if (m > 0u) {
      const float f = __half2float(__ushort_as_half((unsigned short)m));
      e = 14 - ((int)((__float_as_uint(f) >> 23) & 0xFFu) - 127);
    }
    erow[row] = e;
  }
}

// K-quants: the same exponent from a bound on the row's largest |w|, the
// largest over its superblocks of |d| cd + |dmin| cm: Q4_K and Q5_K |d| 63 qmax
// + |dmin| 63 (qmax 15 or 31), Q6_K |d| 128 x 32 (d at byte 208, no dmin),
// IQ4_XS |d| 32 x 127 (no dmin); every weight's magnitude is at most that.
// One warp per row.
__global__ void row_exp_kq_kernel(const uint8_t* __restrict__ W, int n, int nsb, int sbb, int doff, float cd,
                                  float cm, int* __restrict__ erow) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;
  const uint8_t* base = W + (size_t)row * nsb * sbb;
  float m = 0.f;
  for (int b = lane; b < nsb; b += 32) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(base + (size_t)b * sbb + doff);  // 2-byte aligned
    const float d = fabsf(__half2float(__ushort_as_half(p[0])));
    const float dmin = cm != 0.f ? fabsf(__half2float(__ushort_as_half(p[1]))) : 0.f;
    m = fmaxf(m, d * cd + dmin * cm);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) {
    int e = 0;
    if (m > 0.f) e = 14 - ((int)((__float_as_uint(m) >> 23) & 0xFFu) - 127);
    erow[row] = e;
  }
}

// Per token row of X: the exponent e with max_j |x_j| 2^e in [2^14, 2^15)
// (clamped to [-126, 126]; 0 for a zero row), then X1 = fp16(x 2^e) and
// X2 = fp16(x 2^e - X1), both round to nearest even: X1 + X2 carries 22 of
// x's 24 bits. One CTA per row.
__global__ void __launch_bounds__(256) x_split_kernel(const float* __restrict__ X, int k, uint16_t* __restrict__ X1,
                                                      uint16_t* __restrict__ X2, int* __restrict__ etok) {
  // launched in plain stream order; the GEMM after it may start streaming
  // its weights at once
  grid_launch_dependents();
  const size_t row = blockIdx.x;
  const float4* x4 = reinterpret_cast<const float4*>(X + row * (size_t)k);
  const int k4 = k / 4;
  float m = 0.f;
  for (int i = threadIdx.x; i < k4; i += blockDim.x) {
    const float4 v = x4[i];
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[8];
  __shared__ int se;
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t = fmaxf(t, wm[i]);
    int e = 0;
    if (t > 0.f) e = 14 - ((int)((__float_as_uint(t) >> 23) & 0xFFu) - 127);
    e = e < -126 ? -126 : (e > 126 ? 126 : e);
    se = e;
    etok[row] = e;
  }
  __syncthreads();
  const float sc = __int_as_float((127 + se) << 23);
  uint2* y1 = reinterpret_cast<uint2*>(X1 + row * (size_t)k);
  uint2* y2 = reinterpret_cast<uint2*>(X2 + row * (size_t)k);
  for (int i = threadIdx.x; i < k4; i += blockDim.x) {
    const float4 v = x4[i];
    uint32_t a0, b0, a1, b1;
    split2(v.x * sc, v.y * sc, a0, b0);
    split2(v.z * sc, v.w * sc, a1, b1);
    y1[i] = make_uint2(a0, a1);
    y2[i] = make_uint2(b0, b1);
  }
}

// The exact leg's k splits added in split order (fp32), plus the residual:
// Y[t][i] = sum_z P[z][t][i] (+ R[t][i]); P dense [ks][T][n]. R may be Y.
__global__ void xs_reduce_kernel(const float* __restrict__ P, int ks, int T, int n, float* Y, int ldy, const float* R) {
  const size_t total = (size_t)T * n;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    float v = P[idx];
    for (int z = 1; z < ks; ++z) v += P[(size_t)z * total + idx];
    const size_t t = idx / (size_t)n, i = idx - t * (size_t)n;
    const size_t o = t * (size_t)ldy + i;
    if (R) v += R[o];
    Y[o] = v;
  }
}

// Independent k splits of the exact leg (at most 4, at least one 256-k chunk
// each) when its 128 x 128 tiles leave most SMs idle: as many as keep the
// grid within one wave.
int xs_ksplit(int n, int k, int T) {
  const long ctas = (long)((n + BM - 1) / BM) * ((T + 127) / 128);
  long ks = ctas > 0 ? (long)num_sms() / ctas : 1;
  if (ks > 4) ks = 4;
  if (ks > k / CHUNK) ks = k / CHUNK;
  return ks < 1 ? 1 : (int)ks;
}

template <int QT>
int launch_xs(const void* W, const void* Wu, int n, int k, const uint16_t* X1, const uint16_t* X2, const int* erow,
              const int* etok, int T, float* Y, int ldy, const float* R, unsigned* status, cudaStream_t s, char* msg,
              size_t msg_len, int ks, float* part) {
  (void)Wu;
  const int xr = padded_x_rows(T);  // the split's scratch holds that many rows
  if (ks > 1) {  // independent k splits into dense partials, then their sum (and R) into Y
    if (launch_cfg<QT, kEpiPlain, 128, true>(W, Wu, n, k, X1, T, part, n, nullptr, status, s, msg, msg_len, ks,
                                              kEarlyW | 32, xr, X2, erow, etok))
      return -1;
    const size_t total = (size_t)T * n;
    size_t blocks = (total + 255) / 256;
    if (blocks > (size_t)num_sms() * 8) blocks = (size_t)num_sms() * 8;
    xs_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(part, ks, T, n, Y, ldy, R);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      snprintf(msg, msg_len, "exact-leg split sum: %s", cudaGetErrorString(e));
      return -1;
    }
    return 0;
  }
  if (R)
    return launch_cfg<QT, kEpiResidual, 128, true>(W, Wu, n, k, X1, T, Y, ldy, R, status, s, msg, msg_len, 1, kEarlyW,
                                                    xr, X2, erow, etok);
  return launch_cfg<QT, kEpiPlain, 128, true>(W, Wu, n, k, X1, T, Y, ldy, R, status, s, msg, msg_len, 1, kEarlyW, xr,
                                               X2, erow, etok);
}

// y = silu(g) * u, silu(g) = g / (1 + e^-g), for T rows of n (rows of Y ldy
// apart; G and U dense); the exact leg's gate/up product from its two GEMMs.
__global__ void swiglu_rows_kernel(const float* __restrict__ G, const float* __restrict__ U, int T, int n, float* Y,
                                   int ldy) {
  const size_t total = (size_t)T * n;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / n, c = i - t * n;
    const float g = G[i];
    Y[t * ldy + c] = g / (1.0f + expf(-g)) * U[i];
  }
}

}  // namespace

cudaError_t launch_swiglu_rows(const float* G, const float* U, int T, int n, float* Y, int ldy, cudaStream_t s) {
  const size_t total = (size_t)T * n;
  size_t blocks = (total + 255) / 256;
  const size_t cap = (size_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  swiglu_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(G, U, T, n, Y, ldy);
  return cudaGetLastError();
}

size_t gemm_xs_scratch_bytes(int n, int k, int T, bool swiglu) {
  const size_t xb = ((size_t)padded_x_rows(T) * k * 2 + 255) & ~(size_t)255;
  const size_t base =
      2 * xb + (((size_t)T * 4 + 255) & ~(size_t)255) + (((size_t)(swiglu ? 2 : 1) * n * 4 + 255) & ~(size_t)255);
  const int ks = xs_ksplit(n, k, T);
  return base + (ks > 1 ? (size_t)ks * T * n * 4 : 0);  // the splits' partial outputs
}

int launch_gemm_xs(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                   const float* R, void* scratch, unsigned* status, cudaStream_t s, char* msg, size_t msg_len) {
  const size_t xb = ((size_t)padded_x_rows(T) * k * 2 + 255) & ~(size_t)255;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  uint16_t* X1 = reinterpret_cast<uint16_t*>(base);
  uint16_t* X2 = reinterpret_cast<uint16_t*>(base + xb);
  int* etok = reinterpret_cast<int*>(base + 2 * xb);
  int* erow = reinterpret_cast<int*>(base + 2 * xb + (((size_t)T * 4 + 255) & ~(size_t)255));
  // the k splits' partial outputs, after the exponents (the layout of
  // gemm_xs_scratch_bytes with swiglu = Wu != nullptr)
  const int ks = xs_ksplit(n, k, T);
  float* part = reinterpret_cast<float*>(base + 2 * xb + (((size_t)T * 4 + 255) & ~(size_t)255) +
                                         (((size_t)(Wu ? 2 : 1) * n * 4 + 255) & ~(size_t)255));
  const int bb = block_bytes(qtype);
  const float qmax = qtype == kQ4_0 ? 8.f : 128.f;
  // plain stream order: the splits start once everything before is complete
  const unsigned rblocks = (unsigned)((n + 7) / 8);
  if (qtype == kF16) {
    row_exp_f16_kernel<<<rblocks, 256, 0, s>>>(static_cast<const uint16_t*>(W), n, k, erow);
    if (Wu) row_exp_f16_kernel<<<rblocks, 256, 0, s>>>(static_cast<const uint16_t*>(Wu), n, k, erow + n);
  } else if (kquant(qtype)) {
    const int sbb = qtype == kQ4_K ? 144 : (qtype == kQ5_K ? 176 : (qtype == kQ6_K ? 210 : 136));
    const int doff = qtype == kQ6_K ? 208 : 0;
    const float cd = qtype == kQ4_K   ? 63.f * 15.f
                     : qtype == kQ5_K ? 63.f * 31.f
                     : qtype == kQ6_K ? 128.f * 32.f
                                      : 32.f * 127.f;  // IQ4_XS: |ls - 32| <= 32, |book| <= 127
    const float cm = qtype == kQ4_K || qtype == kQ5_K ? 63.f : 0.f;
    row_exp_kq_kernel<<<rblocks, 256, 0, s>>>(static_cast<const uint8_t*>(W), n, k / 256, sbb, doff, cd, cm, erow);
    if (Wu)
      row_exp_kq_kernel<<<rblocks, 256, 0, s>>>(static_cast<const uint8_t*>(Wu), n, k / 256, sbb, doff, cd, cm,
                                                erow + n);
  } else {
    row_exp_kernel<<<rblocks, 256, 0, s>>>(static_cast<const uint8_t*>(W), n, k / 32, bb, qmax, erow);
    if (Wu) row_exp_kernel<<<rblocks, 256, 0, s>>>(static_cast<const uint8_t*>(Wu), n, k / 32, bb, qmax, erow + n);
  }
  x_split_kernel<<<(unsigned)T, 256, 0, s>>>(X, k, X1, X2, etok);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, msg_len, "exact-leg splits: %s", cudaGetErrorString(e));
    return -1;
  }
  if (qtype == kF16) return launch_xs<kF16>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks,
                                           part);
  if (qtype == kQ4_K) return launch_xs<kQ4_K>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks,
                                           part);
  if (qtype == kQ5_K) return launch_xs<kQ5_K>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks,
                                           part);
  if (qtype == kQ6_K) return launch_xs<kQ6_K>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks,
                                           part);
  if (qtype == kIQ4_XS)
    return launch_xs<kIQ4_XS>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks, part);
  return qtype == kQ4_0
             ? launch_xs<kQ4_0>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks, part)
             : launch_xs<kQ8_0>(W, Wu, n, k, X1, X2, erow, etok, T, Y, ldy, R, status, s, msg, msg_len, ks, part);
}

cudaError_t launch_x_to_f16(const float* X, uint16_t* X16, size_t count, cudaStream_t s) {
  // the GEMM's shared-memory carveout, so that its CTAs may start on an SM
  // that still runs a conversion CTA
  static int carveout_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !carveout_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(x_to_f16_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    carveout_set[dev] = 1;
  }
  size_t blocks = (count / 8 + 255) / 256;
  if (blocks > (size_t)num_sms()) blocks = (size_t)num_sms();
  if (blocks == 0) blocks = 1;
  // plain stream order: launched programmatically after a GEMM, its CTAs
  // would sit beside that GEMM's for the GEMM's whole run (the GEMM lets the
  // next kernel launch at its start), which measured about 2 us slower per
  // call on GB300
  x_to_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(X, X16, count);
  return cudaGetLastError();
}

GemmPlan plan_gemm_tc(int n, int k, int T, bool swiglu) {
  GemmPlan pl;
  if (swiglu) {
    // a CTA pair per 256-token tile (one weight each) once a tile's second
    // half holds tokens; else one CTA per 128-token tile with both weights
    pl.pair = T > 128;
    return pl;
  }
  const int sms = num_sms();
  const long rt = (n + BM - 1) / BM, tiles256 = rt * ((T + 255) / 256), tiles192 = rt * ((T + 191) / 192);
  // 256-token tiles halve the MMA instructions per flop: taken when they
  // still keep most SMs busy, or, split over k in two, fit in one wave.
  // 192-token tiles instead when they need no more waves: each does three
  // quarters of the work and the SMs a 256-token grid leaves idle take the
  // rest. Measured on GB300 (k = 4096, Q4_0 / Q4_K): 6144 rows at T = 512
  // 24.5 / 31.2 us against 26.3 / 31.0 (96 tiles of 256 leave 56 SMs idle),
  // 12288 rows at T = 512 45.4 / 57.7 us against 51.3 / 59.0; at T = 2048
  // (7 waves of 192 against 6 of 256) 159.8 / 199.0 us against 154.9 / 178.6,
  // so there they are not taken
  if (10 * tiles256 >= 6L * sms) {
    const long w256 = (tiles256 + sms - 1) / sms, w192 = (tiles192 + sms - 1) / sms;
    pl.bn = T > 128 && w192 <= w256 ? 192 : 256;
  } else if (2 * tiles256 <= sms && k / CHUNK >= 2) {
    pl.bn = 256;
    pl.nsplit = 2;
  }
  return pl;
}

int launch_gemm_tc(const GemmPlan& pl, int qtype, const void* W, const void* Wu, int n, int k, const uint16_t* X16,
                   int T, float* Y, int ldy, const float* R, unsigned* status, cudaStream_t s, char* msg,
                   size_t msg_len, int early, int x_rows, const OutRegions* regions) {
  const int w = early;
  const OutRegions reg = regions ? *regions : OutRegions{nullptr, nullptr, 0, 0, 0, 0};
  if (qtype == kF16) return launch_q<kF16>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows,
                                          reg);
  if (qtype == kQ4_K) return launch_q<kQ4_K>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows,
                                          reg);
  if (qtype == kQ5_K) return launch_q<kQ5_K>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows,
                                          reg);
  if (qtype == kQ6_K) return launch_q<kQ6_K>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows,
                                          reg);
  if (qtype == kIQ4_XS)
    return launch_q<kIQ4_XS>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows, reg);
  return qtype == kQ4_0 ? launch_q<kQ4_0>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows, reg)
                        : launch_q<kQ8_0>(pl, W, Wu, n, k, X16, T, Y, ldy, R, status, s, msg, msg_len, w, x_rows, reg);
}

}  // namespace apr
