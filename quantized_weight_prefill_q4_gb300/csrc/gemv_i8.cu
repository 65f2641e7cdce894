// Single-token GEMV (T = 1) over Q4_0 / Q8_0 blocks and Q4_K / Q5_K / Q6_K /
// IQ4_XS superblocks with integer dot products, exact to fp32 level (the
// single-token GEMVs gemv_q4_0_pf / gemv_q8_0_pf of oxibonsai-kernels 0.1.4
// src/gpu_backend/cuda_q_std_prefill.rs, HBM-bound form). A superblock lane
// takes the 64 weights of one X block pair (Q4_K / Q5_K: one code group of a
// superblock, two 32-weight sub-blocks; Q6_K: one 64-weight stage, four
// 16-weight sub-blocks; IQ4_XS: two 32-weight sub-blocks, their codes looked
// up in the code book four at a time) and applies the sub-block scales, and
// for Q4_K / Q5_K the mins against the block's sum of X, after the integer
// sums.
//
// X in fixed point per 32-block: for block b, e_b makes max_j |x_j| 2^e_b lie
// in [2^21, 2^22), and X_j = rint(x_j 2^e_b) (a 23-bit integer, off by at most
// 1/2: 2^-22 of the block's largest |x|) is written with three signed byte
// digits, X_j = 2^16 p2 + 2^8 p1 + p0. A block's code-times-X sum is then
//   sum_j q'_j X_j = 2^16 A2 + 2^8 A1 + A0,   A_k = sum_j q'_j p_kj,
// each A_k an exact int32 of at most 2^17, accumulated four products at a
// time by dp4a. Q4_0 multiplies the unsigned nibbles n_j (dp4a.u32.s32) and
// starts A_k at -8 sum_j p_kj, so that A_k sums (n_j - 8) p_kj; Q8_0 multiplies
// the signed codes directly. The three A_k become one float (rounded once at
// fp32 level) and the row accumulates d_b 2^-e_b times it in fp32. Per weight
// element this is 3/4 dp4a and about 3/8 of an instruction to unpack the
// codes, against about two and a half for a decode to fp32 and an FMA.
//
// Work and data movement as the whole-row GEMV (gemv_rows.cu): persistent
// CTAs, one per SM, each a contiguous range of rows; a producer warp streams
// whole rows (the W rows then the Wu rows for gate/up) into a ring of
// 16 KB stages with one bulk copy per stage; consumer warps take the rows
// round-robin, each lane one block pair of a row, its X digits held in
// registers for the whole kernel. A warp decodes two rows at a time and
// reduces their lane partials with interleaved shuffles, and the partials of
// a row's warps are parked in shared memory and added once, after the last
// stage, in a fixed order: no per-row fence or atomic. Measured on GB300, a
// kernel that only streams the bytes reads 7.5 MB in 4.2 us and 27 MB in
// 8.2 us (1.8 and 3.3 TB/s: the launch's ramp-up and tail, not the HBM rate,
// bound weights of this size), and a deeper ring does not change that. So
// the CTA keeps to half an SM when it can (5 stages of 16 KB, the X table,
// 8 consumer warps at under 113 registers): the next launch's CTA then
// starts beside it and streams its weights while this one finishes. Rows of
// k above about 8192 (a larger X table) take a whole SM and a ring of up to
// 13 stages.
//
// Programmatic dependent launch: the producer streams W before the preceding
// kernel has finished (W must not be its output); X, R and Y are touched only
// after griddepcontrol.wait, and the kernel lets the next kernel launch once
// that wait has returned.

#include <cstdint>
#include <cuda_fp16.h>

#include "apr_internal.h"
#include "dev_common.cuh"
#include "host_common.h"
#include "iq4.cuh"
#include "q4k.cuh"

namespace apr {
namespace {

constexpr int ICW = 8;                         // consumer warps
constexpr int ITHREADS = 32 * (ICW + 1);
constexpr int ISTAGE = 16384;                  // bytes of one stage
constexpr int INS_MAX = 13;                    // stages at most (as many as shared memory holds)
// rows a CTA takes at most: the CTAs split the n rows evenly
__host__ __device__ inline int i8_rcap(int n, int grid) { return (n + grid - 1) / grid; }
constexpr int XBW = 28;                        // table words per block: 3 x 8 digit words, 3 starts, scale

__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The table entries of NB blocks, each built by 8 consecutive lanes (u =
// lane % 8), each lane from its 4 values of X (elements 4u .. 4u + 3 of the
// block): the block's largest |x| and the digit sums by shuffles within the 8
// lanes. The blocks' shuffle chains are interleaved (they are independent);
// out[i] == nullptr skips block i's stores (its shuffles still run: the 8-lane
// groups of a warp take part in every shuffle).
template <int QT, int NB>
__device__ __forceinline__ void block_digits8(const float4 (&x)[NB], int u, uint32_t* const (&out)[NB]) {
  float m[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) m[i] = fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)), fmaxf(fabsf(x[i].z), fabsf(x[i].w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1)
#pragma unroll
    for (int i = 0; i < NB; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
  uint32_t dig[NB][3];
  int psum[NB][3], e[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    int ei = 0;
    if (m[i] > 0.f) ei = 21 - ((int)((__float_as_uint(m[i]) >> 23) & 0xFFu) - 127);
    ei = ei < -126 ? -126 : (ei > 126 ? 126 : ei);
    e[i] = ei;
    const float sc = __int_as_float((127 + ei) << 23);
    const float xv[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
    for (int kd = 0; kd < 3; ++kd) {
      dig[i][kd] = 0u;
      psum[i][kd] = 0;
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int X = __float2int_rn(xv[b] * sc);
      const int p0 = (X << 24) >> 24;
      const int x1 = (X - p0) >> 8;
      const int p1 = (x1 << 24) >> 24;
      const int p2 = (x1 - p1) >> 8;
      dig[i][0] |= (uint32_t)(p0 & 0xFF) << (8 * b);
      dig[i][1] |= (uint32_t)(p1 & 0xFF) << (8 * b);
      dig[i][2] |= (uint32_t)(p2 & 0xFF) << (8 * b);
      psum[i][0] += p0;
      psum[i][1] += p1;
      psum[i][2] += p2;
    }
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1)
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
      for (int kd = 0; kd < 3; ++kd) psum[i][kd] += __shfl_xor_sync(0xffffffffu, psum[i][kd], o);
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    if (!out[i]) continue;
#pragma unroll
    for (int kd = 0; kd < 3; ++kd) out[i][8 * kd + u] = dig[i][kd];
    if (u == 0) {
      if constexpr (QT == kQ4_K || QT == kQ5_K) {
        // the block's sum of X_j (an integer below 2^27, rounded to float)
        // for the dmin m term; no start values
        out[i][24] = __float_as_uint((float)(65536 * psum[i][2] + 256 * psum[i][1] + psum[i][0]));
        out[i][25] = 0u;
        out[i][26] = 0u;
      } else {
#pragma unroll
        for (int kd = 0; kd < 3; ++kd) out[i][24 + kd] = (uint32_t)(QT == kQ4_0 ? -8 * psum[i][kd] : 0);
      }
      out[i][27] = __float_as_uint(__int_as_float((127 - e[i]) << 23));  // 2^-e
    }
  }
}

// sum over one block of q'_j x_j, times d: t = the block's table entry
// (registers), p = its 4 (Q4_0: 16 bytes of nibbles) or 8 (Q8_0) payload words.
template <int QT>
__device__ __forceinline__ float block_dot(const uint32_t* p, const uint32_t (&t)[XBW], float d) {
  int a0 = (int)t[24], a1 = (int)t[25], a2 = (int)t[26];
  if constexpr (QT == kQ4_0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = p[i] & 0x0F0F0F0Fu;          // elements 4i .. 4i + 3
      const uint32_t hi = (p[i] >> 4) & 0x0F0F0F0Fu;   // elements 16 + 4i ..
      a0 = dp4a_us(lo, (int)t[i], a0);
      a1 = dp4a_us(lo, (int)t[8 + i], a1);
      a2 = dp4a_us(lo, (int)t[16 + i], a2);
      a0 = dp4a_us(hi, (int)t[4 + i], a0);
      a1 = dp4a_us(hi, (int)t[12 + i], a1);
      a2 = dp4a_us(hi, (int)t[20 + i], a2);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a0 = dp4a_ss(p[i], (int)t[i], a0);
      a1 = dp4a_ss(p[i], (int)t[8 + i], a1);
      a2 = dp4a_ss(p[i], (int)t[16 + i], a2);
    }
  }
  const float v = fmaf((float)a2, 65536.f, fmaf((float)a1, 256.f, (float)a0));
  return v * (d * __uint_as_float(t[27]));
}

// Q4_K / Q5_K: the sum over a lane's 64 weights (group g of a superblock:
// sub-block 2 g in the low nibbles of its 32 code bytes, 2 g + 1 in the high
// ones; X blocks A and B). w[0] = d | dmin << 16, w[1..3] the packed scales,
// (Q5_K) w[4..11] the fifth-bit bytes, then the group's 8 code words. For
// each sub-block sum_j w_j x_j = 2^-e (d sc sum_j q_j X_j - dmin m sum_j X_j),
// with the digit sums of q_j X_j exact in int32 (dp4a of the unsigned codes)
// and the products and the difference rounded at fp32 level.
template <int QT>
__device__ __forceinline__ float kq_pair_dot(const uint32_t* w, uint32_t g, const uint32_t (&ta)[XBW],
                                             const uint32_t (&tb)[XBW]) {
  constexpr bool FIVE = QT == kQ5_K;
  constexpr int CW = FIVE ? 12 : 4;  // first code word
  const float d = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half((unsigned short)(w[0] >> 16)));
  uint32_t scA, mA, scB, mB;
  const uint32_t sw[3] = {w[1], w[2], w[3]};
  q4k_scale_min_w(sw, 2 * g, scA, mA);
  q4k_scale_min_w(sw, 2 * g + 1, scB, mB);
  int a0 = 0, a1 = 0, a2 = 0, b0 = 0, b1 = 0, b2 = 0;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    uint32_t lo = w[CW + v] & 0x0F0F0F0Fu, hi = (w[CW + v] >> 4) & 0x0F0F0F0Fu;
    if constexpr (FIVE) {  // the fifth bits: bit 2 g (low) and 2 g + 1 (high) of each byte
      lo |= ((w[4 + v] >> (2 * g)) & 0x01010101u) << 4;
      hi |= ((w[4 + v] >> (2 * g + 1)) & 0x01010101u) << 4;
    }
    a0 = dp4a_us(lo, (int)ta[v], a0);
    a1 = dp4a_us(lo, (int)ta[8 + v], a1);
    a2 = dp4a_us(lo, (int)ta[16 + v], a2);
    b0 = dp4a_us(hi, (int)tb[v], b0);
    b1 = dp4a_us(hi, (int)tb[8 + v], b1);
    b2 = dp4a_us(hi, (int)tb[16 + v], b2);
  }
  const float vA = fmaf((float)a2, 65536.f, fmaf((float)a1, 256.f, (float)a0));
  const float vB = fmaf((float)b2, 65536.f, fmaf((float)b1, 256.f, (float)b0));
  const float sA = fmaf(d * (float)scA, vA, -(dmin * (float)mA) * __uint_as_float(ta[24]));
  const float sB = fmaf(d * (float)scB, vB, -(dmin * (float)mB) * __uint_as_float(tb[24]));
  return fmaf(sA, __uint_as_float(ta[27]), sB * __uint_as_float(tb[27]));
}

// Q6_K: the sum over a lane's 64 weights (stage g of a superblock, X blocks A
// and B), from shared-memory words that start at the word holding the
// superblock's first byte, sh bytes (0 or 2) into it: w[0..16] over the low
// nibble bytes 64 h .. (h = g / 2), w[17..25] over the high-bit bytes 128 +
// 32 h .., w[26..27] over the scale bytes 192 + 4 g .., w[28] the word holding
// d. The codes are centred to q - 32 as signed bytes, so each 16-weight
// sub-block is d sc_j 2^-e sum (q - 32) X, its digit sums exact in int32.
__device__ __forceinline__ float q6k_pair_dot(const uint32_t* w, uint32_t g, uint32_t sh, const uint32_t (&ta)[XBW],
                                              const uint32_t (&tb)[XBW]) {
  const uint32_t s8 = 8 * sh;
  auto at = [&](int m) { return __funnelshift_r(w[m], w[m + 1], s8); };
  const float d = __half2float(__ushort_as_half((unsigned short)((w[28] >> s8) & 0xFFFFu)));
  const uint32_t scw = at(26);
  const uint32_t nib = 4 * (g & 1u), hb = 4 * (g & 1u);
  int acc[4][3];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = 0;
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    const uint32_t q = ((at(v) >> nib) & 0x0F0F0F0Fu) | (((at(17 + (v & 7)) >> (hb + 2 * (v >> 3))) & 0x03030303u) << 4);
    // q - 32 in each byte: (q | 0x80) - 0x20 cannot borrow, and ^ 0x80 makes it signed
    const uint32_t c = ((q | 0x80808080u) - 0x20202020u) ^ 0x80808080u;
    const uint32_t (&t)[XBW] = v < 8 ? ta : tb;
    const int j = v >> 2, u = v & 7;
    acc[j][0] = dp4a_ss(c, (int)t[u], acc[j][0]);
    acc[j][1] = dp4a_ss(c, (int)t[8 + u], acc[j][1]);
    acc[j][2] = dp4a_ss(c, (int)t[16 + u], acc[j][2]);
  }
  float r = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float v = fmaf((float)acc[j][2], 65536.f, fmaf((float)acc[j][1], 256.f, (float)acc[j][0]));
    const float sc = (float)((int)(scw << (24 - 8 * j)) >> 24);
    r = fmaf(d * sc * __uint_as_float((j < 2 ? ta : tb)[27]), v, r);
  }
  return r;
}

// IQ4_XS: the sum over a lane's 64 weights (stage g of a superblock:
// sub-blocks 2 g and 2 g + 1, X blocks A and B). w[0] = d | high scale bits
// << 16, w[1] the low scale nibbles, w[2..9] the stage's code words. The book
// lookup gives each word's codes as (A0, B0, A1, B1) and (A2, B2, A3, B3)
// (A_i: element 4 v + i, B_i: 16 + 4 v + i), signed bytes book[c], and the X
// digit words of IQ4_XS lanes were put in that order when the table was
// loaded (words 2 v and 2 v + 1 of each digit plane), so each sub-block is
// d (ls - 32) 2^-e sum book[c] X with its digit sums exact in int32.
__device__ __forceinline__ float iq4_pair_dot(const uint32_t* w, uint32_t g, const uint32_t (&ta)[XBW],
                                              const uint32_t (&tb)[XBW]) {
  const float d = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
  int acc[2][3];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t (&t)[XBW] = h ? tb : ta;
    acc[h][0] = acc[h][1] = acc[h][2] = 0;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t u0, u1;
      iq4_word(w[2 + 4 * h + v], u0, u1);
      u0 ^= 0x80808080u;  // book[c] + 128 to the signed byte book[c]
      u1 ^= 0x80808080u;
#pragma unroll
      for (int kd = 0; kd < 3; ++kd) {
        acc[h][kd] = dp4a_ss(u0, (int)t[8 * kd + 2 * v], acc[h][kd]);
        acc[h][kd] = dp4a_ss(u1, (int)t[8 * kd + 2 * v + 1], acc[h][kd]);
      }
    }
  }
  const float vA = fmaf((float)acc[0][2], 65536.f, fmaf((float)acc[0][1], 256.f, (float)acc[0][0]));
  const float vB = fmaf((float)acc[1][2], 65536.f, fmaf((float)acc[1][1], 256.f, (float)acc[1][0]));
  const float sA = d * (float)iq4_scale(w[0], w[1], 2 * g) * __uint_as_float(ta[27]);
  const float sB = d * (float)iq4_scale(w[0], w[1], 2 * g + 1) * __uint_as_float(tb[27]);
  return fmaf(sA, vA, sB * vB);
}

// The X digit words of a block in the order of the IQ4_XS lookup's bytes:
// word 2 v of a plane = (x_4v, x_16+4v, x_4v+1, x_17+4v), word 2 v + 1 =
// (x_4v+2, x_18+4v, x_4v+3, x_19+4v)
__device__ __forceinline__ void iq4_order_table(uint32_t (&t)[XBW]) {
#pragma unroll
  for (int kd = 0; kd < 3; ++kd) {
    uint32_t o[8];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      o[2 * v] = __byte_perm(t[8 * kd + v], t[8 * kd + 4 + v], 0x5140);
      o[2 * v + 1] = __byte_perm(t[8 * kd + v], t[8 * kd + 4 + v], 0x7362);
    }
#pragma unroll
    for (int v = 0; v < 8; ++v) t[8 * kd + v] = o[v];
  }
}

int rows_per_stage(int qtype, int k, bool swiglu) {
  const long row_bytes = (long)row_bytes_of(qtype, k);
  return (int)(ISTAGE / ((swiglu ? 2 : 1) * row_bytes));
}

// NT tokens (1 or 2): with two, one CTA an SM (the two tokens' digit tables
// stay in registers), X rows k apart, Y and R rows ldy apart.
template <int QT, bool SWI, int NT>
__global__ void __launch_bounds__(ITHREADS, NT == 1 ? 2 : 1)
    gemv_i8_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ Wu, int n, int k,
                   const float* __restrict__ X, float* Y, const float* R, unsigned* status, int rs, int ns,
                   int ldy) {
  constexpr int NM = SWI ? 2 : 1;
  constexpr bool KQ = QT == kQ4_K || QT == kQ5_K || QT == kQ6_K || QT == kIQ4_XS;
  constexpr int BB = QT == kQ4_0 ? 18 : 34;  // block formats
  constexpr int SBB = QT == kQ4_K ? 144 : (QT == kQ5_K ? 176 : (QT == kQ6_K ? 210 : 136));  // superblocks
  constexpr int PW_WORDS = 2 * BB / 4;                                // words of one block pair
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int nblk = k / 32, npk = nblk / 2;
  const int PW = (npk + 31) / 32;  // warps per row
  uint32_t* xt = reinterpret_cast<uint32_t*>(smem + (size_t)ns * ISTAGE);  // X tables, [NT][nblk][XBW]
  const int rcap = i8_rcap(n, gridDim.x);
  float* part = reinterpret_cast<float*>(xt + (size_t)NT * nblk * XBW);  // [row slot][NM][NT][PW]
  float* rres = part + (((size_t)rcap * NM * NT * PW + 1) & ~(size_t)1);  // [NT][row slot] residuals
  uint64_t* bars = reinterpret_cast<uint64_t*>(rres + ((NT * rcap + 1) & ~1));
  uint64_t* full = bars;
  uint64_t* empty = bars + INS_MAX;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * INS_MAX);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row_bytes = KQ ? (size_t)(k / 256) * SBB : (size_t)nblk * BB;
  const int r0 = (int)((long)n * blockIdx.x / gridDim.x);
  const int r1 = (int)((long)n * (blockIdx.x + 1) / gridDim.x);
  const int nst = (r1 - r0 + rs - 1) / rs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], ICW);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == ICW) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      int last[INS_MAX];
      for (int i = 0; i < INS_MAX; ++i) last[i] = -1;
      bool ok = true;
      for (int s = 0; s < nst && ok; ++s) {
        const int st = s % ns;
        ok = mbar_wait(&empty[st], ((s / ns) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        const int rb = r0 + s * rs, rows = min(rs, r1 - rb);
        const uint32_t bytes = (uint32_t)(rows * row_bytes);
        mbar_arrive_expect_tx(&full[st], bytes * NM);
        bulk_load_1d(smem + st * ISTAGE, W + (size_t)rb * row_bytes, bytes, &full[st]);
        if (SWI) bulk_load_1d(smem + st * ISTAGE + rs * row_bytes, Wu + (size_t)rb * row_bytes, bytes, &full[st]);
        last[st] = s;
      }
      if (!ok)  // let the copies in flight land before the CTA exits
        for (int i = 0; i < ns; ++i)
          if (last[i] >= 0) mbar_wait(&full[i], (last[i] / ns) & 1, abort_flag + 1, status);
    }
    return;
  }

  // ------------------------------------------------ consumers
  const int RG = ICW / PW;          // row groups
  const int g = warp / PW, wi = warp % PW;
  const int P = wi * 32 + lane;     // this lane's block pair
  const bool act = g < RG && P < npk;

  // X, R and Y may belong to the preceding kernel until it completes; once it
  // has, the next kernel may launch
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  // 8 lanes a block, 32 blocks a pass of the consumers (nblk is a multiple of
  // 8, so a warp's 4 blocks of a pass are all present or all absent); the X
  // loads of four passes are issued before any is used
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) {
    const float4* x4 = reinterpret_cast<const float4*>(X + (size_t)tk * k);
    uint32_t* xtt = xt + (size_t)tk * nblk * XBW;
    for (int base = (int)threadIdx.x / 8; base < nblk; base += 4 * (ICW * 32 / 8)) {
      float4 xv[4];
      uint32_t* dst[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int b0 = base + u * (ICW * 32 / 8);
        xv[u] = b0 < nblk ? __ldg(x4 + (size_t)b0 * 8 + (threadIdx.x & 7)) : make_float4(0.f, 0.f, 0.f, 0.f);
        dst[u] = b0 < nblk ? xtt + (size_t)b0 * XBW : nullptr;
      }
      block_digits8<QT, 4>(xv, threadIdx.x & 7, dst);
    }
  }
  if (!SWI && R)
#pragma unroll
    for (int tk = 0; tk < NT; ++tk)
      for (int i = threadIdx.x; i < r1 - r0; i += ICW * 32) rres[tk * rcap + i] = R[(size_t)tk * ldy + r0 + i];
  named_sync(1, ICW * 32);
  uint32_t ta[NT][XBW], tb[NT][XBW];
  if (act) {
#pragma unroll
    for (int tk = 0; tk < NT; ++tk) {
      const uint4* src = reinterpret_cast<const uint4*>(xt + ((size_t)tk * nblk + 2 * P) * XBW);
#pragma unroll
      for (int v = 0; v < XBW / 4; ++v) {
        const uint4 a = src[v], b = src[XBW / 4 + v];
        ta[tk][4 * v] = a.x; ta[tk][4 * v + 1] = a.y; ta[tk][4 * v + 2] = a.z; ta[tk][4 * v + 3] = a.w;
        tb[tk][4 * v] = b.x; tb[tk][4 * v + 1] = b.y; tb[tk][4 * v + 2] = b.z; tb[tk][4 * v + 3] = b.w;
      }
      if constexpr (QT == kIQ4_XS) {
        iq4_order_table(ta[tk]);
        iq4_order_table(tb[tk]);
      }
    }
  }

  // one row's partials of this lane (its block pair), weight m, one a token
  auto row_part = [&](int st, int m, int rr, float (&res)[NT]) {
#pragma unroll
    for (int tk = 0; tk < NT; ++tk) res[tk] = 0.f;
    if (!act) return;
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(smem + st * ISTAGE + (size_t)(m * rs + rr) * row_bytes);
    if constexpr (QT == kQ6_K) {
      // superblock P / 4 from the word holding its first byte (2 (P / 4 mod
      // 2) bytes into it: rows start on 16-byte boundaries); stage P mod 4
      const uint32_t* w = rw + (((uint32_t)P >> 2) * 210u >> 2);
      const int h = (P & 3) >> 1;
      uint32_t wq[29];
#pragma unroll
      for (int v = 0; v < 17; ++v) wq[v] = w[16 * h + v];
#pragma unroll
      for (int v = 0; v < 9; ++v) wq[17 + v] = w[32 + 8 * h + v];
      wq[26] = w[48 + (P & 3)];
      wq[27] = w[49 + (P & 3)];
      wq[28] = w[52];
#pragma unroll
      for (int tk = 0; tk < NT; ++tk)
        res[tk] = q6k_pair_dot(wq, (uint32_t)P & 3u, 2u * (((uint32_t)P >> 2) & 1u), ta[tk], tb[tk]);
      return;
    } else if constexpr (QT == kIQ4_XS) {
      // superblock P / 4 (34 words, rows on 16-byte boundaries): header words,
      // then stage P mod 4's 8 code words
      const uint32_t* w = rw + ((uint32_t)P >> 2) * 34u;
      uint32_t wq[10];
      wq[0] = w[0];
      wq[1] = w[1];
#pragma unroll
      for (int v = 0; v < 8; ++v) wq[2 + v] = w[2 + 8 * (P & 3) + v];
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) res[tk] = iq4_pair_dot(wq, (uint32_t)P & 3u, ta[tk], tb[tk]);
      return;
    } else if constexpr (KQ) {
      // superblock P / 4: header and scales, (Q5_K) fifth bits, then group P mod 4's codes
      constexpr int CW = QT == kQ5_K ? 12 : 4;
      const uint32_t* w = rw + ((uint32_t)P >> 2) * (SBB / 4);
      uint32_t wq[CW + 8];
#pragma unroll
      for (int v = 0; v < CW; ++v) wq[v] = w[v];
#pragma unroll
      for (int v = 0; v < 8; ++v) wq[CW + v] = w[CW + 8 * (P & 3) + v];
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) res[tk] = kq_pair_dot<QT>(wq, (uint32_t)P & 3u, ta[tk], tb[tk]);
      return;
    }
    const uint32_t* w = rw + P * PW_WORDS;
    uint32_t wr[PW_WORDS];
#pragma unroll
    for (int i = 0; i < PW_WORDS; ++i) wr[i] = w[i];
    uint32_t pa[QT == kQ4_0 ? 4 : 8];
    if constexpr (QT == kQ4_0) {
      // block A: d in bytes 0-1, nibbles 2..17; block B: d in 18-19, nibbles 20..35
#pragma unroll
      for (int i = 0; i < 4; ++i) pa[i] = __byte_perm(wr[i], wr[i + 1], 0x5432);
      const float dA = __half2float(__ushort_as_half((unsigned short)(wr[0] & 0xFFFFu)));
      const float dB = __half2float(__ushort_as_half((unsigned short)(wr[4] >> 16)));
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) res[tk] = block_dot<QT>(pa, ta[tk], dA) + block_dot<QT>(wr + 5, tb[tk], dB);
    } else {
      // block A: d in bytes 0-1, codes 2..33; block B: d in 34-35, codes 36..67
#pragma unroll
      for (int i = 0; i < 8; ++i) pa[i] = __byte_perm(wr[i], wr[i + 1], 0x5432);
      const float dA = __half2float(__ushort_as_half((unsigned short)(wr[0] & 0xFFFFu)));
      const float dB = __half2float(__ushort_as_half((unsigned short)(wr[8] >> 16)));
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) res[tk] = block_dot<QT>(pa, ta[tk], dA) + block_dot<QT>(wr + 9, tb[tk], dB);
    }
  };

  bool ok = true;
  for (int s = 0; s < nst; ++s) {
    const int st = s % ns;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (s / ns) & 1, abort_flag, status));
    if (!ok) break;
    const int rb = r0 + s * rs, rows = min(rs, r1 - rb);
    if (g < RG) {
      // the stage's rows whose index within the CTA is g modulo RG, two at a time
      for (int rr = ((g - (rb - r0)) % RG + RG) % RG; rr < rows; rr += 2 * RG) {
        const bool two = rr + RG < rows;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          float a[NT], b[NT];
          row_part(st, m, rr, a);
          if (two) {
            row_part(st, m, rr + RG, b);
          } else {
#pragma unroll
            for (int tk = 0; tk < NT; ++tk) b[tk] = 0.f;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int tk = 0; tk < NT; ++tk) {
              a[tk] += __shfl_xor_sync(0xffffffffu, a[tk], o);
              b[tk] += __shfl_xor_sync(0xffffffffu, b[tk], o);
            }
          // the warp's share of the row, added with the others' after the
          // last stage
          if (lane == 0)
#pragma unroll
            for (int tk = 0; tk < NT; ++tk) {
              part[(((rb + rr - r0) * NM + m) * NT + tk) * PW + wi] = a[tk];
              if (two) part[(((rb + rr + RG - r0) * NM + m) * NT + tk) * PW + wi] = b[tk];
            }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage's rows
  }
  // every row's warp shares are in shared memory: add them in warp order
  named_sync(1, ICW * 32);
  if (ok)
    for (int slot = threadIdx.x; slot < r1 - r0; slot += ICW * 32)
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) {
        float acc[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          float v = 0.f;
          for (int w2 = 0; w2 < PW; ++w2) v += part[((slot * NM + m) * NT + tk) * PW + w2];
          acc[m] = v;
        }
        float y;
        if (SWI) {
          y = acc[0] / (1.0f + expf(-acc[0])) * acc[NM - 1];
        } else {
          y = acc[0] + (R ? rres[tk * rcap + slot] : 0.f);
        }
        Y[(size_t)tk * ldy + r0 + slot] = y;
      }
}

// shared memory besides the ring (the nt tokens' X tables, the row partials
// [rows][2 weights at most][nt][warps a row], the residuals, the barriers)
// for a grid of `grid` CTAs, and the stages that fit beside it
size_t i8_fixed_smem_grid(int k, int n, int grid, int nt) {
  const size_t rcap = (size_t)i8_rcap(n, grid), pw = (size_t)((k / 64 + 31) / 32);
  return 128 + (size_t)nt * (k / 32) * XBW * 4 + ((rcap * 2 * nt * pw + 1) & ~(size_t)1) * 4 +
         ((nt * rcap + 1) & ~(size_t)1) * 4 + 2 * INS_MAX * 8 + 16;
}
int i8_stages_for(int k, int n, int grid, int nt) {
  // one token: two CTAs an SM (228 KB of shared memory, 1 KB reserved per
  // CTA) when 5 stages fit beside the X table, else one with as many as fit;
  // two tokens: one CTA an SM
  if (nt == 1) {
    const long half = 232448L / 2 - 1024 - (long)i8_fixed_smem_grid(k, n, grid, 1);
    if (half / ISTAGE >= 5) return 5;
  }
  const long ns = (232448L - (long)i8_fixed_smem_grid(k, n, grid, nt)) / ISTAGE;
  return (int)(ns < INS_MAX ? ns : INS_MAX);
}
// One token: one CTA an SM (half of one when it fits, so that the next
// launch's CTAs start beside it), or, for weights of 16 MiB and more when the
// half-SM form fits them, two half-SM CTAs an SM: twice the consumer warps to
// hide the latency of the dot products' dependent chains, which bound larger
// weights (measured on GB300 with a 49152 x 4096 Q4_0 weight: 2 warps a
// scheduler issuing 45 % of cycles, stalled mostly on fixed-latency
// dependencies, while the same launch shape only streaming the bytes reaches
// the HBM rate). Two CTAs an SM measured faster from about 16 MiB (Q4_0
// 8192 x 4096: 8.0 -> 7.6 us, Q8_0 4096 x 4096: 7.8 -> 7.2, 12288 x 4096:
// 17.3 -> 13.5) and slower below, where the next launch's start beside this
// one counts for more (Q4_0 / Q4_K 4096 x 4096: 5.4 -> 5.5, 6.3 -> 6.5 us).
// Two tokens: one CTA an SM.
int i8_grid(int qtype, int k, int n, int nt) {
  const int sms = num_sms();
  if (n < sms) return n;
  if (nt == 1 && (double)n * (double)row_bytes_of(qtype, k) >= 16.0 * 1048576.0 &&
      i8_stages_for(k, n, 2 * sms, 1) == 5)
    return 2 * sms;
  return sms;
}
int i8_stages(int qtype, int k, int n, int nt) { return i8_stages_for(k, n, i8_grid(qtype, k, n, nt), nt); }
size_t i8_smem(int qtype, int k, int n, int nt) {
  return i8_fixed_smem_grid(k, n, i8_grid(qtype, k, n, nt), nt) + (size_t)i8_stages(qtype, k, n, nt) * ISTAGE;
}

template <int QT, bool SWI, int NT>
cudaError_t launch_i8(const void* W, const void* Wu, int n, int k, const float* X, float* Y, int ldy, const float* R,
                      unsigned* status, cudaStream_t s) {
  const size_t smem = i8_smem(QT, k, n, NT);
  auto kern = gemv_i8_kernel<QT, SWI, NT>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)i8_grid(QT, k, n, NT));
  cfg.blockDim = dim3(ITHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, (const uint8_t*)W, (const uint8_t*)Wu, n, k, X, Y, R, status,
                         rows_per_stage(QT, k, SWI), i8_stages(QT, k, n, NT), ldy);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e;
}

template <int QT, bool SWI>
cudaError_t launch_i8_t(const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                        const float* R, unsigned* status, cudaStream_t s) {
  return T == 2 ? launch_i8<QT, SWI, 2>(W, Wu, n, k, X, Y, ldy, R, status, s)
                : launch_i8<QT, SWI, 1>(W, Wu, n, k, X, Y, ldy, R, status, s);
}

// The GEMV's data movement alone: each CTA streams its contiguous share of
// `bytes` into a ring of 16 KB stages by bulk copies, exactly as the GEMV's
// producer does, and the consumer warps only release the stages. A measured
// reference for the GEMV's roofline; nothing is computed or written.
__global__ void __launch_bounds__(ITHREADS, 2) read_stream_kernel(const uint8_t* __restrict__ src, long long bytes,
                                                                  unsigned* status, int ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)ns * ISTAGE);
  uint64_t* empty = full + INS_MAX;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + INS_MAX);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long units = bytes / 16;  // 16-byte units, split evenly over the CTAs
  const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
  const long long my = (u1 - u0) * 16;
  const int nst = (int)((my + ISTAGE - 1) / ISTAGE);
  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], ICW);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == ICW) {
    if (lane == 0) {
      int last[INS_MAX];
      for (int i = 0; i < INS_MAX; ++i) last[i] = -1;
      bool ok = true;
      for (int s = 0; s < nst && ok; ++s) {
        const int st = s % ns;
        ok = mbar_wait(&empty[st], ((s / ns) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        const long long off = (long long)s * ISTAGE;
        const uint32_t b = (uint32_t)(my - off < ISTAGE ? my - off : ISTAGE);
        mbar_arrive_expect_tx(&full[st], b);
        bulk_load_1d(smem + st * ISTAGE, src + u0 * 16 + off, b, &full[st]);
        last[st] = s;
      }
      if (!ok)
        for (int i = 0; i < ns; ++i)
          if (last[i] >= 0) mbar_wait(&full[i], (last[i] / ns) & 1, abort_flag + 1, status);
    }
    return;
  }
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  bool ok = true;
  for (int s = 0; s < nst; ++s) {
    const int st = s % ns;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (s / ns) & 1, abort_flag, status));
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

}  // namespace

cudaError_t launch_read_stream(const void* src, long long bytes, unsigned* status, cudaStream_t s) {
  const int ns = 5;
  const size_t smem = 128 + (size_t)ns * ISTAGE + 2 * INS_MAX * 8 + 16;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(read_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms());
  cfg.blockDim = dim3(ITHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, read_stream_kernel, (const uint8_t*)src, bytes, status, ns);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e;
}

bool gemv_i8_fits(int qtype, int n, int k, int T, bool swiglu) {
  // block formats and K-quants, one or two tokens; k % 256 == 0 (whole rows
  // 16-byte aligned in a stage); a row's warps within the consumer warps; a
  // ring of at least 4 stages beside the X tables and the CTA's row sums
  if ((!block32_format(qtype) && !kquant(qtype)) || T < 1 || T > 2 || k % 256 != 0 || (k / 64 + 31) / 32 > 8)
    return false;
  // two tokens of Q8_0 below 2^25 weight elements: the bulk CUDA-core kernel
  // measured faster (4096 x 4096: 9.4 against 10.5 us; at 12288 x 4096 this
  // kernel takes 21.4 against 22.4 us on the tensor cores, and Q4_0 8.5 / 15.9
  // against 10.2 / 20.8 us)
  if (T == 2 && qtype == kQ8_0 && (long)n * k < (1L << 25)) return false;
  return rows_per_stage(qtype, k, swiglu) >= 1 && i8_stages(qtype, k, n, T) >= 4;
}

cudaError_t launch_gemv_i8(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y,
                           int ldy, const float* R, unsigned* status, cudaStream_t s) {
  const bool swi = Wu != nullptr;
  if (qtype == kQ4_K)
    return swi ? launch_i8_t<kQ4_K, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
               : launch_i8_t<kQ4_K, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (qtype == kQ5_K)
    return swi ? launch_i8_t<kQ5_K, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
               : launch_i8_t<kQ5_K, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (qtype == kQ6_K)
    return swi ? launch_i8_t<kQ6_K, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
               : launch_i8_t<kQ6_K, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (qtype == kIQ4_XS)
    return swi ? launch_i8_t<kIQ4_XS, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
               : launch_i8_t<kIQ4_XS, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  if (qtype == kQ4_0)
    return swi ? launch_i8_t<kQ4_0, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
               : launch_i8_t<kQ4_0, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
  return swi ? launch_i8_t<kQ8_0, true>(W, Wu, n, k, X, T, Y, ldy, R, status, s)
             : launch_i8_t<kQ8_0, false>(W, Wu, n, k, X, T, Y, ldy, R, status, s);
}

}  // namespace apr
