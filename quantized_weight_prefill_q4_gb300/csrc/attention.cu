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
// Before the kernel, the K and V cache rows 0 .. pos0 + T - 1 (every KV head)
// are converted to fp16 into the stream's scratch: K as it is
// ([positions][num_kv_heads * 256]), V transposed ([num_kv_heads * 256]
// [positions, rounded up to 8]), so that both operands of the two products are K-major tiles
// that TMA copies straight into the 128-byte-swizzled MMA layout.
//
// One CTA per (128 query rows, query head); the CTAs of the last query rows,
// which see the most keys, are launched first. When that grid would leave
// SMs idle, each query tile's key tiles are cut into parts of at most P
// tiles (P the smallest that keeps the grid within one CTA per SM) and every
// part gets its own CTA: a CTA of a cut tile writes its unnormalized O, its
// reference max and its sum into the stream's scratch, and a second kernel
// combines the parts of each row, O = sum_s 2^(m_s - m) O_s / sum_s 2^(m_s -
// m) l_s (m the largest m_s of the parts the row sees keys in), in part
// order. Keys go in tiles of 64. The
// roles hand work to each other through mbarriers, so that the tensor cores
// compute the scores of tile j + 1 while the softmax of tile j runs:
//   warps 0-3   own the 128 query rows (one row per thread, TMEM lane = row):
//               they write fp16 Q into shared memory once (128-byte swizzled,
//               K-major), then per key tile read the 64 scores, update the
//               running max and sum, write the fp16 weights P into tensor
//               memory, and at the end scale O by 1 / sum
//   warp 4      issues the MMAs (one elected lane), in the order S_0, then per
//               tile j: S_{j+1} = Q . K_{j+1}^T (M = 128, N = 64, 16 steps of
//               K = 16 over the head dim, both operands in shared memory) and,
//               once P_j is written, O += P_j . V_j (M = 128, N = 256, 4 steps
//               of K = 16 over the keys, P read from tensor memory)
//   warp 5      TMA producer: per tile four K boxes [64 keys][64 dims] into a
//               ring of three K buffers, each refilled once the scores of its
//               previous tile are computed, and one V box [256 dims][64 keys]
//               into a ring of two V buffers, each refilled once the O product
//               of its previous tile is done; positions past pos0 + T lie
//               outside the tensor maps and arrive as zeros
// Tensor memory (512 columns allocated): O fp32 [0, 256), S fp32 two buffers
// [256, 384), P fp16 pairs two buffers [384, 448).
// The softmax works in base 2 (scores times log2(e) / 16). The weights are
// taken against a reference max m_ref that is moved (rescaling O and the sum,
// after the previous O product is done) only when the running max exceeds it
// by more than 8, so a weight is at most 2^8 and O is rewritten only when the
// max jumps; the sum adds the weights as rounded to fp16, the values the MMA
// multiplies.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the device
// status word and an abort flag that ends every role's waits; the MMA warp
// then waits (bounded) for its MMAs in flight, the producer for its copies,
// and the CTA frees its tensor memory.

#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "apr_internal.h"
#include "dev_common.cuh"
#include "host_common.h"

namespace apr {
namespace {

constexpr int AD = 256;                          // head dim
constexpr int AQ = 128;                          // query rows per CTA (MMA M, TMEM lanes)
constexpr int AKEY = 64;                         // keys per tile
constexpr int KBUF = 3;                          // K tile ring
constexpr int VBUF = 3;                          // V tile ring
constexpr int PBUF = 2;                          // P tiles (softmax weights) in shared memory
constexpr int SOFT_WARPS = 4;
constexpr int MMA_WARP = 4;
constexpr int TMA_WARP = 5;
constexpr int A_THREADS = 32 * 6;
constexpr int K_PANEL = AKEY * 128;              // [64 keys][64 dims] fp16, 8 KB
constexpr int K_BYTES = (AD / 64) * K_PANEL;     // four panels, 32 KB
constexpr int V_BYTES = AD * 128;                // [256 dims][64 keys] fp16, 32 KB
constexpr int P_BYTES = AQ * 128;                // [128 rows][64 keys] fp16, 16 KB
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KBUF * K_BYTES;
constexpr int OFF_P = OFF_V + VBUF * V_BYTES;
constexpr int OFF_BAR = OFF_P + PBUF * P_BYTES;
// Q arrives as fp32 boxes of [128 rows][32 dims] (128-byte swizzled), 8 of
// them, staged in K buffer 2 and the V ring before those receive tiles (K
// buffers 0 and 1 fill meanwhile)
constexpr int QBOX_BYTES = AQ * 128;
constexpr int OFF_QST = OFF_K + 2 * K_BYTES;
static_assert(OFF_QST + (AD / 32) * QBOX_BYTES <= OFF_P, "Q staging fits K buffer 2 and the V ring");
// O leaves the same way, fp32 boxes of [128 rows][32 dims] staged from offset
// 0 once every product is done (the rings are idle then)
constexpr int OFF_OST = 0;
static_assert(OFF_OST + (AD / 32) * QBOX_BYTES <= OFF_P, "O staging fits the rings");
constexpr int A_SMEM = OFF_BAR + 192 + 1024;     // barriers, TMEM holder, flags; alignment slack
// tensor memory: O fp32 [0, 256), Q fp16 pairs [256, 384), S fp32 two buffers [384, 512)
constexpr uint32_t COL_O = 0, COL_Q = 256, COL_S = 384;
constexpr uint32_t A_TMEM_COLS = 512;
constexpr float kRescaleAbove = 8.0f;            // log2 of the largest weight kept unscaled
static_assert(A_SMEM <= 232448, "shared memory budget");
static_assert(COL_S + 2 * AKEY <= A_TMEM_COLS, "tensor memory budget");

// D[tmem] (+)= A[smem] . B[smem]^T: both operands K-major in shared memory
// (128-byte swizzle descriptors, smem_desc_sw128), fp32 accumulate.
__device__ __forceinline__ void mma_f16_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x, the hardware approximation with results below float's normal range
// flushed to zero
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The cache rows 0 .. rows - 1 to fp16 (round to nearest) in one launch:
// K as it is ([rows][cols] -> K16, 8 values a thread step) and V transposed
// ([rows][cols] -> VT [cols][ldv], ldv a multiple of 16, positions past rows
// written as zeros). A warp transposes 16 positions x 32 columns through
// registers: lane l reads column c0 + l of the 16 rows (every load a
// coalesced 128-byte row segment) and writes its 16 fp16 values as 32
// contiguous bytes of row c0 + l of VT. No shared memory, so that the
// attention kernel, launched programmatically behind it, can take an SM
// beside its blocks.
__global__ void __launch_bounds__(256) kv_to_f16_kernel(const float* __restrict__ K, const float* __restrict__ V,
                                                        int rows, int cols, uint16_t* __restrict__ K16,
                                                        uint16_t* __restrict__ VT, int ldv) {
  grid_launch_dependents();
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  // K: rows * cols is a multiple of 8 (cols is a multiple of 256)
  const size_t n8 = (size_t)rows * cols / 8;
  const float4* k4 = reinterpret_cast<const float4*>(K);
  uint4* o4 = reinterpret_cast<uint4*>(K16);
  for (size_t i = tid; i < n8; i += nthreads) {
    const float4 a = __ldg(k4 + 2 * i), b = __ldg(k4 + 2 * i + 1);
    o4[i] = make_uint4(pack_half2(a.x, a.y), pack_half2(a.z, a.w), pack_half2(b.x, b.y), pack_half2(b.z, b.w));
  }
  // V: units of 16 positions x 32 columns, one per warp step
  const int lane = threadIdx.x & 31;
  const size_t nwarps = nthreads / 32, wid = tid / 32;
  const int pblocks = ldv / 16, cblocks = cols / 32;
  for (size_t u = wid; u < (size_t)pblocks * cblocks; u += nwarps) {
    const int p0 = (int)(u % pblocks) * 16, c = (int)(u / pblocks) * 32 + lane;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = p0 + i < rows ? __ldg(V + (size_t)(p0 + i) * cols + c) : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(VT + (size_t)c * ldv + p0);
    dst[0] = make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]), pack_half2(v[6], v[7]));
    dst[1] = make_uint4(pack_half2(v[8], v[9]), pack_half2(v[10], v[11]), pack_half2(v[12], v[13]),
                        pack_half2(v[14], v[15]));
  }
}

// key tiles seen by the rows of query tile qt
__host__ __device__ inline int attn_key_tiles(int qt, int T, int pos0) {
  const int last = (qt + 1) * AQ < T ? (qt + 1) * AQ : T;
  return (pos0 + last + AKEY - 1) / AKEY;
}

// The parts of the cut query tiles into O: a thread per 4 dims of a row,
// 32 CTAs of 256 per (query tile, head) (every load of a thread issued at
// once; the threads of a row read its parts' (m, l) through the same cache
// lines). Rows past T are not written, and the query tiles of one part were
// written by the attention kernel itself.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float2* __restrict__ part_ml, void* O, int T,
                                                           int pos0, int num_heads, int P, int o16) {
  constexpr int PER_TILE = AQ * (AD / 4) / 256;  // CTAs per (query tile, head)
  // launched programmatically behind the attention kernel: its parts are
  // complete and visible after the wait
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int nqt = (T + AQ - 1) / AQ;
  const int th = (int)(blockIdx.x / PER_TILE), qt = th / num_heads, h = th % num_heads;
  const int i = (int)(blockIdx.x % PER_TILE) * 256 + (int)threadIdx.x;
  const int r = i / (AD / 4), d4 = i % (AD / 4), t = qt * AQ + r;
  const int ns = (attn_key_tiles(qt, T, pos0) + P - 1) / P;
  if (ns == 1 || t >= T) return;
  int unit = 0;  // the first unit of this query tile (later tiles' parts come first)
  for (int q2 = nqt - 1; q2 > qt; --q2) unit += (attn_key_tiles(q2, T, pos0) + P - 1) / P;
  const size_t slot0 = (size_t)unit * num_heads + h, sstep = (size_t)num_heads;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) {
    const float2 ml = part_ml[(slot0 + s * sstep) * AQ + r];
    if (ml.y > 0.f) m = fmaxf(m, ml.x);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  for (int s = 0; s < ns; ++s) {
    const size_t slot = slot0 + s * sstep;
    const float2 ml = part_ml[slot * AQ + r];
    if (!(ml.y > 0.f)) continue;  // the row sees no key of this part
    const float w = exp2f(ml.x - m);
    const float4 o = reinterpret_cast<const float4*>(part_o + (slot * AQ + r) * AD)[d4];
    acc.x = fmaf(w, o.x, acc.x);
    acc.y = fmaf(w, o.y, acc.y);
    acc.z = fmaf(w, o.z, acc.z);
    acc.w = fmaf(w, o.w, acc.w);
    L = fmaf(w, ml.y, L);
  }
  const float inv = 1.0f / L;
  const size_t at = (size_t)t * ((size_t)num_heads * AD) + (size_t)h * AD + 4 * d4;
  if (o16) {
    const __half2 a = __floats2half2_rn(acc.x * inv, acc.y * inv), b = __floats2half2_rn(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(O) + at) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(O) + at) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

__global__ void __launch_bounds__(A_THREADS, 1)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                             const __grid_constant__ CUtensorMap tmP, int T, int pos0, int num_heads,
                             int num_kv_heads, unsigned* status, int o16, int P, float2* __restrict__ part_ml) {
  // P > 0: key tiles in parts of at most P (see above); CTA b's unnormalized
  // O goes to rows 128 b .. of tmP, its (m, l) per row to part_ml[128 b + r]
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sP = smem + OFF_P;
  uint64_t* kFull = reinterpret_cast<uint64_t*>(smem + OFF_BAR);  // [3] a K tile has landed
  uint64_t* kEmpty = kFull + 3;                                   // [3] the scores of a K buffer's tile are done
  uint64_t* vFull = kFull + 6;                                    // [3] a V tile has landed
  uint64_t* vEmpty = kFull + 9;                                   // [3] the O product of a V buffer's tile is done
  uint64_t* sFull = kFull + 12;                                   // [2] S_j computed (and every MMA before it)
  uint64_t* pFull = kFull + 14;                                   // [2] P_j written (one arrival per softmax warp)
  uint64_t* oDone = kFull + 16;                                   // O += P_j . V_j done
  uint64_t* oLast = kFull + 17;                                   // the last O product done (one phase)
  uint64_t* drain = kFull + 18;
  uint64_t* qFull = kFull + 19;                                   // Q's fp32 boxes have landed
  uint64_t* qFree = kFull + 20;                                   // Q is in tensor memory: its staging is free
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(kFull + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(kFull + 22);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = (T + AQ - 1) / AQ;
  const int h = blockIdx.x % num_heads;
  // the query tile, and with parts which part: units of num_heads CTAs, the
  // last query tile's parts first
  int qt = nqt - 1 - (int)(blockIdx.x / num_heads), part = 0, nparts = 1;
  if (P > 0) {
    int u = (int)(blockIdx.x / num_heads);
    for (qt = nqt - 1; qt > 0; --qt) {
      const int ns = (attn_key_tiles(qt, T, pos0) + P - 1) / P;
      if (u < ns) break;
      u -= ns;
    }
    nparts = (attn_key_tiles(qt, T, pos0) + P - 1) / P;
    part = u;
  }
  const int t0 = qt * AQ;
  const int g = h / (num_heads / num_kv_heads);
  const int nkt_all = attn_key_tiles(qt, T, pos0);   // key tiles this CTA's rows see
  const int kt0 = part * nkt_all / nparts;          // this CTA's key tiles kt0 .. kt0 + nkt - 1
  const int nkt = (part + 1) * nkt_all / nparts - kt0;
  const bool partial = nparts > 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 3; ++i) {
      mbar_init(&kFull[i], 1);
      mbar_init(&kEmpty[i], 1);
      mbar_init(&vFull[i], 1);
      mbar_init(&vEmpty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sFull[i], 1);
      mbar_init(&pFull[i], SOFT_WARPS);
    }
    mbar_init(oDone, 1);
    mbar_init(oLast, 1);
    mbar_init(drain, 1);
    mbar_init(qFull, 1);
    mbar_init(qFree, SOFT_WARPS);
    abort_flag[0] = 0;
    abort_flag[1] = 0;   // never set: the drain waits ignore the abort
    fence_mbar_init();
    // the next kernel may launch (the parts' combination, or a GEMM that
    // streams its weights on the SMs this grid leaves free); it reads this
    // kernel's output only after its own dependency wait
    grid_launch_dependents();
  }
  if (warp == 0) tmem_alloc(tmem_holder, A_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // two producer lanes, so that K and V are each refilled as soon as their own
  // buffer is free: lane 0 the K ring, lane 1 the V ring
  const bool kprod = warp == TMA_WARP && lane == 0, vprod = warp == TMA_WARP && lane == 1;
  int last_k = -1, last_v = -1;   // the last K (lane 0) and V (lane 1) tiles sent
  auto send_k = [&](int ti) {
    const int b = ti % KBUF;
    mbar_arrive_expect_tx(&kFull[b], K_BYTES);
#pragma unroll
    for (int p = 0; p < AD / 64; ++p)
      tma_load_2d(sK + b * K_BYTES + p * K_PANEL, &tmK, g * AD + 64 * p, (kt0 + ti) * AKEY, &kFull[b]);
    last_k = ti;
  };
  auto send_v = [&](int ti) {
    const int b = ti % VBUF;
    mbar_arrive_expect_tx(&vFull[b], V_BYTES);
    tma_load_2d(sV + b * V_BYTES, &tmV, (kt0 + ti) * AKEY, g * AD, &vFull[b]);
    last_v = ti;
  };

  // softmax rows: thread r = query row t0 + r = TMEM lane r
  const int r = threadIdx.x;
  const int t = t0 + r;
  const uint32_t lane_addr = tmem_base + ((uint32_t)(warp * 32) << 16);

  // ---- prologue: Q's fp32 boxes and K tiles 0, 1 on their way; Q converted
  // into tensor memory; then the rest of the K and V rings
  bool q_sent = false;
  if (kprod) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    mbar_arrive_expect_tx(qFull, (AD / 32) * QBOX_BYTES);
#pragma unroll
    for (int b = 0; b < AD / 32; ++b) tma_load_2d(smem + OFF_QST + b * QBOX_BYTES, &tmQ, h * AD + 32 * b, t0, qFull);
    q_sent = true;
    grid_dependency_wait();   // K16 and VT16 come from the conversion launched just before
    for (int ti = 0; ti < 2 && ti < nkt; ++ti) send_k(ti);
    if (mbar_wait(qFree, 0, abort_flag, status) && nkt > 2) send_k(2);
  } else if (vprod) {
    tma_prefetch_desc(&tmV);
    grid_dependency_wait();
    if (mbar_wait(qFree, 0, abort_flag, status))
      for (int ti = 0; ti < VBUF && ti < nkt; ++ti) send_v(ti);
  } else if (warp < SOFT_WARPS) {
    // row r of the staged boxes (16-byte chunk c of a row at c ^ (r & 7)) as
    // fp16 pairs into TMEM lane r, columns COL_Q + 0 .. 127 (dims in order);
    // rows past T arrived as zeros
    if (__all_sync(0xffffffffu, mbar_wait(qFull, 0, abort_flag, status))) {
#pragma unroll 1
      for (int pair = 0; pair < AD / 64; ++pair) {
        uint32_t w[32];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const uint8_t* row = smem + OFF_QST + (2 * pair + bb) * QBOX_BYTES + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(row + ((c ^ (r & 7)) << 4));
            w[16 * bb + 2 * c] = pack_half2(v.x, v.y);
            w[16 * bb + 2 * c + 1] = pack_half2(v.z, v.w);
          }
        }
        tmem_st_32x32b_x32(lane_addr + COL_Q + 32 * pair, w);
        // the store reads its source registers asynchronously
        tmem_st_wait();
      }
    }
    tc_fence_before();
    // the staging's generic reads before the producers' TMA writes into it
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(qFree);
  }
  __syncthreads();

  if (warp == MMA_WARP) {
    // ------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t IDESC_S = idesc_f16_f32(AQ, AKEY);
    constexpr uint32_t IDESC_O = idesc_f16_f32(AQ, AD);
    tc_fence_after();   // Q's tensor-memory stores came before the block barrier
    // S_ti = Q . K_ti^T: A = Q from tensor memory (8 columns per 16 dims), B =
    // the K tile in shared memory (panel per 64 dims, +32 bytes per 16)
    auto issue_S = [&](int ti) {
      const uint64_t kdesc = smem_desc_sw128(sK + (ti % KBUF) * K_BYTES);
#pragma unroll
      for (int kk = 0; kk < AD / 16; ++kk)
        mma_f16_ts_elect(tmem_base + COL_S + AKEY * (ti & 1), tmem_base + COL_Q + 8 * kk,
                         kdesc + (uint64_t)(((kk >> 2) * K_PANEL) >> 4) + 2 * (kk & 3), IDESC_S, kk != 0);
      mma_commit_elect(&sFull[ti & 1]);
      mma_commit_elect(&kEmpty[ti % KBUF]);
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(&kFull[0], 0, abort_flag, status));
    if (ok) {
      tc_fence_after();
      issue_S(0);
    }
#pragma unroll 1
    for (int j = 0; j < nkt && ok; ++j) {
      if (j + 1 < nkt) {
        // S_{j+1} into the S buffer that S_{j-1} used: read before P_{j-1} was
        // handed over, which came before O_{j-1} was issued
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&kFull[(j + 1) % KBUF], (uint32_t)(((j + 1) / KBUF) & 1), abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        issue_S(j + 1);
      }
      // V first (it is usually in), then P: one wake-up on the critical path
      ok = __all_sync(0xffffffffu, mbar_wait(&vFull[j % VBUF], (uint32_t)((j / VBUF) & 1), abort_flag, status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&pFull[j & 1], (uint32_t)((j >> 1) & 1), abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      // O += P_j . V_j: A = P_j [128 rows][64 keys], B = V_j [256 dims][64
      // keys], both K-major in shared memory (+32 bytes per 16 keys)
      const uint64_t pdesc = smem_desc_sw128(sP + (j & 1) * P_BYTES);
      const uint64_t vdesc = smem_desc_sw128(sV + (j % VBUF) * V_BYTES);
#pragma unroll
      for (int kk = 0; kk < AKEY / 16; ++kk)
        mma_f16_ss_elect(tmem_base + COL_O, pdesc + 2 * kk, vdesc + 2 * kk, IDESC_O, (j | kk) != 0);
      mma_commit_elect(&vEmpty[j % VBUF]);
      mma_commit_elect(oDone);
      if (j == nkt - 1) mma_commit_elect(oLast);
    }
    if (!ok) {  // wait until the MMAs already issued have finished
      mma_commit_elect(drain);
      __all_sync(0xffffffffu, mbar_wait(drain, 0, abort_flag + 1, status));
    }
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------ TMA producers
    if (kprod) {
      // K_n once S_{n-3}, the previous tile of its buffer, is done
      bool ok = true;
#pragma unroll 1
      for (int n = KBUF; n < nkt && ok; ++n) {
        ok = mbar_wait(&kEmpty[n % KBUF], (uint32_t)(((n / KBUF) - 1) & 1), abort_flag, status);
        if (ok) send_k(n);
      }
      // every copy sent has landed before the CTA ends (at once unless a wait
      // gave up); the last tile of a ring slot is the only one that can be pending
      for (int ti = max(0, last_k - KBUF + 1); ti <= last_k; ++ti)
        mbar_wait(&kFull[ti % KBUF], (uint32_t)((ti / KBUF) & 1), abort_flag + 1, status);
      if (q_sent) mbar_wait(qFull, 0, abort_flag + 1, status);
    } else if (vprod) {
      // V_n once O_{n-3}, the previous tile of its buffer, is done
      bool ok = true;
#pragma unroll 1
      for (int n = VBUF; n < nkt && ok; ++n) {
        ok = mbar_wait(&vEmpty[n % VBUF], (uint32_t)(((n / VBUF) - 1) & 1), abort_flag, status);
        if (ok) send_v(n);
      }
      for (int ti = max(0, last_v - VBUF + 1); ti <= last_v; ++ti)
        mbar_wait(&vFull[ti % VBUF], (uint32_t)((ti / VBUF) & 1), abort_flag + 1, status);
    }
  } else {
    // ------------------------------------------------ softmax rows, then the output
    const float sl2 = 1.4426950408889634f / 16.0f;   // log2(e) / sqrt(256)
    const int plim = pos0 + min(t, T - 1);            // last key row t sees (rows past T: the last row's)
    float m_run = -INFINITY, m_ref = 0.f, l = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nkt; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&sFull[j & 1], (uint32_t)((j >> 1) & 1), abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x32(lane_addr + COL_S + AKEY * (j & 1), sv);
      tmem_ld_32x32b_x32(lane_addr + COL_S + AKEY * (j & 1) + 32, sv + 32);
      tmem_ld_wait_regs(sv);
      regs_after_wait(sv + 32);
      const int kb = (kt0 + j) * AKEY;
      float s[64];
      if (kb + AKEY - 1 <= plim) {   // every key of the tile visible to this row
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sv[c]) * sl2;
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = kb + c <= plim ? __uint_as_float(sv[c]) * sl2 : -INFINITY;
      }
      float mq[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int c = 4; c < 64; ++c) mq[c & 3] = fmaxf(mq[c & 3], s[c]);
      const float m_new = fmaxf(m_run, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
      if (j == 0) {
        // the first key of the CTA's range is visible to every row that sees
        // any key of it (visibility is a prefix of the keys); a row that sees
        // none keeps weights of 0 and a sum of 0, which the combination skips
        m_ref = m_new == -INFINITY ? 0.f : m_new;
      } else if (__any_sync(0xffffffffu, m_new > m_ref + kRescaleAbove)) {
        // the whole warp moves its reference (tensor-memory access is per
        // warp), once O += P_{j-1} . V_{j-1} is done (S_j's completion already
        // covers O_{j-2}, so the parity wait cannot be a phase behind)
        ok = __all_sync(0xffffffffu, mbar_wait(oDone, (uint32_t)((j - 1) & 1), abort_flag, status));
        if (!ok) break;
        tc_fence_after();
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
          // the store reads its source registers asynchronously: the next
          // load must not overwrite them before it has completed
          tmem_st_wait();
        }
        m_ref = m_new;
      }
      m_run = m_new;
      // weights 2^(s - m_ref) <= 2^8, rounded to fp16 (a result below
      // float's normal range rounds to fp16 zero either way, so the
      // flush-to-zero form of ex2 gives the same fp16 weights)
      uint32_t pv[32];
      float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const __half2 p = __floats2half2_rn(ex2_ftz(s[2 * c] - m_ref), ex2_ftz(s[2 * c + 1] - m_ref));
        const float2 pf = __half22float2(p);
        lq[c & 3] += pf.x + pf.y;
        pv[c] = *reinterpret_cast<const uint32_t*>(&p);
      }
      l += (lq[0] + lq[1]) + (lq[2] + lq[3]);
      // P_j into shared memory, row r of the P buffer of P_{j-2} (whose O
      // product S_j's completion covers): 16-byte chunk c at c ^ (r & 7)
      uint8_t* prow = sP + (j & 1) * P_BYTES + r * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) =
            make_uint4(pv[4 * cc], pv[4 * cc + 1], pv[4 * cc + 2], pv[4 * cc + 3]);
      fence_proxy_async_smem();   // the MMA reads P through the async proxy
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pFull[j & 1]);
    }
    // ---- O / l to global memory, after the last O product: row r of box cb
    // (dims 32 cb ..) with 16-byte chunk c at c ^ (r & 7), then TMA tensor
    // stores (rows past T are not written). A thread writes 128 contiguous
    // bytes of one row per box; a warp store of scattered rows would move
    // 32 half-filled sectors instead.
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(oLast, 0, abort_flag, status));
    if (ok) {
      tc_fence_after();
      // a part: O as accumulated, with the row's reference max and sum
      const float inv = partial ? 1.0f : 1.0f / l;
      if (partial) part_ml[(size_t)blockIdx.x * AQ + r] = make_float2(m_ref, l);
      if (o16 && !partial) {
        // fp16 O: boxes of 64 dims (128 bytes a row), the same swizzle
#pragma unroll 1
        for (int cb = 0; cb < AD / 64; ++cb) {
          uint32_t ov[64];
          tmem_ld_32x32b_x32(lane_addr + COL_O + cb * 64, ov);
          tmem_ld_32x32b_x32(lane_addr + COL_O + cb * 64 + 32, ov + 32);
          tmem_ld_wait_regs(ov);
          regs_after_wait(ov + 32);
          uint8_t* row = smem + OFF_OST + cb * QBOX_BYTES + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t hv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const __half2 hp = __floats2half2_rn(__uint_as_float(ov[8 * c + 2 * u]) * inv,
                                                   __uint_as_float(ov[8 * c + 2 * u + 1]) * inv);
              hv[u] = *reinterpret_cast<const uint32_t*>(&hp);
            }
            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          }
        }
      } else {
#pragma unroll 1
        for (int cb = 0; cb < AD / 32; ++cb) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(lane_addr + COL_O + cb * 32, ov);
          tmem_ld_wait_regs(ov);
          uint8_t* row = smem + OFF_OST + cb * QBOX_BYTES + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(row + ((c ^ (r & 7)) << 4)) =
                make_float4(__uint_as_float(ov[4 * c]) * inv, __uint_as_float(ov[4 * c + 1]) * inv,
                            __uint_as_float(ov[4 * c + 2]) * inv, __uint_as_float(ov[4 * c + 3]) * inv);
        }
      }
      fence_proxy_async_smem();   // the TMA store reads the boxes through the async proxy
    }
    named_sync(1, 32 * SOFT_WARPS);
    if (threadIdx.x == 0 && ok) {
      const int dims = o16 && !partial ? 64 : 32;  // dims a box
#pragma unroll 1
      for (int cb = 0; cb < AD / dims; ++cb) {
        if (partial)
          tma_store_2d(&tmP, smem + OFF_OST + cb * QBOX_BYTES, dims * cb, (int)blockIdx.x * AQ);
        else
          tma_store_2d(&tmO, smem + OFF_OST + cb * QBOX_BYTES, h * AD + dims * cb, t0);
      }
      bulk_commit_group();
      bulk_wait_read_all();   // the boxes are read before the CTA's shared memory goes
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem_base, A_TMEM_COLS);
}

}  // namespace

// The key-tile part size P: 0 (no parts) when the plain grid already fills
// the SMs or parts would shorten the longest CTA by fewer than 12 key tiles;
// else the smallest P whose grid fits one CTA per SM. Measured on GB300
// (16 / 4 heads): a CTA costs about 7 us besides about 1.1 us a key tile, and
// the parts about 9 us more in all (the combining launch, the partial sums'
// traffic, more CTAs' fixed costs): 512 rows at position 0 (the longest CTA
// 8 tiles, parts of 3) took 21.4 us against 17.9 us whole, 512 rows at 1536
// (32 tiles, parts of 15) 35.2 us against about 44.7.
static int attn_parts(int T, int pos0, int num_heads) {
  const int nqt = (T + AQ - 1) / AQ, sms = num_sms();
  if ((long long)nqt * num_heads >= sms) return 0;
  const int most = attn_key_tiles(nqt - 1, T, pos0);
  for (int P = 1; P + 12 <= most; ++P) {
    long long units = 0;
    for (int qt = 0; qt < nqt; ++qt) units += (attn_key_tiles(qt, T, pos0) + P - 1) / P;
    if (units * num_heads <= sms) return P;
  }
  return 0;
}

// scratch: K16, then VT16, then (parts) one CTA per SM at most of partial O
// [128 rows][256] fp32 and (m, l) per row
static size_t attn_part_offset(size_t rows, size_t kv_dim) {
  const size_t ldv = (rows + 15) & ~(size_t)15;
  return ((rows * kv_dim * 2 + 255) & ~(size_t)255) + ((kv_dim * ldv * 2 + 255) & ~(size_t)255);
}

size_t prefill_attention_scratch_bytes(int T, int pos0, int num_kv_heads) {
  const size_t rows = (size_t)pos0 + (size_t)T, kv_dim = (size_t)num_kv_heads * AD;
  return attn_part_offset(rows, kv_dim) + (size_t)num_sms() * AQ * (AD * 4 + 8);
}

int launch_prefill_attention(const float* Q, const float* K, const float* V, float* O, int T, int pos0,
                             int num_heads, int num_kv_heads, void* scratch, unsigned* status, cudaStream_t s,
                             char* msg, size_t msg_len, bool o16) {
  if (T <= 0) return 0;
  const size_t rows = (size_t)pos0 + (size_t)T, kv_dim = (size_t)num_kv_heads * AD;
  const size_t ldv = (rows + 15) & ~(size_t)15;
  uint16_t* K16 = static_cast<uint16_t*>(scratch);
  uint16_t* VT16 = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(scratch) + ((rows * kv_dim * 2 + 255) & ~(size_t)255));
  const int P = attn_parts(T, pos0, num_heads);
  float* part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + attn_part_offset(rows, kv_dim));
  float2* part_ml = reinterpret_cast<float2*>(part_o + (size_t)num_sms() * AQ * AD);
  auto cuda_fail = [&](cudaError_t e, const char* what) {
    snprintf(msg, msg_len, "%s: %s", what, cudaGetErrorString(e));
    return -1;
  };
  // the fp16 copies of the cache rows 0 .. pos0 + T - 1 (plain stream order:
  // everything before is complete when it starts)
  {
    const size_t units = rows * kv_dim / 8 / 256 + 1;
    const unsigned blocks = (unsigned)(units < (size_t)num_sms() * 4 ? units : (size_t)num_sms() * 4);
    kv_to_f16_kernel<<<blocks, 256, 0, s>>>(K, V, (int)rows, (int)kv_dim, K16, VT16, (int)ldv);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "K and V to fp16");

  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(msg, msg_len);
  if (!fn) return -1;
  CUtensorMap mK, mV;
  if (!make_map_2d(fn, &mK, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K16, kv_dim, rows, kv_dim * 2, 64, AKEY,
                   CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len))
    return -1;
  if (!make_map_2d(fn, &mV, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, VT16, rows, kv_dim, ldv * 2, AKEY, AD,
                   CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len))
    return -1;
  // Q as fp32 boxes of [128 rows][32 dims] (128 bytes, the swizzle span)
  const uint64_t q_dim = (uint64_t)num_heads * AD;
  CUtensorMap mQ, mO;
  if (!make_map_2d(fn, &mQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Q, q_dim, (uint64_t)T, q_dim * 4, 32, AQ,
                   CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len) ||
      !(o16 ? make_map_2d(fn, &mO, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, O, q_dim, (uint64_t)T, q_dim * 2, 64, AQ,
                          CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len)
            : make_map_2d(fn, &mO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, O, q_dim, (uint64_t)T, q_dim * 4, 32, AQ,
                          CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len)))
    return -1;

  // the parts' O: [one CTA per SM x 128 rows][256] fp32, the boxes of O's fp32 form
  CUtensorMap mP = mO;
  if (P > 0 && !make_map_2d(fn, &mP, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, part_o, AD, (uint64_t)num_sms() * AQ, AD * 4,
                            32, AQ, CU_TENSOR_MAP_SWIZZLE_128B, msg, msg_len))
    return -1;

  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, A_SMEM);
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention attributes");
    attr_set[dev] = 1;
  }
  long long grid = (long long)((T + AQ - 1) / AQ) * num_heads;
  if (P > 0) {
    long long units = 0;
    for (int qt = 0; qt < (T + AQ - 1) / AQ; ++qt) units += (attn_key_tiles(qt, T, pos0) + P - 1) / P;
    grid = units * num_heads;  // at most one CTA per SM (attn_parts)
  }
  // launched programmatically: its CTAs start (Q on its way) while the
  // conversion finishes; the K and V producers wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(A_THREADS);
  cfg.dynamicSmemBytes = A_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_attention_kernel, mK, mV, mQ, mO, mP, T, pos0, num_heads, num_kv_heads, status,
                         o16 ? 1 : 0, P, part_ml);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill attention");
  if (P > 0) {
    // launched programmatically: its CTAs wait for the attention grid in
    // griddepcontrol.wait
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3((unsigned)((T + AQ - 1) / AQ * num_heads * (AQ * (AD / 4) / 256)));
    ccfg.blockDim = dim3(256);
    ccfg.stream = s;
    cudaLaunchAttribute cattr[1] = {pdl_attr()};
    ccfg.attrs = cattr;
    ccfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&ccfg, attn_combine_kernel, (const float*)part_o, (const float2*)part_ml, (void*)O, T,
                           pos0, num_heads, P, o16 ? 1 : 0);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention parts");
  }
  return 0;
}

}  // namespace apr
