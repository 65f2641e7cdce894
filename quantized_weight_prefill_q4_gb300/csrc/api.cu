// C ABI of libapr_qgemm: argument checks, the T rule, scratch, launches.
//
// Argument checking follows the pattern of aprender-serve 0.70.2
// src/cuda/executor/gdn_prefill_ops.rs (qp_launch checks every pointer
// argument before a launch; qwen35_dequant_f32 refuses a weight type it has no
// kernel for) and oxibonsai-kernels 0.1.4 try_cuda_prefill_q_std (an empty
// batch returns success without work).

#include <cstdarg>
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "apr_qgemm.h"
#include "apr_internal.h"

using namespace apr;

namespace {

// Status word of the kernels' bounded waits, one per device (module-scope
// __device__ variables exist once per device that loads the library).
__device__ unsigned g_status;

thread_local char t_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
  return code;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int dev = -1;
  int checked = 0;          // APR_OK or APR_E_DEVICE
  unsigned* status = nullptr;
};
DeviceState g_dev[kMaxDevices];

int device_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(APR_E_DEVICE, "no usable CUDA device (%s)", cudaGetErrorString(e));
  }
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    st.dev = dev;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess || prop.major != 10 || prop.minor != 3) {
      cudaGetLastError();
      st.checked = APR_E_DEVICE;
      return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
      cudaGetLastError();
      st.checked = APR_E_DEVICE;
      return;
    }
    st.status = static_cast<unsigned*>(p);
    st.checked = APR_OK;
  });
  if (st.checked != APR_OK)
    return fail(APR_E_DEVICE, "device %d is not a compute capability 10.3 GPU (GB300) or failed to initialise", dev);
  *out = &st;
  return APR_OK;
}

// Scratch owned by the library, one buffer per (device, stream, use): the
// fp16 copy of X for the GEMM, the ticket counters and partial sums of the
// GEMV. Calls on one stream are ordered by it, and every kernel touches
// scratch only after waiting for the kernel before it (griddepcontrol.wait),
// so one buffer serves every call on the stream and successive kernels still
// overlap (no allocation between them). A buffer only grows: a larger one
// replaces it and the old one is kept, so graphs captured with it stay valid.
// Growth uses cudaMalloc with the calling thread's capture mode relaxed for
// the call, so that it also works while the stream is being captured. A graph
// captured from a stream uses that stream's buffers: replay it ordered with
// the stream's other library calls, not concurrently with them.
// The GEMV's buffer starts zeroed (cudaMemsetAsync on the stream) and every
// completed call leaves its counters zero; after a device-side timeout the
// buffers are cleared again before their next use.
enum ScratchUse {
  kScratchX16 = 0,
  kScratchGemv = 1,
  kScratchFfn = 2,
  kScratchNorm = 3,
  kScratchAttn = 4,
  kScratchLayer = 5,
  kScratchExact = 6
};
struct StreamScratch {
  int dev;
  cudaStream_t s;
  int use;
  void* p;
  size_t bytes;
  bool dirty;
};
std::mutex g_scratch_mu;
std::vector<StreamScratch> g_scratch;   // current buffers
std::vector<void*> g_scratch_retired;   // replaced buffers, never freed

int stream_scratch(int dev, cudaStream_t s, int use, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const bool zeroed = use == kScratchGemv;
  StreamScratch* cur = nullptr;
  for (auto& e : g_scratch)
    if (e.dev == dev && e.s == s && e.use == use) cur = &e;
  if (!cur || cur->bytes < bytes) {
    size_t want = (size_t)1 << 20;
    while (want < bytes) want <<= 1;
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    void* p = nullptr;
    const cudaError_t e = cudaMalloc(&p, want);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(APR_E_NOMEM, "scratch of %zu bytes: %s", want, cudaGetErrorString(e));
    }
    if (cur) {
      g_scratch_retired.push_back(cur->p);
      cur->p = p;
      cur->bytes = want;
    } else {
      g_scratch.push_back(StreamScratch{dev, s, use, p, want, false});
      cur = &g_scratch.back();
    }
    cur->dirty = zeroed;
  }
  if (cur->dirty) {
    const cudaError_t e = cudaMemsetAsync(cur->p, 0, cur->bytes, s);
    if (e != cudaSuccess) return fail(APR_E_LAUNCH, "scratch clear: %s", cudaGetErrorString(e));
    cur->dirty = false;
  }
  *out = cur->p;
  return APR_OK;
}

// After a device-side timeout some counters may be left nonzero.
void scratch_mark_dirty(int dev) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (auto& e : g_scratch)
    if (e.dev == dev && e.use == kScratchGemv) e.dirty = true;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct Problem {
  int qtype, leg, path;
  const void* W;
  const void* Wu;
  int n, k, T;
  const float* X;
  const float* R;
  float* Y;
  cudaStream_t s;
  int ldy = 0;  // floats between rows of Y and R; 0: n
};

int ldy_of(const Problem& p) { return p.ldy > 0 ? p.ldy : p.n; }

bool known_qtype(int q) {
  return q == APR_Q4_0 || q == APR_Q8_0 || q == APR_F16 || q == APR_Q4_K || q == APR_Q5_K || q == APR_Q6_K ||
         q == APR_IQ4_XS;
}
// k (the columns of every weight row) a whole number of the format's blocks;
// Q6_K rows (210 bytes per 256) start on 16-byte boundaries only when k is a
// multiple of 2048, IQ4_XS rows (136 bytes per 256) when k is a multiple of
// 512, and every route reads them from such boundaries
int k_unit(int qtype) {
  return qtype == kQ6_K ? 2048 : (qtype == kIQ4_XS ? 512 : (kquant(qtype) ? 256 : 32));
}
bool k_fits(int qtype, int k) { return k > 0 && k % k_unit(qtype) == 0; }

// a streaming GEMV kernel (integer-dot, whole-row, bulk, tensor-core or the K-quant one) takes the shape
bool gemv_streams(int qtype, int n, int k, int T, bool swiglu) {
  return kquant(qtype) || gemv_i8_fits(qtype, n, k, T, swiglu) || gemv_rows_fits(qtype, n, k, T, swiglu) ||
         gemv_bulk_fits(qtype, k, T, swiglu) || (!swiglu && block32_format(qtype) && gemv_tc_takes(n, k, T, false));
}

// Host-side checks; returns APR_OK, an error, or 1 for "nothing to do".
int check(const Problem& p, size_t x_elem_bytes = 4) {
  if (!known_qtype(p.qtype)) return fail(APR_E_QTYPE, "unsupported qtype %d", p.qtype);
  if (p.leg != APR_LEG_F16 && p.leg != APR_LEG_EXACT_F32) return fail(APR_E_INVAL, "unknown leg %d", p.leg);
  if (p.path != APR_PATH_AUTO && p.path != APR_PATH_GEMV && p.path != APR_PATH_GEMM)
    return fail(APR_E_INVAL, "unknown path %d", p.path);
  if (p.n < 0 || p.T < 0 || !k_fits(p.qtype, p.k))
    return fail(APR_E_INVAL, "bad sizes n=%d k=%d T=%d (need n >= 0, T >= 0, k > 0, k a multiple of %d)", p.n, p.k,
                p.T, k_unit(p.qtype));
  if (p.n > (1 << 24) || p.T > (1 << 24) || p.k > (1 << 20) || (int64_t)p.n * (p.k / 32) > (int64_t)1 << 31)
    return fail(APR_E_INVAL, "sizes beyond the supported limits");
  if (p.ldy < 0 || (p.ldy > 0 && p.ldy < p.n) || p.ldy > (1 << 28))
    return fail(APR_E_INVAL, "bad ldy %d (need 0, or n <= ldy <= 2^28; n = %d)", p.ldy, p.n);
  if (p.path == APR_PATH_GEMV && p.T > APR_GEMV_MAX_T)
    return fail(APR_E_INVAL, "the GEMV path takes T <= %d (got %d)", APR_GEMV_MAX_T, p.T);
  if (p.n == 0 || p.T == 0) return 1;
  if (!p.W || !p.X || !p.Y) return fail(APR_E_INVAL, "null pointer (W, X or Y)");
  const void* ptrs[5] = {p.W, p.Wu, p.X, p.R, p.Y};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(APR_E_ALIGN, "pointer %p is not 16-byte aligned", q);
  const size_t wbytes = (size_t)p.n * row_bytes_of(p.qtype, p.k);
  const size_t xbytes = (size_t)p.T * (size_t)p.k * x_elem_bytes;
  const size_t ybytes = ((size_t)(p.T - 1) * (size_t)ldy_of(p) + (size_t)p.n) * 4;  // first to last element
  if (overlap(p.Y, ybytes, p.X, xbytes)) return fail(APR_E_ALIAS, "Y overlaps X");
  if (overlap(p.Y, ybytes, p.W, wbytes)) return fail(APR_E_ALIAS, "Y overlaps W");
  if (p.Wu && overlap(p.Y, ybytes, p.Wu, wbytes)) return fail(APR_E_ALIAS, "Y overlaps Wu");
  if (p.R && p.R != p.Y && overlap(p.Y, ybytes, p.R, ybytes))
    return fail(APR_E_ALIAS, "Y partially overlaps residual");
  if (p.Wu && p.R) return fail(APR_E_INVAL, "the gate/up SwiGLU product takes no residual");
  return APR_OK;
}

int check_f16_in(const Problem& p) { return check(p, 2); }

int launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(APR_E_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
  return APR_OK;
}

int run(const Problem& p) {
  int rc = check(p);
  if (rc == 1) return APR_OK;
  if (rc != APR_OK) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != APR_OK) return rc;

  int path = p.path;
  if (path == APR_PATH_AUTO) path = p.T <= APR_AUTO_GEMV_MAX_T ? APR_PATH_GEMV : APR_PATH_GEMM;
  // The exact leg's tensor-core GEMM beats the CUDA-core GEMVs (their FFMA
  // work grows with T) from T = 5 for Q4_0 / Q8_0 (4096 x 4096 at T = 8: 21.6
  // against 31.6 us; 12288 x 4096: 52.8 against 79.8 us) and from T = 9 for
  // F16 and the K-quants (whose GEMVs take two rows a warp), and wherever no
  // streaming GEMV kernel takes the shape (the staged fallback is several
  // times slower): the GEMV path takes it there.
  int leg = p.leg;
  const int gemv_last_t = block32_format(p.qtype) ? 4 : 8;
  if (path == APR_PATH_GEMV && p.k % 256 == 0 &&
      (p.T > gemv_last_t || (p.qtype != APR_F16 && !gemv_streams(p.qtype, p.n, p.k, p.T, p.Wu != nullptr)))) {
    path = APR_PATH_GEMM;
    leg = APR_LEG_EXACT_F32;
  }
  if (path == APR_PATH_GEMV) {
    // the tensor-core GEMV multiplies integer codes: block formats only; the
    // integer-dot GEMV takes one and two tokens before it
    if (!block32_format(p.qtype) || !gemv_tc_takes(p.n, p.k, p.T, p.Wu != nullptr) ||
        gemv_i8_fits(p.qtype, p.n, p.k, p.T, p.Wu != nullptr))
      return launched(launch_gemv(p.qtype, p.W, p.Wu, p.n, p.k, p.X, p.T, p.Y, ldy_of(p), p.R, st->status, p.s),
                      "gemv");
    // tensor-core GEMV: the stream's scratch holds its split X, scales and
    // partial sums
    void* scratch = nullptr;
    rc = stream_scratch(st->dev, p.s, kScratchGemv, gemv_tc_scratch_bytes(p.n, p.k, p.T), &scratch);
    if (rc != APR_OK) return rc;
    char msg[256] = "";
    if (launch_gemv_tc(p.qtype, p.W, p.n, p.k, p.X, p.T, p.Y, ldy_of(p), p.R, scratch, st->status, p.s, msg,
                       sizeof msg) != 0)
      return fail(APR_E_LAUNCH, "%s", msg);
    return APR_OK;
  }
  // GEMM: the tensor-core kernels need every raw 256-column chunk of a weight
  // row to start on a 16-byte boundary (k % 256 == 0); other k run the FFMA
  // kernel (exact fp32, whatever the leg).
  if (p.k % 256 != 0)
    return launched(launch_gemm_simt(p.qtype, p.W, p.Wu, p.n, p.k, p.X, p.T, p.Y, ldy_of(p), p.R, p.s), "gemm_simt");
  if (leg == APR_LEG_EXACT_F32) {
    // the exact leg on the tensor cores: three fp16 products per term of the
    // split operands; the stream's scratch holds the split X, its token
    // exponents and the weight rows' exponents (and, for gate/up, the two
    // products before the SwiGLU)
    const size_t xs = (gemm_xs_scratch_bytes(p.n, p.k, p.T, false) + 255) & ~(size_t)255;
    const size_t gu = p.Wu ? 2 * (((size_t)p.T * p.n * 4 + 255) & ~(size_t)255) : 0;
    void* scratch = nullptr;
    rc = stream_scratch(st->dev, p.s, kScratchExact, xs + gu, &scratch);
    if (rc != APR_OK) return rc;
    char msg[256] = "";
    if (!p.Wu) {
      if (launch_gemm_xs(p.qtype, p.W, nullptr, p.n, p.k, p.X, p.T, p.Y, ldy_of(p), p.R, scratch, st->status, p.s,
                         msg, sizeof msg) != 0)
        return fail(APR_E_LAUNCH, "%s", msg);
      return APR_OK;
    }
    float* G = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + xs);
    float* U = G + (((size_t)p.T * p.n * 4 + 255) & ~(size_t)255) / 4;
    if (launch_gemm_xs(p.qtype, p.W, nullptr, p.n, p.k, p.X, p.T, G, p.n, nullptr, scratch, st->status, p.s, msg,
                       sizeof msg) != 0 ||
        launch_gemm_xs(p.qtype, p.Wu, nullptr, p.n, p.k, p.X, p.T, U, p.n, nullptr, scratch, st->status, p.s, msg,
                       sizeof msg) != 0)
      return fail(APR_E_LAUNCH, "%s", msg);
    return launched(launch_swiglu_rows(G, U, p.T, p.n, p.Y, ldy_of(p), p.s), "swiglu_rows");
  }

  // the stream's scratch holds the fp16 copy of X (at least kMinXRows rows)
  const GemmPlan plan = plan_gemm_tc(p.n, p.k, p.T, p.Wu != nullptr);
  const size_t count = (size_t)p.T * (size_t)p.k;
  void* x16 = nullptr;
  rc = stream_scratch(st->dev, p.s, kScratchX16, (size_t)padded_x_rows(p.T) * p.k * 2, &x16);
  if (rc != APR_OK) return rc;
  rc = launched(launch_x_to_f16(p.X, static_cast<uint16_t*>(x16), count, p.s), "x_to_f16");
  if (rc != APR_OK) return rc;
  char msg[256] = "";
  if (launch_gemm_tc(plan, p.qtype, p.W, p.Wu, p.n, p.k, static_cast<const uint16_t*>(x16), p.T, p.Y, ldy_of(p), p.R,
                     st->status, p.s, msg, sizeof msg, kEarlyWR, padded_x_rows(p.T)) != 0)
    return fail(APR_E_LAUNCH, "%s", msg);
  return APR_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// FFN sublayer: per chunk of rows, the norm into scratch, then gate/up SwiGLU
// into scratch, then down with the chunk's rows of X as residual and output.
int run_ffn(const apr_ffn_args& a) {
  if (!known_qtype(a.qtype)) return fail(APR_E_QTYPE, "unsupported qtype %d", a.qtype);
  if (a.leg != APR_LEG_F16 && a.leg != APR_LEG_EXACT_F32) return fail(APR_E_INVAL, "unknown leg %d", a.leg);
  if (!k_fits(a.qtype, a.hidden) || !k_fits(a.qtype, a.inter) || a.T < 0)
    return fail(APR_E_INVAL, "bad sizes hidden=%d inter=%d T=%d (need multiples of %d, T >= 0)", a.hidden, a.inter,
                a.T, k_unit(a.qtype));
  if (a.hidden > (1 << 20) || a.inter > (1 << 20) || a.T > (1 << 24) ||
      (int64_t)a.hidden * (a.inter / 32) > (int64_t)1 << 31)
    return fail(APR_E_INVAL, "sizes beyond the supported limits");
  if (!(a.eps >= 0.f) || a.eps > 3.402823466e38f) return fail(APR_E_INVAL, "eps must be finite and >= 0");
  if (a.T == 0) return APR_OK;
  if (!a.Wg || !a.Wu || !a.Wd || !a.norm_weight || !a.X) return fail(APR_E_INVAL, "null pointer");
  const void* ptrs[5] = {a.Wg, a.Wu, a.Wd, a.norm_weight, a.X};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(APR_E_ALIGN, "pointer %p is not 16-byte aligned", q);
  const size_t wgu = (size_t)a.inter * row_bytes_of(a.qtype, a.hidden);
  const size_t wd = (size_t)a.hidden * row_bytes_of(a.qtype, a.inter);
  const size_t xb = (size_t)a.T * a.hidden * 4;
  if (overlap(a.X, xb, a.Wg, wgu) || overlap(a.X, xb, a.Wu, wgu) || overlap(a.X, xb, a.Wd, wd) ||
      overlap(a.X, xb, a.norm_weight, (size_t)a.hidden * 4))
    return fail(APR_E_ALIAS, "X overlaps a weight or the norm weight");
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  const cudaStream_t s = (cudaStream_t)a.stream;
  const int chunk = a.T < APR_FFN_CHUNK_ROWS ? a.T : APR_FFN_CHUNK_ROWS;
  // h: the normed rows, fp32, or fp16 padded to kMinXRows rows
  const size_t h_bytes = align256(std::max((size_t)chunk * a.hidden * 4, (size_t)padded_x_rows(chunk) * a.hidden * 2));
  const size_t act_bytes = align256((size_t)chunk * a.inter * 4);
  void* scratch = nullptr;
  rc = stream_scratch(st->dev, s, kScratchFfn, h_bytes + act_bytes + (size_t)padded_x_rows(chunk) * a.inter * 2,
                      &scratch);
  if (rc != APR_OK) return rc;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  void* h = base;                                          // normed rows (fp16 or fp32)
  float* act = reinterpret_cast<float*>(base + h_bytes);   // SwiGLU output
  uint16_t* act16 = reinterpret_cast<uint16_t*>(base + h_bytes + act_bytes);
  for (int t0 = 0; t0 < a.T; t0 += chunk) {
    const int rows = a.T - t0 < chunk ? a.T - t0 : chunk;
    float* Xc = a.X + (size_t)t0 * a.hidden;
    const bool tc = a.leg == APR_LEG_F16 && rows > APR_AUTO_GEMV_MAX_T && a.hidden % 256 == 0 && a.inter % 256 == 0;
    rc = launched(launch_rmsnorm_rows(Xc, a.norm_weight, a.eps, rows, a.hidden, h, tc, s), "rmsnorm");
    if (rc != APR_OK) return rc;
    if (tc) {
      char msg[256] = "";
      const GemmPlan pg = plan_gemm_tc(a.inter, a.hidden, rows, true);
      // the SwiGLU output straight to fp16, the down GEMM's operand (the same
      // rounding the conversion pass would apply to the fp32 value)
      if (launch_gemm_tc(pg, a.qtype, a.Wg, a.Wu, a.inter, a.hidden, static_cast<const uint16_t*>(h), rows,
                         reinterpret_cast<float*>(act16), a.inter, nullptr, st->status, s, msg, sizeof msg,
                         kEarlyWR | kOutF16, padded_x_rows(rows)) != 0)
        return fail(APR_E_LAUNCH, "%s", msg);
      const GemmPlan pd = plan_gemm_tc(a.hidden, a.inter, rows, false);
      if (launch_gemm_tc(pd, a.qtype, a.Wd, nullptr, a.hidden, a.inter, act16, rows, Xc, a.hidden, Xc, st->status, s,
                         msg, sizeof msg, kEarlyWR, padded_x_rows(rows)) != 0)
        return fail(APR_E_LAUNCH, "%s", msg);
    } else {
      rc = run(Problem{a.qtype, a.leg, APR_PATH_AUTO, a.Wg, a.Wu, a.inter, a.hidden, rows,
                       static_cast<const float*>(h), nullptr, act, s});
      if (rc != APR_OK) return rc;
      rc = run(Problem{a.qtype, a.leg, APR_PATH_AUTO, a.Wd, nullptr, a.hidden, a.inter, rows, act, Xc, Xc, s});
      if (rc != APR_OK) return rc;
    }
  }
  return APR_OK;
}

// Normed projection: per chunk of rows, the norm into scratch (fp16 for the
// fp16 leg's tensor-core path, else fp32), then the projection.
int run_normed(const Problem& p, const float* w, float eps) {
  int rc = check(p);
  if (rc == 1) return APR_OK;
  if (rc != APR_OK) return rc;
  if (!(eps >= 0.f) || eps > 3.402823466e38f) return fail(APR_E_INVAL, "eps must be finite and >= 0");
  if (!w) return fail(APR_E_INVAL, "null norm weight");
  if (!aligned16(w)) return fail(APR_E_ALIGN, "pointer %p is not 16-byte aligned", (const void*)w);
  const size_t ybytes = ((size_t)(p.T - 1) * (size_t)ldy_of(p) + (size_t)p.n) * 4;
  if (overlap(p.Y, ybytes, w, (size_t)p.k * 4)) return fail(APR_E_ALIAS, "Y overlaps the norm weight");
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != APR_OK) return rc;
  int path = p.path;
  if (path == APR_PATH_AUTO) path = p.T <= APR_AUTO_GEMV_MAX_T ? APR_PATH_GEMV : APR_PATH_GEMM;
  const bool tc = p.leg == APR_LEG_F16 && path == APR_PATH_GEMM && p.k % 256 == 0;
  const int chunk = p.T < APR_FFN_CHUNK_ROWS ? p.T : APR_FFN_CHUNK_ROWS;
  void* h = nullptr;
  rc = stream_scratch(st->dev, p.s, kScratchNorm, tc ? (size_t)padded_x_rows(chunk) * p.k * 2 : (size_t)chunk * p.k * 4,
                      &h);
  if (rc != APR_OK) return rc;
  const int ldy = ldy_of(p);
  for (int t0 = 0; t0 < p.T; t0 += chunk) {
    const int rows = p.T - t0 < chunk ? p.T - t0 : chunk;
    const float* Xc = p.X + (size_t)t0 * p.k;
    float* Yc = p.Y + (size_t)t0 * ldy;
    const float* Rc = p.R ? p.R + (size_t)t0 * ldy : nullptr;
    rc = launched(launch_rmsnorm_rows(Xc, w, eps, rows, p.k, h, tc, p.s), "rmsnorm");
    if (rc != APR_OK) return rc;
    if (tc) {
      char msg[256] = "";
      const GemmPlan plan = plan_gemm_tc(p.n, p.k, rows, p.Wu != nullptr);
      if (launch_gemm_tc(plan, p.qtype, p.W, p.Wu, p.n, p.k, static_cast<const uint16_t*>(h), rows, Yc, ldy, Rc,
                         st->status, p.s, msg, sizeof msg, kEarlyWR, padded_x_rows(rows)) != 0)
        return fail(APR_E_LAUNCH, "%s", msg);
    } else {
      rc = run(Problem{p.qtype, p.leg, path, p.W, p.Wu, p.n, p.k, rows, static_cast<const float*>(h), Rc, Yc, p.s,
                       p.ldy});
      if (rc != APR_OK) return rc;
    }
  }
  return APR_OK;
}

// One prefill layer, chunk by chunk: the attention sublayer (norm, q/k/v
// projections with k and v written into the cache rows of the chunk, the
// causal attention, the output projection added into X), then the FFN
// sublayer on the chunk's rows of X.
int run_layer(const apr_layer_args& a) {
  if (!known_qtype(a.qtype)) return fail(APR_E_QTYPE, "unsupported qtype %d", a.qtype);
  if (a.leg != APR_LEG_F16 && a.leg != APR_LEG_EXACT_F32) return fail(APR_E_INVAL, "unknown leg %d", a.leg);
  if (a.head_dim != 256) return fail(APR_E_INVAL, "head_dim must be 256 (got %d)", a.head_dim);
  if (!k_fits(a.qtype, a.hidden) || !k_fits(a.qtype, a.inter) || a.T < 0 || a.pos0 < 0 ||
      a.num_heads <= 0 || a.num_kv_heads <= 0 || a.chunk < 0)
    return fail(APR_E_INVAL, "bad sizes hidden=%d inter=%d T=%d pos0=%d heads=%d kv_heads=%d chunk=%d", a.hidden,
                a.inter, a.T, a.pos0, a.num_heads, a.num_kv_heads, a.chunk);
  if (a.num_heads % a.num_kv_heads != 0)
    return fail(APR_E_INVAL, "num_heads (%d) must be a multiple of num_kv_heads (%d)", a.num_heads, a.num_kv_heads);
  const long long qd = (long long)a.num_heads * 256, kvd = (long long)a.num_kv_heads * 256;
  if (qd > (1 << 20) || !k_fits(a.qtype, (int)qd))
    return fail(APR_E_INVAL, "the out projection's k = num_heads x 256 = %lld must be a multiple of %d", qd,
                k_unit(a.qtype));
  if (a.hidden > (1 << 20) || a.inter > (1 << 20) || a.T > (1 << 24) || a.chunk > (1 << 20) ||
      qd + 2 * kvd > (1 << 24) || (long long)a.pos0 + a.T > (1LL << 30) || kvd / 64 > 65535 ||
      (long long)a.hidden * (a.inter / 32) > (1LL << 31) || (qd + 2 * kvd) * (a.hidden / 32) > (1LL << 31) ||
      (long long)a.hidden * (qd / 32) > (1LL << 31))
    return fail(APR_E_INVAL, "sizes beyond the supported limits");
  if (!(a.eps >= 0.f) || a.eps > 3.402823466e38f) return fail(APR_E_INVAL, "eps must be finite and >= 0");
  if (a.T == 0) return APR_OK;
  const void* ptrs[10] = {a.Wqkv, a.Wo, a.Wg, a.Wu, a.Wd, a.attn_norm, a.ffn_norm, a.X, a.K_cache, a.V_cache};
  for (const void* q : ptrs) {
    if (!q) return fail(APR_E_INVAL, "null pointer");
    if (!aligned16(q)) return fail(APR_E_ALIGN, "pointer %p is not 16-byte aligned", q);
  }
  const size_t hrow = row_bytes_of(a.qtype, a.hidden);  // bytes of a weight row over hidden columns
  const size_t wqkv = (size_t)(qd + 2 * kvd) * hrow, wo = (size_t)a.hidden * row_bytes_of(a.qtype, (int)qd);
  const size_t wgu = (size_t)a.inter * hrow, wd = (size_t)a.hidden * row_bytes_of(a.qtype, a.inter);
  const size_t xb = (size_t)a.T * a.hidden * 4, cb = ((size_t)a.pos0 + a.T) * (size_t)kvd * 4;
  const void* wts[7] = {a.Wqkv, a.Wo, a.Wg, a.Wu, a.Wd, a.attn_norm, a.ffn_norm};
  const size_t wsz[7] = {wqkv, wo, wgu, wgu, wd, (size_t)a.hidden * 4, (size_t)a.hidden * 4};
  for (int i = 0; i < 7; ++i)
    if (overlap(a.X, xb, wts[i], wsz[i]) || overlap(a.K_cache, cb, wts[i], wsz[i]) ||
        overlap(a.V_cache, cb, wts[i], wsz[i]))
      return fail(APR_E_ALIAS, "X or a cache overlaps a weight or a norm weight");
  if (overlap(a.X, xb, a.K_cache, cb) || overlap(a.X, xb, a.V_cache, cb) || overlap(a.K_cache, cb, a.V_cache, cb))
    return fail(APR_E_ALIAS, "X, K_cache and V_cache must not overlap");
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  const cudaStream_t s = (cudaStream_t)a.stream;
  const int chunk = a.chunk > 0 ? a.chunk : 512;
  const int rmax = a.T < chunk ? a.T : chunk;
  // the chunk's normed rows (fp32 at most), q and the attention output
  const size_t h_bytes = align256(std::max((size_t)rmax * a.hidden * 4, (size_t)padded_x_rows(rmax) * a.hidden * 2));
  // (the attention output is fp32, or fp16 over at least the 16 rows the
  // tensor-core GEMM reads)
  const size_t q_bytes = align256(std::max((size_t)rmax * qd * 4, (size_t)padded_x_rows(rmax) * qd * 2));
  void* scratch = nullptr;
  rc = stream_scratch(st->dev, s, kScratchLayer, h_bytes + 2 * q_bytes, &scratch);
  if (rc != APR_OK) return rc;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  void* h = base;
  float* qbuf = reinterpret_cast<float*>(base + h_bytes);
  float* abuf = reinterpret_cast<float*>(base + h_bytes + q_bytes);
  // the attention's fp16 copies of the cache rows, sized for the last chunk
  void* ascratch = nullptr;
  rc = stream_scratch(st->dev, s, kScratchAttn, prefill_attention_scratch_bytes(rmax, a.pos0 + a.T - rmax,
                                                                                a.num_kv_heads),
                      &ascratch);
  if (rc != APR_OK) return rc;
  const uint8_t* Wq = static_cast<const uint8_t*>(a.Wqkv);
  const uint8_t* Wk = Wq + (size_t)qd * hrow;
  const uint8_t* Wv = Wk + (size_t)kvd * hrow;
  for (int t0 = 0; t0 < a.T; t0 += chunk) {
    const int rows = a.T - t0 < chunk ? a.T - t0 : chunk;
    const int pos = a.pos0 + t0;
    float* Xc = a.X + (size_t)t0 * a.hidden;
    // 1. norm, then q, k, v: k and v straight into the cache rows pos ..
    const bool tc = a.leg == APR_LEG_F16 && rows > APR_AUTO_GEMV_MAX_T && a.hidden % 256 == 0;
    rc = launched(launch_rmsnorm_rows(Xc, a.attn_norm, a.eps, rows, a.hidden, h, tc, s), "rmsnorm");
    if (rc != APR_OK) return rc;
    const void* Wp[3] = {Wq, Wk, Wv};
    float* Yp[3] = {qbuf, a.K_cache + (size_t)pos * kvd, a.V_cache + (size_t)pos * kvd};
    const int np[3] = {(int)qd, (int)kvd, (int)kvd};
    if (tc) {
      // one GEMM over the fused weight (its q, k and v row ranges are
      // multiples of 256 rows): q rows to the q buffer, k and v rows straight
      // into the cache rows pos ..
      char msg[256] = "";
      const int nqkv = (int)(qd + 2 * kvd);
      const GemmPlan plan = plan_gemm_tc(nqkv, a.hidden, rows, false);
      const OutRegions reg{Yp[1], Yp[2], (int)qd, (int)(qd + kvd), (int)kvd, (int)kvd};
      if (launch_gemm_tc(plan, a.qtype, a.Wqkv, nullptr, nqkv, a.hidden, static_cast<const uint16_t*>(h), rows,
                         qbuf, (int)qd, nullptr, st->status, s, msg, sizeof msg, kEarlyWR, padded_x_rows(rows),
                         &reg) != 0)
        return fail(APR_E_LAUNCH, "%s", msg);
    } else {
      for (int j = 0; j < 3; ++j) {
        rc = run(Problem{a.qtype, a.leg, APR_PATH_AUTO, Wp[j], nullptr, np[j], a.hidden, rows,
                         static_cast<const float*>(h), nullptr, Yp[j], s});
        if (rc != APR_OK) return rc;
      }
    }
    // 2. causal attention of the chunk's rows over the cache rows 0 .. pos + rows - 1;
    // on the tensor-core route its output is written as fp16, the output
    // projection's operand (the rounding the conversion pass would apply)
    char msg[256] = "";
    if (launch_prefill_attention(qbuf, a.K_cache, a.V_cache, abuf, rows, pos, a.num_heads, a.num_kv_heads, ascratch,
                                 st->status, s, msg, sizeof msg, tc) != 0)
      return fail(APR_E_LAUNCH, "%s", msg);
    // 3. output projection added into the chunk's rows of X
    if (tc) {
      const GemmPlan plan = plan_gemm_tc(a.hidden, (int)qd, rows, false);
      if (launch_gemm_tc(plan, a.qtype, a.Wo, nullptr, a.hidden, (int)qd, reinterpret_cast<const uint16_t*>(abuf),
                         rows, Xc, a.hidden, Xc, st->status, s, msg, sizeof msg, kEarlyWR, padded_x_rows(rows)) != 0)
        return fail(APR_E_LAUNCH, "%s", msg);
    } else {
      rc = run(Problem{a.qtype, a.leg, APR_PATH_AUTO, a.Wo, nullptr, a.hidden, (int)qd, rows, abuf, Xc, Xc, s});
      if (rc != APR_OK) return rc;
    }
    // 4. the FFN sublayer on the same rows
    apr_ffn_args f{a.qtype, a.leg, a.Wg, a.Wu, a.Wd, a.hidden, a.inter, rows, a.ffn_norm, a.eps, Xc, a.stream};
    rc = run_ffn(f);
    if (rc != APR_OK) return rc;
  }
  return APR_OK;
}

}  // namespace

namespace apr {

int set_error(int code, const char* msg) {
  snprintf(t_msg, sizeof t_msg, "%s", msg);
  return code;
}

int check_gemm_args(int qtype, const void* W, int n, int k, const float* X, int T, const float* Y, const float* R) {
  t_msg[0] = 0;
  return check(Problem{qtype, APR_LEG_F16, APR_PATH_GEMM, W, nullptr, n, k, T, X, R, const_cast<float*>(Y), nullptr});
}

unsigned* status_word_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned*>(p);
}

}  // namespace apr

extern "C" {

int apr_gemv_max_T(void) { return APR_GEMV_MAX_T; }

const char* apr_last_error(void) { return t_msg; }

int apr_qgemm(int qtype, const void* W, int n, int k, const float* X, int T, float* Y, const float* residual,
              apr_stream_t stream) {
  t_msg[0] = 0;
  return run(Problem{qtype, APR_LEG_F16, APR_PATH_AUTO, W, nullptr, n, k, T, X, residual, Y, (cudaStream_t)stream});
}

int apr_qgemm_gate_up_swiglu(int qtype, const void* Wg, const void* Wu, int n, int k, const float* X, int T, float* Y,
                             apr_stream_t stream) {
  t_msg[0] = 0;
  if (!Wu && n > 0 && T > 0) return fail(APR_E_INVAL, "null up weight");
  return run(Problem{qtype, APR_LEG_F16, APR_PATH_AUTO, Wg, Wu, n, k, T, X, nullptr, Y, (cudaStream_t)stream});
}

int apr_qgemv(int qtype, const void* W, int n, int k, const float* X, int T, float* Y, const float* residual,
              apr_stream_t stream) {
  t_msg[0] = 0;
  return run(Problem{qtype, APR_LEG_EXACT_F32, APR_PATH_GEMV, W, nullptr, n, k, T, X, residual, Y,
                     (cudaStream_t)stream});
}

int apr_qgemm_ex(const apr_qgemm_args* a) {
  t_msg[0] = 0;
  if (!a) return fail(APR_E_INVAL, "null argument struct");
  return run(Problem{a->qtype, a->leg, a->path, a->W, a->Wu, a->n, a->k, a->T, a->X, a->residual, a->Y,
                     (cudaStream_t)a->stream, a->ldy});
}

int apr_qgemm_rmsnorm(const apr_qgemm_args* a, const float* norm_weight, float eps) {
  t_msg[0] = 0;
  if (!a) return fail(APR_E_INVAL, "null argument struct");
  return run_normed(Problem{a->qtype, a->leg, a->path, a->W, a->Wu, a->n, a->k, a->T, a->X, a->residual, a->Y,
                            (cudaStream_t)a->stream, a->ldy},
                    norm_weight, eps);
}

int apr_ffn_sublayer(const apr_ffn_args* a) {
  t_msg[0] = 0;
  if (!a) return fail(APR_E_INVAL, "null argument struct");
  return run_ffn(*a);
}

int apr_prefill_layer(const apr_layer_args* a) {
  t_msg[0] = 0;
  if (!a) return fail(APR_E_INVAL, "null argument struct");
  return run_layer(*a);
}

int apr_convert_f32_to_f16(const float* X, long long count, void* X16, apr_stream_t stream) {
  t_msg[0] = 0;
  if (count < 0) return fail(APR_E_INVAL, "negative count");
  if (count == 0) return APR_OK;
  if (!X || !X16) return fail(APR_E_INVAL, "null pointer");
  if (!aligned16(X) || !aligned16(X16)) return fail(APR_E_ALIGN, "X and X16 must be 16-byte aligned");
  if (overlap(X, (size_t)count * 4, X16, (size_t)count * 2)) return fail(APR_E_ALIAS, "X16 overlaps X");
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  return launched(launch_x_to_f16(X, static_cast<uint16_t*>(X16), (size_t)count, (cudaStream_t)stream),
                  "convert_f32_to_f16");
}

int apr_qgemm_f16_in(int qtype, const void* W, const void* Wu, int n, int k, const void* X16, int T, float* Y,
                     const float* residual, apr_stream_t stream) {
  t_msg[0] = 0;
  // Checked as an f32 problem of the same shape, then against the fp16 size.
  Problem p{qtype, APR_LEG_F16, APR_PATH_GEMM, W, Wu, n, k, T, static_cast<const float*>(X16), residual, Y,
            (cudaStream_t)stream};
  if (k % 256 != 0 && k > 0) return fail(APR_E_INVAL, "the fp16-input GEMM needs k %% 256 == 0 (got %d)", k);
  int rc = check_f16_in(p);
  if (rc == 1) return APR_OK;
  if (rc != APR_OK) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != APR_OK) return rc;
  const GemmPlan plan = plan_gemm_tc(n, k, T, Wu != nullptr);
  char msg[256] = "";
  if (launch_gemm_tc(plan, qtype, W, Wu, n, k, static_cast<const uint16_t*>(X16), T, Y, n, residual, st->status,
                     (cudaStream_t)stream, msg, sizeof msg, kEarlyW) != 0)
    return fail(APR_E_LAUNCH, "%s", msg);
  return APR_OK;
}

int apr_prefill_attention(const float* Q, const float* K_cache, const float* V_cache, float* out, int T, int pos0,
                          int num_heads, int num_kv_heads, int head_dim, apr_stream_t stream) {
  t_msg[0] = 0;
  if (T < 0 || pos0 < 0 || num_heads <= 0 || num_kv_heads <= 0)
    return fail(APR_E_INVAL, "bad sizes T=%d pos0=%d num_heads=%d num_kv_heads=%d", T, pos0, num_heads,
                num_kv_heads);
  if (num_heads % num_kv_heads != 0)
    return fail(APR_E_INVAL, "num_heads (%d) must be a multiple of num_kv_heads (%d)", num_heads, num_kv_heads);
  if (head_dim != 256) return fail(APR_E_INVAL, "head_dim must be 256 (got %d)", head_dim);
  // positions, the widths of Q and of the caches (the V transpose runs one
  // grid row per 64 cache columns), and the attention grid
  if ((long long)pos0 + T > (1LL << 30) || (long long)num_heads * 256 > (1LL << 24) ||
      (long long)num_kv_heads * 256 / 64 > 65535 || (long long)((T + 127) / 128) * num_heads > 0x7FFFFFFFLL)
    return fail(APR_E_INVAL, "sizes beyond the supported limits");
  if (T == 0) return APR_OK;
  if (!Q || !K_cache || !V_cache || !out) return fail(APR_E_INVAL, "null pointer");
  for (const void* p : {(const void*)Q, (const void*)K_cache, (const void*)V_cache, (const void*)out})
    if (!aligned16(p)) return fail(APR_E_ALIGN, "pointer %p is not 16-byte aligned", p);
  const size_t qbytes = (size_t)T * num_heads * 256 * 4;
  const size_t cbytes = ((size_t)pos0 + T) * num_kv_heads * 256 * 4;
  if (overlap(out, qbytes, Q, qbytes) || overlap(out, qbytes, K_cache, cbytes) || overlap(out, qbytes, V_cache, cbytes))
    return fail(APR_E_ALIAS, "out overlaps Q or the K / V cache");
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  // the stream's scratch holds the fp16 copies of K and of V transposed
  void* scratch = nullptr;
  rc = stream_scratch(st->dev, (cudaStream_t)stream, kScratchAttn,
                      prefill_attention_scratch_bytes(T, pos0, num_kv_heads), &scratch);
  if (rc != APR_OK) return rc;
  char msg[256] = "";
  if (launch_prefill_attention(Q, K_cache, V_cache, out, T, pos0, num_heads, num_kv_heads, scratch, st->status,
                               (cudaStream_t)stream, msg, sizeof msg) != 0)
    return fail(APR_E_LAUNCH, "%s", msg);
  return APR_OK;
}

int apr_dequant(int qtype, const void* W, int n, int k, float* out, apr_stream_t stream) {
  t_msg[0] = 0;
  if (!known_qtype(qtype)) return fail(APR_E_QTYPE, "unsupported qtype %d", qtype);
  if (n < 0 || !k_fits(qtype, k)) return fail(APR_E_INVAL, "bad sizes n=%d k=%d", n, k);
  if (n > (1 << 24) || k > (1 << 20) || (int64_t)n * (k / 32) > (int64_t)1 << 31)
    return fail(APR_E_INVAL, "sizes beyond the supported limits");
  if (n == 0) return APR_OK;
  if (!W || !out) return fail(APR_E_INVAL, "null pointer");
  if (qtype == APR_F16 && ((uintptr_t)W & 1) != 0) return fail(APR_E_ALIGN, "an F16 weight must be 2-byte aligned");
  const size_t wbytes = (size_t)n * row_bytes_of(qtype, k);
  if (overlap(out, (size_t)n * k * 4, W, wbytes)) return fail(APR_E_ALIAS, "out overlaps W");
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  return launched(launch_dequant(qtype, W, n, k, out, (cudaStream_t)stream), "dequant");
}

int apr_read_stream(const void* src, long long bytes, apr_stream_t stream) {
  t_msg[0] = 0;
  if (bytes < 0 || bytes % 16 != 0) return fail(APR_E_INVAL, "bytes must be a non-negative multiple of 16");
  if (bytes == 0) return APR_OK;
  if (!src) return fail(APR_E_INVAL, "null pointer");
  if (!aligned16(src)) return fail(APR_E_ALIGN, "pointer %p is not 16-byte aligned", src);
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  return launched(launch_read_stream(src, bytes, st->status, (cudaStream_t)stream), "read_stream");
}

int apr_test_bounded_wait(unsigned limit_us, apr_stream_t stream) {
  t_msg[0] = 0;
  if (limit_us < 1 || limit_us > 1000000) return fail(APR_E_INVAL, "limit_us must be in [1, 1000000] (got %u)", limit_us);
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  return launched(launch_bounded_wait(1000ull * limit_us, st->status, (cudaStream_t)stream), "bounded_wait");
}

int apr_stream_status(apr_stream_t stream) {
  t_msg[0] = 0;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != APR_OK) return rc;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(APR_E_LAUNCH, "stream: %s", cudaGetErrorString(e));
  unsigned v = 0;
  e = cudaMemcpy(&v, st->status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(APR_E_LAUNCH, "status read: %s", cudaGetErrorString(e));
  if (v) {
    const unsigned zero = 0;
    cudaMemcpy(st->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    scratch_mark_dirty(st->dev);
    return fail(APR_E_TIMEOUT, "a kernel's bounded wait gave up (status 0x%x)", v);
  }
  return APR_OK;
}

}  // extern "C"
