// Launchers shared between the C ABI (api.cu) and the kernel files. Host only.
// Y (and the residual R) hold T rows of n floats, ldy floats apart (ldy >= n).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace apr {

constexpr int kF16 = 1;
constexpr int kQ4_0 = 2;
constexpr int kQ8_0 = 8;
constexpr int kQ4_K = 12;  // 256-element superblocks of 144 bytes (k % 256 == 0)
constexpr int kQ5_K = 13;  // 256-element superblocks of 176 bytes (k % 256 == 0)
constexpr int kQ6_K = 14;  // 256-element superblocks of 210 bytes (k % 2048 == 0: rows on 16-byte boundaries)
constexpr int kIQ4_XS = 23;  // 256-element superblocks of 136 bytes (k % 512 == 0: rows on 16-byte boundaries)
// the 256-element superblock formats (the K-quants and IQ4_XS)
inline bool kquant(int qtype) { return qtype == kQ4_K || qtype == kQ5_K || qtype == kQ6_K || qtype == kIQ4_XS; }

// bytes of 32 consecutive elements of a weight row (one block; 64 for F16; an
// eighth of a Q4_K, Q5_K or IQ4_XS superblock); 0 for Q6_K, whose eighth of a
// superblock is not a whole number of bytes
inline int block_bytes(int qtype) {
  return qtype == kQ4_0 || qtype == kQ4_K
             ? 18
             : (qtype == kQ8_0 ? 34 : (qtype == kQ5_K ? 22 : (qtype == kQ6_K ? 0 : (qtype == kIQ4_XS ? 17 : 64))));
}
// bytes of one weight row of k elements (k a multiple of the format's unit)
inline size_t row_bytes_of(int qtype, int k) {
  return qtype == kQ6_K ? (size_t)(k / 256) * 210 : (size_t)(k / 32) * (size_t)block_bytes(qtype);
}
// formats of one scale and 32 codes per 32-element block (the block-GEMV kernels)
inline bool block32_format(int qtype) { return qtype == kQ4_0 || qtype == kQ8_0; }

// Epilogue of a projection. kEpiGluPair: gate/up SwiGLU computed by a
// cluster pair of CTAs, one per weight (gemm_tc.cu).
enum Epilogue { kEpiPlain = 0, kEpiResidual = 1, kEpiSwiGLU = 2, kEpiGluPair = 3 };

// Standalone dequant (dequant.cu).
cudaError_t launch_dequant(int qtype, const void* W, int n, int k, float* out, cudaStream_t s);

// Small-T GEMV, exact fp32. Wu != nullptr: gate/up SwiGLU. Takes the
// whole-row streaming kernel (gemv_rows.cu) when a stage holds a row, else the
// chunked bulk-copy kernel (gemv_bulk.cu), else the staged kernel (gemv.cu).
// The first two read W before the preceding kernel on the stream has
// finished (it must not be that kernel's output).
cudaError_t launch_gemv(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T,
                        float* Y, int ldy, const float* R, unsigned* status, cudaStream_t s);
size_t gemv_rows_smem(int qtype, int k, int T);
bool gemv_rows_fits(int qtype, int n, int k, int T, bool swiglu);
cudaError_t launch_gemv_rows(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T,
                             float* Y, const float* R, unsigned* status, cudaStream_t s);
// T = 1, 2 with integer dot products (gemv_i8.cu): X per 32-block in fixed
// point as three signed byte digits, dp4a against the codes, fp32 per block;
// Y and R rows ldy apart.
bool gemv_i8_fits(int qtype, int n, int k, int T, bool swiglu);
cudaError_t launch_gemv_i8(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y,
                           int ldy, const float* R, unsigned* status, cudaStream_t s);
// The T = 1 GEMV's data movement alone (gemv_i8.cu): `bytes` (a multiple of
// 16, src 16-byte aligned) streamed into shared memory and dropped.
cudaError_t launch_read_stream(const void* src, long long bytes, unsigned* status, cudaStream_t s);
size_t gemv_bulk_smem(int qtype, int k, int T, bool swiglu);
bool gemv_bulk_fits(int qtype, int k, int T, bool swiglu);
cudaError_t launch_gemv_bulk(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T,
                             float* Y, int ldy, const float* R, unsigned* status, cudaStream_t s);

// Tensor-core GEMV (gemv_tc.cu): fp16 integer codes x three fp16 pieces of X
// (every product exact), block scales applied in fp32. gemv_tc_takes() is the
// dispatch rule: T <= kGemvTcMaxT, k % 256 == 0, n <= 2097152, no gate/up,
// and T large enough that it beats the CUDA-core kernels. Needs
// gemv_tc_scratch_bytes() of device scratch whose first bytes (the ticket
// counters) are zero; each completed launch leaves them zero, so successive
// launches on one stream may share it. The kernel reads W before the
// preceding kernel on the stream has finished (it must not be that kernel's
// output). Returns 0, or -1 with a message in msg.
constexpr int kGemvTcMaxT = 4;
bool gemv_tc_takes(int n, int k, int T, bool swiglu);
size_t gemv_tc_scratch_bytes(int n, int k, int T);
int launch_gemv_tc(int qtype, const void* W, int n, int k, const float* X, int T, float* Y, int ldy, const float* R,
                   void* scratch, unsigned* status, cudaStream_t s, char* msg, size_t msg_len);

// Row RMSNorm y = x / sqrt(mean(x^2) + eps) * w over T rows of k floats
// (k % 4 == 0), into fp16 (f16) or fp32 rows of k (rmsnorm.cu). Plain stream
// order; it lets the next kernel launch at its start.
cudaError_t launch_rmsnorm_rows(const float* X, const float* w, float eps, int T, int k, void* out, bool f16,
                                cudaStream_t s);

// Causal prefill attention, head_dim 256, fp16 tensor-core inputs, fp32
// online softmax (attention.cu): Q and O [T][num_heads * 256], the caches
// [>= pos0 + T][num_kv_heads * 256], all f32 and 16-byte aligned; rows of the
// caches at or past pos0 + T are never read. Three plain launches in stream
// order: K and V (transposed) to fp16 into `scratch`
// (prefill_attention_scratch_bytes, 256-byte aligned), then the attention.
// Returns 0, or -1 with a message.
size_t prefill_attention_scratch_bytes(int T, int pos0, int num_kv_heads);
// o16: O is written as fp16 (round to nearest even of the fp32 value; O
// then points to uint16 [T][num_heads * 256]), the next GEMM's operand.
int launch_prefill_attention(const float* Q, const float* K, const float* V, float* O, int T, int pos0,
                             int num_heads, int num_kv_heads, void* scratch, unsigned* status, cudaStream_t s,
                             char* msg, size_t msg_len, bool o16 = false);

// Exact-fp32 FFMA GEMM for any k % 32 == 0 (gemm_simt.cu).
cudaError_t launch_gemm_simt(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T,
                             float* Y, int ldy, const float* R, cudaStream_t s);

// fp16 copy of X, round to nearest even (gemm_tc.cu). Launched in plain
// stream order, so it starts after the preceding kernel has completed.
cudaError_t launch_x_to_f16(const float* X, uint16_t* X16, size_t count, cudaStream_t s);

// Shape of a tensor-core GEMM launch: token-tile width (128 or 256) and split
// over k (1, or 2 CTAs per tile as a cluster that combines its halves in
// distributed shared memory; no workspace either way).
struct GemmPlan {
  int bn = 128;
  int nsplit = 1;
  bool pair = false;  // gate/up: a cluster pair of CTAs per 256-token tile, one weight each
};
GemmPlan plan_gemm_tc(int n, int k, int T, bool swiglu);

// tcgen05 fp16-input GEMM; needs k % 256 == 0 and X16 = fp16(X) (gemm_tc.cu).
// `status` is the device status word. Launched with programmatic stream
// serialization: it waits for the preceding kernel before it touches X16 and
// Y. `early` says what it reads before that: kEarlyW the weights (never the
// preceding kernel's output: the header's stream-order rule), kEarlyWR the
// weights and the residual (launched right after the library's own
// conversion or norm kernel, which starts only once everything before it has
// completed), kEarlyNone nothing.
enum { kEarlyNone = 0, kEarlyWR = 1, kEarlyW = 2 };
// Output rows of a plain tensor-core GEMM sent to up to three places by row
// range: rows [0, r1) to Y (ldy apart), rows [r1, r2) to y1 (row - r1, ld1
// apart), rows [r2, n) to y2 (row - r2, ld2 apart); y1 == nullptr: all to Y.
// r1 and r2 are multiples of 128 (a tile's rows go to one place).
struct OutRegions {
  float* y1;
  float* y2;
  int r1, r2, ld1, ld2;
};

// A flag or-ed into `early` for a gate/up GEMM: the SwiGLU output is written
// as fp16 (round to nearest even; Y is then a uint16 buffer, ldy counted in
// its elements), the operand the next GEMM reads.
constexpr int kOutF16 = 64;
// x_rows: the rows of X16 the kernel may read (>= T; 0 means T). Rows past T
// only feed output columns that are never stored; a buffer of at least
// kMinXRows rows avoids the slow TMA loads from a tensor of fewer rows
// (measured on GB300: 28.7 against 12.6 us at T = 15 and 16).
constexpr int kMinXRows = 16;
inline int padded_x_rows(int T) { return T < kMinXRows ? kMinXRows : T; }
int launch_gemm_tc(const GemmPlan& plan, int qtype, const void* W, const void* Wu, int n, int k, const uint16_t* X16,
                   int T, float* Y, int ldy, const float* R, unsigned* status, cudaStream_t s, char* msg,
                   size_t msg_len, int early, int x_rows = 0, const OutRegions* regions = nullptr);

// A kernel that waits (bounded, limit_ns) on an mbarrier nothing arrives on,
// then records the timeout in the status word and returns (selftest.cu).
cudaError_t launch_bounded_wait(unsigned long long limit_ns, unsigned* status, cudaStream_t s);

// Exact leg on the tensor cores (gemm_tc.cu), k % 256 == 0, one weight (Wu
// must be null): per weight row an exponent e (max |d| * max |q'| * 2^e in
// [2^14, 2^15)), X split per token into two fp16 pieces of X * 2^e', then
// W1.X1 + W1.X2 + W2.X1 per 16-k step with W * 2^e = W1 + W2, fp32
// accumulation restarted every 256 k and summed in fp32, the powers of two
// undone in the epilogue. Two plain launches (row exponents, the X split)
// and the GEMM; `scratch` holds gemm_xs_scratch_bytes(). Returns 0, or -1
// with a message.
size_t gemm_xs_scratch_bytes(int n, int k, int T, bool swiglu);
// y = silu(g) * u over T rows of n (G, U dense; rows of Y ldy apart).
cudaError_t launch_swiglu_rows(const float* G, const float* U, int T, int n, float* Y, int ldy, cudaStream_t s);
int launch_gemm_xs(int qtype, const void* W, const void* Wu, int n, int k, const float* X, int T, float* Y, int ldy,
                   const float* R, void* scratch, unsigned* status, cudaStream_t s, char* msg, size_t msg_len);

// Shared with the allocation-free entry point (api.cu): sets this thread's error
// message and returns `code`; checks the arguments of a plain / residual GEMM
// call (APR_OK, an error, or 1 for "nothing to do"); device address of the
// status word of the current device (nullptr on failure). None allocates.
int set_error(int code, const char* msg);
int check_gemm_args(int qtype, const void* W, int n, int k, const float* X, int T, const float* Y, const float* R);
unsigned* status_word_address();

}  // namespace apr
