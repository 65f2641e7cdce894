/*
 * apr_qgemm.h — C ABI of the GB300 (sm_103a) prefill projections over GGUF
 * Q4_0 / Q8_0 / Q4_K / Q5_K / Q6_K / IQ4_XS block-quantized weights and F16
 * weights.
 *
 * Every projection of a batched (chunked) prompt prefill is ONE product over
 * the chunk's T token rows, instead of T per-token GEMVs:
 *
 *     Y[T][n] = X[T][k] . dequant(W)[n][k]^T  (+ R[T][n])
 *
 * (aprender-serve 0.70.2, src/cuda/executor/gdn_prefill_ops.rs, doc of
 * qwen35_project_rows: all operands row major, W is [n x k]; the chunked
 * driver of src/gguf/cuda/forward_qwen35_cuda_prefill.rs, module doc, runs
 * every projection as one product over the chunk's rows.)
 *
 * Weight format (GGUF blocks of 32 weights along k, kept in their on-disk
 * array-of-blocks order — oxibonsai-kernels 0.1.4,
 * src/gpu_backend/cuda_q_std_prefill.rs, module doc "Weight layout"; block
 * size and scale position from that page's test make_q4_0_zeros):
 *   Q4_0 (18 bytes): fp16 d (little endian) then 16 bytes; byte j holds
 *                    element j in its low nibble and element j+16 in its high
 *                    nibble; w = d * (nibble - 8).
 *   Q8_0 (34 bytes): fp16 d then 32 int8 q; w = d * q.
 *   F16  (64 bytes per 32 weights): each weight its own IEEE binary16 value,
 *                    little endian (the F16 arm of aprender-serve
 *                    qwen35_dequant_f32, and its test
 *                    f16_weight_dequantizes_on_the_device). Every F16 call
 *                    takes k % 32 == 0 like the block formats; on the fp16
 *                    leg the weights enter the tensor cores unrounded.
 *   Q4_K (144 bytes per 256 weights, k % 256 == 0): a format the pages
 *                    dispatch (qwen35_dequant_f32, grid (n, k.div_ceil(256)))
 *                    without printing its layout, taken as the GGUF
 *                    superblock: fp16 d, fp16 dmin, 12 bytes of 6-bit
 *                    sub-block scales sc and mins m (scales 0-3 and mins 0-3
 *                    in the low 6 bits of bytes 0-3 and 4-7; scales 4-7 and
 *                    mins 4-7 in the low and high nibbles of bytes 8-11, their
 *                    top two bits in the top two bits of bytes 0-3 and 4-7),
 *                    then 128 code bytes: byte 32g + l holds element 64g + l
 *                    (low nibble) and 64g + 32 + l (high nibble);
 *                    w = d * sc_j * q - dmin * m_j for element e, j = e / 32.
 *   Q5_K (176 bytes per 256 weights, k % 256 == 0): also dispatched by the
 *                    pages without a printed layout; taken as the GGUF
 *                    superblock: the first 16 bytes as in Q4_K, then 32 bytes
 *                    of fifth code bits (bit 2g + h of byte l is the fifth
 *                    bit, worth 16, of element 64g + 32h + l), then the 128
 *                    code bytes as in Q4_K; q in 0..31, w as for Q4_K.
 *   Q6_K (210 bytes per 256 weights, k % 2048 == 0 so that every row starts
 *                    on a 16-byte boundary): also dispatched without a printed
 *                    layout; taken as the GGUF superblock: 128 bytes of low
 *                    code nibbles, 64 bytes of high code bit pairs, 16 int8
 *                    scales (one per 16 weights), fp16 d in bytes 208-209.
 *                    Element 128h + 32c + l (c < 4, l < 32) has nibble c / 2
 *                    of byte 64h + 32(c % 2) + l and bits 2c, 2c + 1 of byte
 *                    128 + 32h + l as its 6-bit code q; w = d * sc * (q - 32).
 *   IQ4_XS (136 bytes per 256 weights, k % 512 == 0 so that every row starts
 *                    on a 16-byte boundary): dispatched by the pages
 *                    (Iq4XsDequantKernel, iq4_xs_dequant_to_f32) without its
 *                    layout or code book; taken as the GGUF superblock: fp16
 *                    d, a little-endian word of high scale bits, 4 bytes of
 *                    low scale nibbles, then 128 code bytes, 16 per 32
 *                    weights. Sub-block j (weights 32j ..) has the 6-bit
 *                    scale ls_j (low nibble: nibble j % 2 of byte 4 + j / 2;
 *                    top two bits: bits 2j, 2j + 1 of the word); byte
 *                    8 + 16j + l holds the code c of weight 32j + l (low
 *                    nibble) and of 32j + 16 + l (high nibble);
 *                    w = d * (ls_j - 32) * book[c], book the IQ4_NL code
 *                    book {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13,
 *                    25, 38, 53, 69, 89, 113}.
 * Row i of W is the k/32 consecutive blocks starting at byte i*(k/32)*bytes
 * (the superblock formats: k/256 superblocks).
 *
 * Memory and streams. Every pointer argument named W, Wu, X, residual, Y or
 * out is a DEVICE pointer on the current CUDA device, owned by the caller and
 * never freed or retained by the library. Every call is asynchronous on the
 * given stream (NULL = the legacy default stream): a return of APR_OK means the
 * work was enqueued. X, residual, Y and out are float32, row major, densely
 * packed (row stride = number of columns). Device pointers must be 16-byte
 * aligned. Weights are never dequantized to memory: blocks are decoded in
 * registers.
 *
 * Scratch. The library owns device scratch per (device, stream): the fp16
 * copy of X for the GEMM path (T*k*2 bytes), and, for the tensor-core GEMV
 * (T = 3 or 4, or T = 2 where the integer-dot GEMV does not run), ticket counters
 * and partial sums (64 KiB plus 2 KiB per 128 weight rows and per SM, at
 * most), for the exact leg its split copies of X, exponents and, when k is
 * split over CTAs, up to four partial outputs of T*n floats, and, for
 * apr_prefill_attention, the fp16 copies of the K and V cache rows it reads. Calls on one stream share their stream's buffers,
 * which are ordered by the stream. A buffer grows on demand with cudaMalloc (also during a
 * stream capture: the calling thread's capture mode is relaxed for that
 * call) and is never freed while the process runs; a grown buffer replaces
 * the old one for later calls and the old one is kept. A graph captured from
 * a stream uses that stream's buffers: replay it ordered with the other
 * library calls on that stream, not concurrently with them.
 *
 * Errors. Arguments are checked on the host before anything is enqueued:
 *   APR_E_INVAL   null pointer with nonzero sizes, n < 0, T < 0, k <= 0,
 *                 k % 32 != 0 (k % 256 != 0 for Q4_K, Q5_K; k % 2048 != 0
 *                 for Q6_K; k % 512 != 0 for IQ4_XS), a size beyond the
 *                 documented limits, or an
 *                 unknown leg / path
 *   APR_E_QTYPE   qtype is not APR_Q4_0, APR_Q8_0, APR_F16, APR_Q4_K, APR_Q5_K,
 *                 APR_Q6_K or APR_IQ4_XS
 *   APR_E_ALIGN   a pointer is not 16-byte aligned
 *   APR_E_ALIAS   Y overlaps X, W or Wu, or overlaps residual without being
 *                 exactly the same buffer (Y == residual is allowed: it gives
 *                 Y += X.W^T, the accumulate form of the pages' batch kernels)
 *   APR_E_DEVICE  no CUDA device, or the device is not compute capability 10.3
 *   APR_E_NOMEM   the scratch could not be allocated
 *   APR_E_LAUNCH  a CUDA launch or API call failed (see apr_last_error)
 *   APR_E_TIMEOUT reported by apr_stream_status: a bounded device-side wait
 *                 expired and the kernel gave up (results are garbage)
 * T == 0 or n == 0 is a successful no-op (oxibonsai-kernels
 * try_cuda_prefill_q_std returns at once for an empty batch). On any error Y
 * is unspecified and must be discarded.
 *
 * Stream order: every call is ordered after the work before it on its stream,
 * with one relaxation. The library's kernels start while the preceding kernel
 * of the library on the same stream finishes, and read the weights (W, Wg,
 * Wu) before it has finished; X, residual and Y are touched only after it has.
 * So a call's weights must not be an output (Y, or the X16 of
 * apr_convert_f32_to_f16) of the immediately preceding call of this library
 * on that stream. Kernels of other code on the stream are always complete
 * first.
 *
 * Limits: n, T <= 2^24, k <= 2^20, n*k/32 blocks <= 2^31.
 */
#ifndef APR_QGEMM_H
#define APR_QGEMM_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* apr_stream_t;

/* GGUF tensor type ids. */
enum { APR_F16 = 1, APR_Q4_0 = 2, APR_Q8_0 = 8, APR_Q4_K = 12, APR_Q5_K = 13, APR_Q6_K = 14, APR_IQ4_XS = 23 };

/*
 * Arithmetic legs (aprender-serve gdn_prefill_ops.rs, module doc, group 1):
 *   APR_LEG_F16        X and the decoded weights are rounded to fp16, products
 *                      accumulate in fp32 on the tensor cores, Y is fp32
 *                      (the pages' f16 leg, their default).
 *   APR_LEG_EXACT_F32  fp32 inputs, fp32 accumulation, no reduced-precision
 *                      rounding of X or W (the pages' f32 leg, kept for
 *                      projections that feed a recurrence).
 */
enum { APR_LEG_F16 = 0, APR_LEG_EXACT_F32 = 1 };

/* Kernel choice: AUTO applies the T rule below; the others force a path. */
enum { APR_PATH_AUTO = 0, APR_PATH_GEMV = 1, APR_PATH_GEMM = 2 };

enum {
  APR_OK = 0,
  APR_E_INVAL = -1,
  APR_E_QTYPE = -2,
  APR_E_ALIGN = -3,
  APR_E_ALIAS = -4,
  APR_E_DEVICE = -5,
  APR_E_LAUNCH = -6,
  APR_E_TIMEOUT = -7,
  APR_E_NOMEM = -8
};

/*
 * The T rule, fixed and measured on GB300 (Q4_0 and Q8_0, 4096 x 4096 and
 * 12288 x 4096 weights, each call with its fp32 X): with APR_PATH_AUTO,
 * 1 <= T <= APR_AUTO_GEMV_MAX_T runs the small-T GEMV (exact fp32 arithmetic
 * whatever the leg), larger T runs the GEMM of the call's leg. The fp16-leg
 * GEMM call costs the same at every T up to its 256-token tile (15.6 us at
 * 4096 x 4096, 23.7 us at 12288 x 4096, Q4_0); the GEMV costs 5.6, 10.0, 14.6
 * and 15.0 us at T = 1 to 4 and 22.0 us at T = 5 (4096 x 4096), 11.3 to 26.3 us
 * at T = 1 to 4 (12288 x 4096), because its FFMA work grows with T.
 * APR_GEMV_MAX_T (apr_gemv_max_T()) is the largest T the GEMV path itself
 * takes (APR_PATH_GEMV, apr_qgemv).
 */
#define APR_AUTO_GEMV_MAX_T 4
#define APR_GEMV_MAX_T 16
int apr_gemv_max_T(void);

/*
 * Y = X . dequant(W)^T (+ residual), fp16 leg, T rule.
 *   qtype     APR_Q4_0, APR_Q8_0, APR_F16, APR_Q4_K, APR_Q5_K, APR_Q6_K or
 *             APR_IQ4_XS
 *   W         [n rows][k/32 blocks] GGUF blocks
 *   X         [T][k] f32;  Y [T][n] f32, overwritten
 *   residual  [T][n] f32 or NULL; may be Y itself (accumulate)
 * The residual variant is the residual-add GEMM of oxibonsai-kernels
 * (gemm_q4_0_residual / gemm_q8_0_residual; the down and output projections
 * are followed by a residual add in encode_q_std_ffn_phase step 3 and
 * prefill_ffn_rows).
 */
int apr_qgemm(int qtype, const void* W, int n, int k, const float* X, int T,
              float* Y, const float* residual, apr_stream_t stream);

/*
 * Fused gate/up SwiGLU: Y = silu(X . Wg^T) * (X . Wu^T), silu(g) = g/(1+e^-g).
 * Wg and Wu are two [n][k] weights of the same qtype (the pages keep them as
 * one buffer, gate rows then up rows: oxibonsai-kernels try_cuda_prefill_q_std
 * and launch_fused_gate_up_swiglu_q4_0; here they are two pointers, which
 * covers that buffer with Wu = Wg + n*k/32*bytes). No residual. fp16 leg,
 * T rule.
 */
int apr_qgemm_gate_up_swiglu(int qtype, const void* Wg, const void* Wu, int n, int k,
                             const float* X, int T, float* Y, apr_stream_t stream);

/*
 * Small-T GEMV, 1 <= T <= APR_GEMV_MAX_T (T == 0 is a no-op), exact fp32
 * arithmetic, optional residual (gemv_q4_0_pf / gemv_q8_0_pf of
 * oxibonsai-kernels, used for the last-token lm_head in
 * try_cuda_prefill_q_std). Weight rows stream by bulk copies into T fp32
 * accumulators for T <= 4 with Q4_0 / Q8_0 (integer dot products of X in
 * fixed point against the codes for T = 1, 2, also for the K-quants and
 * IQ4_XS; tensor cores for T = 3, 4) and T <= 8 with F16, K-quant and IQ4_XS
 * weights (CUDA cores); for larger T up to 16,
 * and for smaller T where no streaming kernel takes the shape (the X table of
 * a long row does not fit shared memory), the exact leg's tensor-core GEMM
 * runs instead when k % 256 == 0 (22-24 us at 4096 x 4096 for T <= 16, with k
 * split over CTAs when the grid is small; 53-57 us at 12288 x 4096; against
 * 30-80 us for the CUDA-core kernels at T = 8). T > APR_GEMV_MAX_T gives
 * APR_E_INVAL. The weights are read early (see stream order above).
 */
int apr_qgemv(int qtype, const void* W, int n, int k, const float* X, int T,
              float* Y, const float* residual, apr_stream_t stream);

/*
 * Full form. Wu != NULL selects the gate/up SwiGLU product (W is the gate;
 * residual must be NULL). leg and path as above; APR_PATH_GEMV needs
 * T <= APR_GEMV_MAX_T. The exact leg on the GEMM path runs on the tensor
 * cores when k % 256 == 0: the weight (times a power of two per row) and X
 * (per token) split into two fp16 pieces each, three products per term
 * (W1.X1 + W1.X2 + W2.X1), fp32 accumulation restarted every 256 k and the
 * partial sums added in fp32 (relative error about 1e-6 at k = 4096 and
 * 12288); when its 128 x 128 tiles leave most SMs idle, k is split over up to
 * four CTAs whose partial outputs (scratch) a second kernel adds in a fixed
 * order; gate/up takes two such products and an elementwise SwiGLU. Other k
 * run fp32 FFMA.
 * ldy: strided output. Row t of Y starts at Y + t * ldy (and row t of
 * residual at residual + t * ldy), so Y can be a slice of a wider buffer, such
 * as the rows of a KV cache (aprender-serve writes attn_v straight into the
 * cache this way: forward_qwen35_cuda_prefill.rs). 0 means n (dense); else
 * n <= ldy <= 2^28 (APR_E_INVAL otherwise). Only the n floats of each row are
 * written. With residual == Y it accumulates into the strided rows. The
 * tensor-core path writes Y from registers (each warp 32 consecutive
 * floats of a row). X stays dense [T][k].
 */
typedef struct apr_qgemm_args {
  int qtype;
  int leg;
  int path;
  const void* W;
  const void* Wu;
  int n;
  int k;
  int T;
  const float* X;
  const float* residual;
  float* Y;
  apr_stream_t stream;
  int ldy;  /* floats from one row of Y (and of residual) to the next; 0: n */
} apr_qgemm_args;
int apr_qgemm_ex(const apr_qgemm_args* args);

/*
 * The fp16 leg in two calls, for callers that keep their own fp16 copy of the
 * activations (the pages' f16 leg also rounds the activation rows to fp16 in a
 * pass of its own, convert_f32_to_f16, before its fp16 GEMM:
 * aprender-serve gdn_prefill_ops.rs qwen35_project_rows_f16).
 *
 * apr_convert_f32_to_f16: X16[i] = fp16(X[i]) (round to nearest even) for
 *   0 <= i < count; X (f32) and X16 (fp16, 2 bytes each) are device buffers,
 *   16-byte aligned, not overlapping. count == 0 is a no-op.
 * apr_qgemm_f16_in: as apr_qgemm (Wu == NULL) or apr_qgemm_gate_up_swiglu
 *   (Wu != NULL, residual must be NULL) on the tensor cores, with X16 [T][k]
 *   fp16 already converted; needs k % 256 == 0 (APR_E_INVAL otherwise), takes
 *   no scratch and ignores the T rule (always the GEMM).
 */
int apr_convert_f32_to_f16(const float* X, long long count, void* X16, apr_stream_t stream);
int apr_qgemm_f16_in(int qtype, const void* W, const void* Wu, int n, int k, const void* X16, int T,
                     float* Y, const float* residual, apr_stream_t stream);

/*
 * apr_qgemm_noalloc: Y = X . dequant(W)^T (+ residual) on the tensor cores (the
 * fp16 leg's GEMM path, whatever T is), allocating no device memory. The pages
 * have no counterpart: it exists for callers that cannot allocate device
 * memory once they run (a serving process that has reserved nearly all of HBM
 * for weights and its KV-cache arena and treats a later allocation as a fault,
 * or a runtime that allows allocation only at start-up). apr_qgemm keeps its
 * T*k*2-byte fp16 copy of X in scratch it grows on demand; this variant uses
 * a fixed scratch array of APR_NOALLOC_MAX_TK fp16 values (16 MiB) that exists
 * on every GPU that loads the library, from module load until the process
 * exits.
 *   - T*k > APR_NOALLOC_MAX_TK or k % 256 != 0: APR_E_INVAL with a message.
 *   - The first call on each device looks up the scratch's device address (and
 *     checks the device); make that first call before any stream capture. A
 *     lookup that fails returns APR_E_DEVICE and is tried again by the next
 *     call; once it has succeeded it is kept for the process.
 *   - Every call shares the one array, which keeps the last call's contents
 *     (each call overwrites the T*k values it reads, so nothing needs
 *     clearing). Calls whose work overlaps on the GPU (on different streams,
 *     or from different threads) race on it: order them on one stream.
 * Other arguments, errors and the status word as for apr_qgemm.
 */
#define APR_NOALLOC_MAX_TK (8 * 1024 * 1024)
int apr_qgemm_noalloc(int qtype, const void* W, int n, int k, const float* X, int T,
                      float* Y, const float* residual, apr_stream_t stream);

/*
 * Normed projection: apr_qgemm_ex with X replaced by its row RMSNorm,
 *   h = X / sqrt(mean(X^2, per row) + eps) * norm_weight,
 * so Y = h . W^T (+ residual), or silu(h . Wg^T) * (h . Wu^T) with Wu. The
 * pages' prefill layer runs the norm and then the projection as two steps
 * (aprender-serve forward_qwen35_cuda_prefill.rs: batched_rmsnorm_into with
 * attn_norm, then attn_qkv; post_attention_norm, then gate and up). Here, on
 * the fp16 leg's tensor-core path, the norm writes the fp16 rows the GEMM
 * reads, in one pass. args as for apr_qgemm_ex (ldy included; X is the
 * un-normed input, read only); norm_weight [k] fp32, 16-byte aligned; eps >= 0
 * and finite. Rows are processed in chunks of APR_FFN_CHUNK_ROWS; scratch per
 * stream (the normed rows of a chunk). Errors as for apr_qgemm_ex, and
 * APR_E_ALIAS if Y overlaps norm_weight.
 */
int apr_qgemm_rmsnorm(const apr_qgemm_args* args, const float* norm_weight, float eps);

/*
 * FFN sublayer of a prefill layer over T rows of the residual stream, in place:
 *   h = RMSNorm(X) = X / sqrt(mean(X^2, per row) + eps) * norm_weight
 *   X = X + (silu(h . Wg^T) * (h . Wu^T)) . Wd^T
 * The pages' batched FFN phase (oxibonsai-kernels 0.1.4
 * cuda_q_std_prefill.rs encode_q_std_ffn_phase: batched RMSNorm, fused
 * gate/up SwiGLU GEMM, down GEMM with the residual added; aprender-serve
 * forward_qwen35_cuda_prefill.rs prefill_ffn_rows). The norm is not printed
 * there; this is the usual RMSNorm of a row, eps inside the square root.
 *   qtype      any qtype above, the same for all three
 *   leg        APR_LEG_F16 or APR_LEG_EXACT_F32, as for apr_qgemm_ex; the f16
 *              leg writes the normed rows straight as fp16 (norm and
 *              conversion in one pass) for the tensor-core GEMMs
 *   Wg, Wu     [inter][hidden] weights (rows of hidden / 32 blocks)
 *   Wd         [hidden][inter] weight
 *   hidden, inter  multiples of 32 (hidden also of 4); the tensor-core path
 *              needs both multiples of 256, else the FFMA kernels run
 *   T          rows (0: no-op); processed in chunks of up to
 *              APR_FFN_CHUNK_ROWS rows, each chunk one norm and three
 *              projections that follow the T rule of apr_qgemm_ex
 *   norm_weight  [hidden] fp32; eps >= 0 and finite
 *   X          [T][hidden] fp32, dense, read and updated in place
 * Scratch per stream as for apr_qgemm (the normed rows and the activations of
 * a chunk, at most APR_FFN_CHUNK_ROWS * (4 hidden + 6 inter) bytes). Errors:
 * as for apr_qgemm_ex, and APR_E_ALIAS if X overlaps a weight or norm_weight.
 */
#define APR_FFN_CHUNK_ROWS 2048
typedef struct apr_ffn_args {
  int qtype;
  int leg;
  const void* Wg;
  const void* Wu;
  const void* Wd;
  int hidden;
  int inter;
  int T;
  const float* norm_weight;
  float eps;
  float* X;
  apr_stream_t stream;
} apr_ffn_args;
int apr_ffn_sublayer(const apr_ffn_args* args);

/*
 * Causal prefill attention over a KV cache, the step between the attention
 * sublayer's qkv projection and its output projection (aprender-serve 0.70.2
 * gdn_prefill_ops.rs: qwen35_prefill_attention / qwen35_attention_pass define
 * the layouts, the mask and the head grouping; qwen35_flash_prefill_attention
 * the fused form taken here, fp16 tensor-core inputs with fp32 accumulation
 * and an fp32 online softmax, no score matrix in memory). For query row t
 * (position pos0 + t) and query head h,
 *   out[t][h] = sum_{j <= pos0 + t} softmax_j(Q[t][h] . K[j][g] / sqrt(d)) V[j][g]
 * with g = h / (num_heads / num_kv_heads) and d = head_dim.
 *   Q          [T][num_heads * head_dim] fp32 query rows (normed and rotated
 *              by the caller), dense
 *   K_cache, V_cache  [>= pos0 + T][num_kv_heads * head_dim] fp32 rows, with
 *              this chunk's rows already written; rows at or past pos0 + T are
 *              never read
 *   out        [T][num_heads * head_dim] fp32, overwritten
 *   T          query rows (0: no-op); pos0 >= 0 their first position
 *   num_heads  a multiple of num_kv_heads (grouped-query attention);
 *              num_heads <= 65536, num_kv_heads <= 16383
 *   head_dim   256 (the only size the fused form takes)
 * q, k and v enter the products rounded to fp16; the result is within fp16
 * input rounding of the exact attention (the tests bound it). When its
 * (128 query rows, head) tiles leave SMs idle and the longest sees many key
 * tiles, the call cuts each tile's keys into parts whose softmax sums a
 * second kernel combines; a row's result then depends on the call's shape at
 * rounding level (within the same bound). All pointers
 * 16-byte aligned, caller owned. Scratch per stream as for apr_qgemm: the
 * fp16 copies of the cache rows 0 .. pos0 + T - 1 that the call makes, K as
 * it is and V transposed (4 * (pos0 + T) * num_kv_heads * 256 bytes, plus
 * padding), and the parts' sums (132 KB per SM). Errors: APR_E_INVAL for negative sizes, num_heads not a multiple
 * of num_kv_heads, head_dim != 256, sizes past 2^30 positions, or a null
 * pointer with T > 0; APR_E_ALIGN; APR_E_ALIAS if out overlaps Q or a cache;
 * APR_E_NOMEM; APR_E_DEVICE; APR_E_LAUNCH. Asynchronous on the stream; apr_stream_status reports a
 * bounded wait that gave up (out is then unspecified).
 */
int apr_prefill_attention(const float* Q, const float* K_cache, const float* V_cache, float* out, int T, int pos0,
                          int num_heads, int num_kv_heads, int head_dim, apr_stream_t stream);

/*
 * One prefill layer over T rows of the residual stream, chunk by chunk (the
 * pages' chunked prefill: oxibonsai-kernels 0.1.4 cuda_q_std_prefill.rs
 * encode_q_std_prefill_layer runs batched RMSNorm, the qkv projection, the
 * causal attention over the KV cache, the attention output projection with the
 * residual added and then the FFN phase for every chunk; aprender-serve 0.70.2
 * forward_qwen35_cuda_prefill.rs prefill_chunk, chunks of 512 rows by default,
 * writes the chunk's k and v rows into the cache before the attention). For
 * the chunk's rows of X at positions p = pos0 + t:
 *   h = RMSNorm(X) * attn_norm
 *   q = h . Wq^T;  K_cache[p] = h . Wk^T;  V_cache[p] = h . Wv^T
 *   X += attention(q, K_cache, V_cache) . Wo^T      (as apr_prefill_attention)
 *   X += down(silu(h2 . Wg^T) * (h2 . Wu^T)),  h2 = RMSNorm(X) * ffn_norm
 * RoPE and the per-head q/k norm, which the pages apply between the qkv
 * projection and the attention, are not part of this call (a caller that needs
 * them runs the steps one by one with apr_qgemm_rmsnorm, apr_qgemm_ex with
 * ldy, apr_prefill_attention, apr_qgemm and apr_ffn_sublayer).
 *   qtype, leg  as for apr_qgemm_ex, for every projection (the attention takes
 *               fp16 inputs on both legs)
 *   Wqkv     [(num_heads + 2 num_kv_heads) * 256][hidden]: the q rows, then the
 *            k rows, then the v rows (the pages' fused qkv weight)
 *   Wo       [hidden][num_heads * 256];  Wg, Wu [inter][hidden];  Wd [hidden][inter]
 *   hidden, inter  multiples of the format's unit (32; 256 for Q4_K, Q5_K;
 *            2048 for Q6_K; 512 for IQ4_XS), and so must num_heads * 256 be
 *            (Wo's columns)
 *   num_heads, num_kv_heads, head_dim  as for apr_prefill_attention (256)
 *   T, pos0  rows of X and the position of the first; T == 0 is a no-op
 *   attn_norm, ffn_norm  [hidden] fp32;  eps >= 0 and finite
 *   X        [T][hidden] fp32, dense, updated in place
 *   K_cache, V_cache  [>= pos0 + T][num_kv_heads * 256] fp32; rows pos0 ..
 *            pos0 + T - 1 are written, rows before are read, rows after untouched
 *   chunk    rows per chunk (0: 512)
 * All pointers device, 16-byte aligned, caller owned; X and the caches must not
 * overlap each other, a weight or a norm weight (APR_E_ALIAS). Scratch per
 * stream as for apr_qgemm (the chunk's normed rows, q and attention output,
 * and what the steps take). Errors as for apr_qgemm_ex and
 * apr_prefill_attention. Asynchronous on the stream.
 */
typedef struct apr_layer_args {
  int qtype;
  int leg;
  const void* Wqkv;
  const void* Wo;
  const void* Wg;
  const void* Wu;
  const void* Wd;
  int hidden;
  int inter;
  int num_heads;
  int num_kv_heads;
  int head_dim;
  int T;
  int pos0;
  const float* attn_norm;
  const float* ffn_norm;
  float eps;
  float* X;
  float* K_cache;
  float* V_cache;
  int chunk;
  apr_stream_t stream;
} apr_layer_args;
int apr_prefill_layer(const apr_layer_args* args);

/*
 * Standalone dequant: out[n][k] f32 = f32(d) * f32(q'), bit exact (the product
 * of an fp16 scale and a code of at most 8 bits is exact in fp32); for F16
 * out = f32(w), also exact; for Q4_K and Q5_K the exact d * sc * q - dmin * m
 * rounded once to f32; for Q6_K d * sc * (q - 32) and for IQ4_XS
 * d * (ls - 32) * book[c], both exact. The device dequant of aprender-serve
 * gdn_prefill_ops.rs qwen35_dequant_f32 (Q8_0, F16 and the other formats it
 * dispatches), here for every qtype above and meant for tests: the
 * projections never write decoded weights to memory. An F16 W needs only
 * 2-byte alignment here (APR_E_ALIGN otherwise).
 */
int apr_dequant(int qtype, const void* W, int n, int k, float* out, apr_stream_t stream);

/*
 * Synchronizes the stream, then reports and clears the device status word:
 * APR_OK, APR_E_TIMEOUT if a kernel's bounded wait expired since the last
 * call, or APR_E_LAUNCH if the stream reported a CUDA error.
 */
int apr_stream_status(apr_stream_t stream);

/*
 * Measurement reference (the pages have no counterpart): streams `bytes`
 * bytes from the device buffer src into shared memory exactly as the T = 1
 * GEMV streams its weight (one CTA per SM, a contiguous share each, bulk
 * copies of 16 KB into a ring of 5 stages, programmatic dependent launch) and
 * computes nothing. Timing it beside apr_qgemv on the same number of bytes
 * separates the GEMV's own cost from the cost of moving its weight. bytes a
 * multiple of 16 (0: no-op), src 16-byte aligned, only read. Errors:
 * APR_E_INVAL, APR_E_ALIGN, APR_E_DEVICE, APR_E_LAUNCH.
 */
int apr_read_stream(const void* src, long long bytes, apr_stream_t stream);

/*
 * Test of the failure detection (the pages have no counterpart): enqueues one
 * kernel that waits on an mbarrier nothing arrives on, through the same
 * bounded wait every kernel of the library uses, with a limit of limit_us
 * microseconds (1 .. 1000000; APR_E_INVAL otherwise) instead of the library's
 * 2 s. The wait runs out, the kernel records the timeout in the device status
 * word and returns: no trap, no fault, the context stays usable. After it,
 * apr_stream_status on the stream returns APR_E_TIMEOUT (and clears the
 * word), and the library's calls on that stream work as before. Errors:
 * APR_E_INVAL, APR_E_DEVICE, APR_E_LAUNCH.
 */
int apr_test_bounded_wait(unsigned limit_us, apr_stream_t stream);

/* Message of the last failed call on this thread ("" if none). */
const char* apr_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* APR_QGEMM_H */
