"""Plain CPU oracle for the Q4_0 / Q8_0 / F16 / Q4_K / Q5_K / Q6_K / IQ4_XS prefill projections (float64).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
this module. The product path (the CUDA library and its binding) never does,
and this module imports nothing from it.

What is computed, and where the pages define it:

* Block formats (the GGUF blocks, which the pages' kernels read in their
  on-disk array-of-blocks order: oxibonsai-kernels 0.1.4
  src/gpu_backend/cuda_q_std_prefill.rs, module doc, section "Weight layout"):
  Q4_0 = fp16 ``d`` (little endian, bytes 0-1) + 16 bytes, byte ``j`` holding
  element ``j`` in its low nibble and ``j+16`` in its high nibble,
  ``w = d * (q - 8)``; the same page's test ``make_q4_0_zeros`` fixes the block
  size (18 bytes), the position of ``d`` and the fp16 encoding of 1.0
  (``0x00, 0x3C``). Q8_0 = fp16 ``d`` + 32 int8, ``w = d * q`` (32 elements per
  block, the ``k.div_ceil(32)`` dequant grid of aprender-serve 0.70.2
  src/cuda/executor/gdn_prefill_ops.rs, ``qwen35_dequant_f32``). F16 = each
  element its own IEEE binary16 value, two little-endian bytes, row after row
  (the F16 arm of that dispatch, with the same ``(n, k.div_ceil(32))`` grid,
  and its test ``f16_weight_dequantizes_on_the_device``, which writes the
  weight as ``f16::from_f32(v).to_le_bytes()`` per element and expects the
  values back unchanged). Here a "block" of F16 is 32 consecutive elements
  (64 bytes), so that every format is addressed the same way; ``k`` is a
  multiple of 32 for every format.
* Q4_K, a format the pages dispatch (``qwen35_dequant_f32``, grid
  ``(n, k.div_ceil(256))``) without printing its layout; read as the GGUF
  Q4_K superblock of 256 elements in 144 bytes: fp16 ``d`` (bytes 0-1), fp16
  ``dmin`` (2-3), 12 bytes of packed 6-bit sub-block scales and mins
  (``q4_k_scales_mins``), then 128 bytes of 4-bit codes: byte ``32 g + l``
  holds element ``64 g + l`` in its low nibble and ``64 g + 32 + l`` in its
  high nibble; element ``e`` of sub-block ``j = e / 32`` is
  ``w = d sc_j q - dmin m_j``. Q5_K (176 bytes) likewise, with 32 bytes of
  fifth code bits between the scales and the codes (bit ``2 g`` of byte ``l``
  for element ``64 g + l``, bit ``2 g + 1`` for ``64 g + 32 + l``, each worth
  16), the codes at bytes 48-175.
* Q6_K, also dispatched without a printed layout; read as the GGUF Q6_K
  superblock of 256 elements in 210 bytes: 128 bytes of low code nibbles, 64
  bytes of high code bit pairs, 16 int8 sub-block scales (one per 16
  elements), then fp16 ``d`` (bytes 208-209). Element ``e = 128 h + 32 c + l``
  (half ``h``, quarter ``c``, lane ``l`` < 32) takes nibble ``c / 2`` of low
  byte ``64 h + 32 (c % 2) + l`` and bits ``2 c .. 2 c + 1`` of high byte
  ``32 h + l`` as its six-bit code ``q``; ``w = d sc_{e/16} (q - 32)``.
* IQ4_XS, dispatched by the same page (``Iq4XsDequantKernel``, kernel
  ``iq4_xs_dequant_to_f32``, grid ``(n, k.div_ceil(256))``) without its
  layout or its code table; read as the GGUF IQ4_XS superblock of 256
  elements in 136 bytes: fp16 ``d`` (bytes 0-1), a little-endian 16-bit word
  of high scale bits (2-3), 4 bytes of low scale nibbles (4-7), then 128 bytes
  of 4-bit codes, 16 bytes a 32-element sub-block. Sub-block ``j`` has the
  six-bit scale ``ls_j`` (low nibble: nibble ``j % 2`` of byte ``4 + j / 2``;
  top two bits: bits ``2 j, 2 j + 1`` of the word) and byte ``8 + 16 j + l``
  holds element ``32 j + l`` in its low nibble and ``32 j + 16 + l`` in its
  high nibble (Q4_0's order). A code ``c`` does not stand for ``c - 8`` but
  for entry ``c`` of the non-linear 16-value table ``IQ4_NL_VALUES`` (GGUF's
  IQ4_NL code book); ``w = d (ls_j - 32) table[c]``. PARITY UNPINNED for the
  table's values: nothing on the pages fixes them, so the pins check the
  layout (with a linear table the superblock equals eight Q4_0 blocks) and
  take the values as given.
* Projection ``Y[T][n] = X[T][k] . W[n][k]^T`` (aprender-serve 0.70.2
  src/cuda/executor/gdn_prefill_ops.rs, doc of ``qwen35_project_rows``),
  optionally ``+ R[T][n]`` (the residual add that follows the down / output
  projections: oxibonsai-kernels 0.1.4 ``encode_q_std_ffn_phase`` step 3 and
  aprender-serve src/gguf/cuda/forward_qwen35_cuda_prefill.rs
  ``prefill_ffn_rows``).
* Fused gate/up SwiGLU ``silu(X . Wg^T) * (X . Wu^T)`` with
  ``silu(g) = g / (1 + exp(-g))`` (oxibonsai-kernels ``encode_q_std_ffn_phase``
  step 2; the unfused twin gate GEMM, up GEMM, ``fused_swiglu_into`` in
  ``prefill_ffn_rows``).

* The FFN sublayer of a prefill layer over a chunk of rows (oxibonsai-kernels
  0.1.4, doc of ``encode_q_std_ffn_phase``: batched RMSNorm of the input rows,
  the fused gate/up SwiGLU GEMM, the down GEMM whose result is added back into
  the input rows; aprender-serve src/gguf/cuda/forward_qwen35_cuda_prefill.rs,
  ``prefill_ffn_rows``: the same steps with ``batched_rmsnorm_into`` over
  ``hidden_dim`` with ``d.eps``). The pages call the norm without printing it;
  this module reads it as the usual RMSNorm of a row,
  ``y = x / sqrt(mean(x^2) + eps) * w``, ``w`` the norm weight per column.

* Causal prefill attention over a KV cache (aprender-serve 0.70.2
  src/cuda/executor/gdn_prefill_ops.rs, docs of ``qwen35_prefill_attention``
  and ``qwen35_attention_pass``, and ``qwen35_flash_prefill_attention`` for the
  fused form): query row ``t`` of a chunk sits at position ``pos0 + t`` and
  attends to the cache rows ``0 .. pos0 + t``; scores are ``q . k / sqrt(d)``,
  softmax over those keys, output ``sum_j p_j v_j``; query head ``h`` reads KV
  head ``h / (num_heads / num_kv_heads)``. ``q`` is ``[rows][num_heads * d]``,
  the caches ``[>= pos0 + rows][num_kv_heads * d]``, the output like ``q``.

* One prefill layer over a chunk of rows (oxibonsai-kernels 0.1.4
  ``encode_q_std_prefill_layer``: batched RMSNorm, the qkv projection, the
  causal attention over the KV cache, the attention output projection with the
  residual added, then the FFN phase; aprender-serve
  src/gguf/cuda/forward_qwen35_cuda_prefill.rs, ``prefill_chunk``: the chunk's
  k and v rows are written into the cache at positions ``pos0 ..`` before the
  attention reads it). The fused qkv weight holds the q rows, then the k rows,
  then the v rows. RoPE and the per-head q/k norm, which the pages apply
  between the qkv projection and the attention, are model plumbing and are
  not part of this layer.

Every product is accumulated in float64 and the result is rounded to float32
once. The f16-input mode rounds ``X`` and the dequantized ``W`` to fp16 first
(the fp16 leg of ``qwen35_project_rows_f16``: fp16 in, fp32 accumulate), then
accumulates exactly the same way.
"""

from __future__ import annotations

import numpy as np

F16 = 1
Q4_0 = 2
Q8_0 = 8
Q4_K = 12
Q5_K = 13
Q6_K = 14
IQ4_XS = 23
_QK = 32
_QK_K = 256
_BLOCK_BYTES = {F16: 64, Q4_0: 18, Q8_0: 34}
_SUPER_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, IQ4_XS: 136}
# the code book of IQ4_XS (and IQ4_NL): code c stands for entry c
IQ4_NL_VALUES = (-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113)


# --------------------------------------------------------------------------
# fp16 decode, written from the IEEE 754 binary16 definition:
# 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
#   e == 0        : (-1)^s * 2^-14 * (f / 1024)          (zero / subnormal)
#   0 < e < 31    : (-1)^s * 2^(e-15) * (1 + f / 1024)   (normal)
#   e == 31       : (-1)^s * inf if f == 0, else NaN
# --------------------------------------------------------------------------
def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = (bits >> 15) & 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    sign = np.where(s == 1, -1.0, 1.0)
    frac = f.astype(np.float64) / 1024.0
    normal = sign * np.ldexp(1.0 + frac, (e - 15).astype(np.int64))
    sub = sign * np.ldexp(frac, -14)
    special = np.where(f == 0, sign * np.inf, np.nan)
    return np.where(e == 0, sub, np.where(e == 31, special, normal))


def _superblocks(qtype: int, W: np.ndarray, n: int, k: int) -> np.ndarray:
    if k % _QK_K:
        raise ValueError("k must be a multiple of 256 for a superblock format")
    sb = _SUPER_BYTES[qtype]
    raw = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
    if raw.size != n * (k // _QK_K) * sb:
        raise ValueError("weight byte count does not match n, k")
    return raw.reshape(n, k // _QK_K, sb)


def q4_k_scales_mins(scales: np.ndarray):
    """The eight 6-bit sub-block scales and mins of a Q4_K superblock from its
    12 packed bytes ``[..., 12]`` (reading: bytes 0-3 hold scales 0-3 in their
    low 6 bits, bytes 4-7 mins 0-3 likewise; bytes 8-11 hold scales 4-7 in
    their low nibble and mins 4-7 in their high nibble, whose top two bits sit
    in the top two bits of bytes 0-3 (scales) and 4-7 (mins))."""
    s = scales.astype(np.int64)
    sc = np.empty(s.shape[:-1] + (8,), np.int64)
    mn = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = s[..., j] & 63
        mn[..., j] = s[..., j + 4] & 63
        sc[..., j + 4] = (s[..., j + 8] & 0x0F) | ((s[..., j] >> 6) << 4)
        mn[..., j + 4] = (s[..., j + 8] >> 4) | ((s[..., j + 4] >> 6) << 4)
    return sc, mn


def _dequant_k(qtype: int, W: np.ndarray, n: int, k: int) -> np.ndarray:
    """Q4_K and Q5_K (the same header, scales and code bytes; Q5_K adds 32
    bytes of fifth bits after the scales: bit 2 g of byte l for element
    64 g + l, bit 2 g + 1 for element 64 g + 32 + l, worth 16)."""
    sb = _superblocks(qtype, W, n, k)
    d = fp16_bits_to_f64(sb[..., 0].astype(np.uint16) | (sb[..., 1].astype(np.uint16) << 8))
    dmin = fp16_bits_to_f64(sb[..., 2].astype(np.uint16) | (sb[..., 3].astype(np.uint16) << 8))
    sc, mn = q4_k_scales_mins(sb[..., 4:16])
    qoff = 16 if qtype == Q4_K else 48
    qs = sb[..., qoff:].reshape(n, k // _QK_K, 4, 32).astype(np.int64)  # group g: bytes 32 g .. 32 g + 31
    q = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)  # group g: 64 elements, low nibbles first
    if qtype == Q5_K:
        qh = sb[..., 16:48].astype(np.int64)[:, :, None, :]      # [.., 1, 32]
        g = np.arange(4).reshape(1, 1, 4, 1)
        hb = np.concatenate([(qh >> (2 * g)) & 1, (qh >> (2 * g + 1)) & 1], axis=-1)
        q = q + 16 * hb
    q = q.reshape(n, k // _QK_K, 8, 32).astype(np.float64)  # sub-block j = 2 g + (high nibble)
    w = d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None]
    return w.reshape(n, k)


def _dequant_q6_k(W: np.ndarray, n: int, k: int) -> np.ndarray:
    """Q6_K: six-bit codes from a low nibble and a high bit pair, a signed
    8-bit scale per 16 elements, ``w = d sc (q - 32)``."""
    sb = _superblocks(Q6_K, W, n, k)
    nsb = k // _QK_K
    ql = sb[..., 0:128].astype(np.int64).reshape(n, nsb, 2, 2, 32)    # [half][c % 2][l]
    qh = sb[..., 128:192].astype(np.int64).reshape(n, nsb, 2, 1, 32)  # [half][.][l]
    sc = sb[..., 192:208].view(np.int8).astype(np.int64)               # [16]
    d = fp16_bits_to_f64(sb[..., 208].astype(np.uint16) | (sb[..., 209].astype(np.uint16) << 8))
    low = np.concatenate([ql & 0x0F, ql >> 4], axis=3)                 # [half][c][l], c = 0 .. 3
    c = np.arange(4).reshape(1, 1, 1, 4, 1)
    high = (qh >> (2 * c)) & 3
    q = (low | (high << 4)).reshape(n, nsb, 16, 16).astype(np.float64)  # sub-block e / 16
    w = d[..., None, None] * sc[..., None].astype(np.float64) * (q - 32.0)
    return w.reshape(n, k)


def iq4_xs_scales(sb: np.ndarray) -> np.ndarray:
    """The eight signed sub-block scales ``ls_j - 32`` of IQ4_XS superblocks
    ``[..., 136]``: the low nibble of ``ls_j`` is nibble ``j % 2`` of byte
    ``4 + j / 2``, its top two bits are bits ``2 j, 2 j + 1`` of the
    little-endian word at bytes 2-3."""
    hi = sb[..., 2].astype(np.int64) | (sb[..., 3].astype(np.int64) << 8)
    ls = np.empty(sb.shape[:-1] + (8,), np.int64)
    for j in range(8):
        low = (sb[..., 4 + j // 2].astype(np.int64) >> (4 * (j % 2))) & 0x0F
        ls[..., j] = low | (((hi >> (2 * j)) & 3) << 4)
    return ls - 32


def _dequant_iq4_xs(W: np.ndarray, n: int, k: int, table=IQ4_NL_VALUES) -> np.ndarray:
    """IQ4_XS: ``w = d (ls_j - 32) table[c]`` for the code ``c`` of each
    element, the codes of sub-block ``j`` in bytes ``8 + 16 j ..`` (low
    nibbles the first 16 elements, high nibbles the next 16). ``table`` is a
    parameter only so that a test can substitute a linear one."""
    sb = _superblocks(IQ4_XS, W, n, k)
    nsb = k // _QK_K
    d = fp16_bits_to_f64(sb[..., 0].astype(np.uint16) | (sb[..., 1].astype(np.uint16) << 8))
    s = iq4_xs_scales(sb).astype(np.float64)                           # [n][nsb][8]
    qs = sb[..., 8:].astype(np.int64).reshape(n, nsb, 8, 16)
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)              # [n][nsb][8][32]
    vals = np.asarray(table, dtype=np.float64)[codes]
    w = d[..., None, None] * s[..., None] * vals
    return w.reshape(n, k)


def _row_bytes(qtype: int, k: int) -> int:
    """Bytes of one weight row of k elements."""
    if qtype in _SUPER_BYTES:
        return k // _QK_K * _SUPER_BYTES[qtype]
    return k // _QK * _BLOCK_BYTES[qtype]


def _blocks(qtype: int, W: np.ndarray, n: int, k: int) -> np.ndarray:
    if qtype not in _BLOCK_BYTES:
        raise ValueError(f"unsupported qtype {qtype}")
    if k % _QK:
        raise ValueError("k must be a multiple of 32")
    bb = _BLOCK_BYTES[qtype]
    raw = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
    if raw.size != n * (k // _QK) * bb:
        raise ValueError("weight byte count does not match n, k")
    return raw.reshape(n, k // _QK, bb)


def block_scales_and_codes(qtype: int, W: np.ndarray, n: int, k: int):
    """Split the blocks into fp16 scale bits ``[n][k/32]`` and signed codes ``q'``.

    ``q'`` is ``nibble - 8`` for Q4_0 and the int8 value for Q8_0, shape
    ``[n][k/32][32]`` (int64), element order as stored.
    """
    if qtype not in _BLOCK_BYTES or qtype == F16:
        raise ValueError("only Q4_0 and Q8_0 have one scale and codes per 32-element block")
    blk = _blocks(qtype, W, n, k)
    d_bits = blk[..., 0].astype(np.uint16) | (blk[..., 1].astype(np.uint16) << 8)
    payload = blk[..., 2:]
    if qtype == Q4_0:
        low = (payload & 0x0F).astype(np.int64)   # elements 0..15
        high = (payload >> 4).astype(np.int64)    # elements 16..31
        codes = np.concatenate([low, high], axis=-1) - 8
    else:
        codes = payload.view(np.int8).astype(np.int64)
    return d_bits, codes


def dequant_f64(qtype: int, W: np.ndarray, n: int, k: int) -> np.ndarray:
    """``Wf[i][j] = fp16(d_{i, j/32}) * q'_{i,j}`` in float64, shape ``[n][k]``;
    for F16 the binary16 value of element ``(i, j)``."""
    if qtype == Q6_K:
        return _dequant_q6_k(W, n, k)
    if qtype == IQ4_XS:
        return _dequant_iq4_xs(W, n, k)
    if qtype in _SUPER_BYTES:
        return _dequant_k(qtype, W, n, k)
    if qtype == F16:
        raw = _blocks(qtype, W, n, k).reshape(n, k, 2)
        bits = raw[..., 0].astype(np.uint16) | (raw[..., 1].astype(np.uint16) << 8)
        return fp16_bits_to_f64(bits)
    d_bits, codes = block_scales_and_codes(qtype, W, n, k)
    d = fp16_bits_to_f64(d_bits)
    return (d[..., None] * codes.astype(np.float64)).reshape(n, k)


def dequant_f32(qtype: int, W: np.ndarray, n: int, k: int) -> np.ndarray:
    """The standalone dequant export: ``f32(d) * f32(q')`` (F16: ``f32(w)``).

    ``d`` has at most 11 significant bits and ``|q'| <= 128`` at most 8, so the
    float64 product is exact and so is its conversion to float32 (the range of
    an fp16 scale times 128 is well inside float32's normal range, and fp16
    subnormal scales times small integers stay exact in float32). Every fp16
    value, subnormals included, is a float32 value. Q4_K and Q5_K: the exact
    float64 value ``d sc q - dmin m`` rounded once to float32. Q6_K: ``d sc
    (q - 32)`` has at most 11 + 7 + 6 significant bits, so it is exact in
    float32 too. IQ4_XS: ``d (ls - 32) table[c]`` has at most 11 + 5 + 7 bits
    (|ls - 32| <= 32, every table entry below 128 in magnitude): exact.
    """
    return dequant_f64(qtype, W, n, k).astype(np.float32)


def _as_f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def qgemm_f64(qtype: int, W, n: int, k: int, X, residual=None) -> np.ndarray:
    """``Y = X . Wf^T (+ R)`` in float64, shape ``[T][n]``."""
    Wf = dequant_f64(qtype, W, n, k)
    X64 = _as_f64(X).reshape(-1, k)
    Y = X64 @ Wf.T
    if residual is not None:
        Y = Y + _as_f64(residual).reshape(Y.shape)
    return Y


def qgemm(qtype: int, W, n: int, k: int, X, residual=None) -> np.ndarray:
    """``Y = X . Wf^T (+ R)``, accumulated in float64, rounded to float32 once."""
    return qgemm_f64(qtype, W, n, k, X, residual).astype(np.float32)


def silu_f64(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def gate_up_swiglu_f64(qtype: int, Wg, Wu, n: int, k: int, X) -> np.ndarray:
    g = qgemm_f64(qtype, Wg, n, k, X)
    u = qgemm_f64(qtype, Wu, n, k, X)
    return silu_f64(g) * u


def gate_up_swiglu(qtype: int, Wg, Wu, n: int, k: int, X) -> np.ndarray:
    """``silu(X . Wg^T) * (X . Wu^T)`` in float64, rounded to float32 once."""
    return gate_up_swiglu_f64(qtype, Wg, Wu, n, k, X).astype(np.float32)


# --------------------------------------------------------------------------
# fp16-input mode: the same products after rounding both operands to fp16
# (round to nearest even, numpy's float32 -> float16 conversion). Isolates
# the accumulation error of an fp16-input leg from its input rounding.
# --------------------------------------------------------------------------
def qgemm_f16_inputs_f64(qtype: int, W, n: int, k: int, X, residual=None) -> np.ndarray:
    W16 = dequant_f32(qtype, W, n, k).astype(np.float16).astype(np.float64)
    X16 = np.asarray(X, dtype=np.float32).reshape(-1, k).astype(np.float16).astype(np.float64)
    Y = X16 @ W16.T
    if residual is not None:
        Y = Y + _as_f64(residual).reshape(Y.shape)
    return Y


def gate_up_swiglu_f16_inputs_f64(qtype: int, Wg, Wu, n: int, k: int, X) -> np.ndarray:
    g = qgemm_f16_inputs_f64(qtype, Wg, n, k, X)
    u = qgemm_f16_inputs_f64(qtype, Wu, n, k, X)
    return silu_f64(g) * u


# --------------------------------------------------------------------------
# FFN sublayer (the norm, then SwiGLU, then down + residual)
# --------------------------------------------------------------------------
def rmsnorm_f64(X, weight, eps: float) -> np.ndarray:
    """Row-wise ``x / sqrt(mean(x^2) + eps) * w`` in float64, shape of ``X``."""
    X64 = _as_f64(X)
    w64 = _as_f64(weight).reshape(1, -1)
    ms = np.mean(X64 * X64, axis=-1, keepdims=True)
    return X64 / np.sqrt(ms + float(eps)) * w64


def ffn_sublayer_f64(qtype: int, X, weight, eps: float, Wg, Wu, Wd, hidden: int, inter: int) -> np.ndarray:
    """``X + down(silu(h . Wg^T) * (h . Wu^T))`` with ``h = rmsnorm(X)``:
    Wg, Wu are ``[inter][hidden]`` blocks, Wd ``[hidden][inter]``; float64."""
    X64 = _as_f64(X).reshape(-1, hidden)
    h = rmsnorm_f64(X64, weight, eps)  # kept in float64, as every intermediate
    g = h @ dequant_f64(qtype, Wg, inter, hidden).T
    u = h @ dequant_f64(qtype, Wu, inter, hidden).T
    act = silu_f64(g) * u
    return X64 + act @ dequant_f64(qtype, Wd, hidden, inter).T


def normed_qgemm_f64(qtype: int, W, n: int, k: int, X, weight, eps: float, residual=None, Wu=None) -> np.ndarray:
    """``h . W^T (+ R)``, or ``silu(h . W^T) * (h . Wu^T)`` with ``Wu``, where
    ``h = rmsnorm(X)`` (the norm before a projection: rms_norm(x, attn_norm)
    then attn_qkv in the pages' prefill layer); float64 throughout."""
    h = rmsnorm_f64(_as_f64(X).reshape(-1, k), weight, eps)
    g = h @ dequant_f64(qtype, W, n, k).T
    if Wu is not None:
        return silu_f64(g) * (h @ dequant_f64(qtype, Wu, n, k).T)
    if residual is not None:
        g = g + _as_f64(residual).reshape(g.shape)
    return g


# --------------------------------------------------------------------------
# Causal prefill attention over a KV cache
# --------------------------------------------------------------------------
def prefill_attention_f64(Q, K_cache, V_cache, T: int, pos0: int, num_heads: int, num_kv_heads: int,
                          head_dim: int, rows=None) -> np.ndarray:
    """``out[t, h] = sum_{j <= pos0+t} softmax_j(q_{t,h} . k_{j,g} / sqrt(d)) v_{j,g}``
    with ``g = h // (num_heads // num_kv_heads)``; float64, shape
    ``[len(rows)][num_heads * head_dim]`` (``rows`` defaults to all ``T``)."""
    return _attention_f64(_as_f64(Q), _as_f64(K_cache), _as_f64(V_cache), T, pos0, num_heads, num_kv_heads,
                          head_dim, rows)


def _attention_f64(Q64, K64, V64, T, pos0, num_heads, num_kv_heads, head_dim, rows=None):
    """The attention on float64 operands (see prefill_attention_f64)."""
    d = head_dim
    hpk = num_heads // num_kv_heads
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    Q64 = np.asarray(Q64, dtype=np.float64).reshape(T, num_heads * d)[rows]
    nk = pos0 + int(rows.max()) + 1 if len(rows) else 0
    K64 = np.asarray(K64, dtype=np.float64).reshape(-1, num_kv_heads * d)[:nk]
    V64 = np.asarray(V64, dtype=np.float64).reshape(-1, num_kv_heads * d)[:nk]
    out = np.zeros((len(rows), num_heads * d), dtype=np.float64)
    if not len(rows):
        return out
    # key j is visible to row t when j <= pos0 + t
    visible = np.arange(nk)[None, :] <= (pos0 + rows)[:, None]
    for h in range(num_heads):
        g = h // hpk
        q = Q64[:, h * d:(h + 1) * d]
        k = K64[:, g * d:(g + 1) * d]
        v = V64[:, g * d:(g + 1) * d]
        s = (q @ k.T) / np.sqrt(d)
        s = np.where(visible, s, -np.inf)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h * d:(h + 1) * d] = (e @ v) / e.sum(axis=1, keepdims=True)
    return out


def prefill_attention_f16_inputs_f64(Q, K_cache, V_cache, T: int, pos0: int, num_heads: int,
                                     num_kv_heads: int, head_dim: int, rows=None) -> np.ndarray:
    """The same attention after rounding ``q``, ``k`` and ``v`` to fp16 (the
    flash form's tensor-core inputs), then in float64."""
    r16 = lambda a: np.asarray(a, dtype=np.float32).astype(np.float16).astype(np.float64)  # noqa: E731
    return prefill_attention_f64(r16(Q), r16(K_cache), r16(V_cache), T, pos0, num_heads, num_kv_heads,
                                 head_dim, rows=rows)


# --------------------------------------------------------------------------
# One prefill layer over a chunk: norm -> qkv (k, v into the cache) ->
# attention -> output projection + residual -> FFN sublayer
# --------------------------------------------------------------------------
def prefill_layer_f64(qtype: int, X, attn_norm, ffn_norm, eps: float, Wqkv, Wo, Wg, Wu, Wd, hidden: int,
                      inter: int, num_heads: int, num_kv_heads: int, head_dim: int, K_cache, V_cache,
                      pos0: int):
    """The layer on the T rows of ``X`` (positions ``pos0 .. pos0 + T - 1``):

    * ``h = rmsnorm(X) * attn_norm``; ``q, k, v = h . Wq^T, h . Wk^T, h . Wv^T``
      with ``Wqkv`` = the ``H d`` q rows, then the ``KV d`` k rows, then the v rows;
    * the cache rows ``pos0 .. pos0 + T - 1`` become ``k`` and ``v``;
    * ``a = attention(q, caches)`` (causal, grouped KV heads);
    * ``X1 = X + a . Wo^T`` (``Wo`` is ``[hidden][H d]``);
    * ``X2 = X1 + down(silu(h2 . Wg^T) * (h2 . Wu^T))``, ``h2 = rmsnorm(X1) * ffn_norm``.

    Returns ``(X2, K, V)`` in float64; ``K`` and ``V`` are the updated caches
    (copies; rows outside the chunk as given)."""
    def norm(rows, w):  # float64 in, float64 out (no float32 round trip)
        w64 = _as_f64(w).reshape(1, -1)
        return rows / np.sqrt(np.mean(rows * rows, axis=-1, keepdims=True) + float(eps)) * w64

    X64 = _as_f64(X).reshape(-1, hidden)
    T = X64.shape[0]
    qd, kvd = num_heads * head_dim, num_kv_heads * head_dim
    row_bytes = _row_bytes(qtype, hidden)
    Wqkv_b = np.ascontiguousarray(Wqkv, dtype=np.uint8).reshape(-1)
    Wq = Wqkv_b[:qd * row_bytes]
    Wk = Wqkv_b[qd * row_bytes:(qd + kvd) * row_bytes]
    Wv = Wqkv_b[(qd + kvd) * row_bytes:(qd + 2 * kvd) * row_bytes]
    h = norm(X64, attn_norm)
    q = h @ dequant_f64(qtype, Wq, qd, hidden).T
    k = h @ dequant_f64(qtype, Wk, kvd, hidden).T
    v = h @ dequant_f64(qtype, Wv, kvd, hidden).T
    K = np.array(K_cache, dtype=np.float64).reshape(-1, kvd)
    V = np.array(V_cache, dtype=np.float64).reshape(-1, kvd)
    K[pos0:pos0 + T] = k
    V[pos0:pos0 + T] = v
    a = _attention_f64(q, K, V, T, pos0, num_heads, num_kv_heads, head_dim)
    X1 = X64 + a @ dequant_f64(qtype, Wo, hidden, qd).T
    h2 = norm(X1, ffn_norm)
    act = silu_f64(h2 @ dequant_f64(qtype, Wg, inter, hidden).T) * (h2 @ dequant_f64(qtype, Wu, inter, hidden).T)
    X2 = X1 + act @ dequant_f64(qtype, Wd, hidden, inter).T
    return X2, K, V
