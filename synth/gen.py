"""Seeded generators and the GGUF weight encoders (Q4_0, Q8_0, F16, Q4_K, Q5_K, Q6_K, IQ4_XS).

Recipe (the same for every workload):

* weights ``W ~ N(0, 0.02)``, activations ``X ~ N(0, 1)`` and residuals
  ``R ~ N(0, 1)`` are drawn with numpy's ``default_rng(seed)`` (PCG64) as
  float64 ``standard_normal`` values, scaled, then cast to float32;
* seeds: ``W`` uses ``seed``, ``X`` ``seed+1``, ``R`` ``seed+2``, the up weight of
  a gate/up pair ``seed+3`` and a down weight ``seed+4``;
* the f32 weight is encoded into GGUF blocks of 32 elements:

  - Q4_0 (18 bytes): fp16 scale ``d`` (little endian), then 16 bytes; byte ``j``
    holds element ``j`` in its low nibble and element ``j+16`` in its high
    nibble. The encoder takes the block's signed element of largest magnitude
    ``m`` and sets ``d = m / -8`` so that ``m`` itself maps to nibble 0; every
    element gets ``q = clamp(round(w / d) + 8, 0, 15)``.
  - Q8_0 (34 bytes): fp16 ``d = max|w| / 127`` then 32 int8
    ``q = clamp(round(w / d), -127, 127)``.

  ``round`` is half away from zero, ``w / d`` uses the f32 ``d`` before it is
  rounded to fp16 (round to nearest even) for storage, and an all-zero block
  gets ``d = 0`` with ``q = 8`` (Q4_0) or ``q = 0`` (Q8_0).
* or stored as F16: every element rounded to its nearest binary16 value (ties
  to even), two little-endian bytes each, ``[n][2k]`` bytes.

Prefill attention (``attention_case``): the query rows ``Q`` and the K and V
caches are ``N(0, 1)`` float32 draws with seeds ``seed``, ``seed+1`` and
``seed+2`` (rows of unit RMS, as the pages' per-head QK norm leaves them).

This is the inverse direction of what the prefill path computes; the decoding
and the products are not here.
"""

from __future__ import annotations

import numpy as np

F16 = 1   # GGUF type id
Q4_0 = 2  # GGUF type id
Q8_0 = 8  # GGUF type id
Q4_K = 12  # GGUF type id (256-element superblocks of 144 bytes)
Q5_K = 13  # GGUF type id (256-element superblocks of 176 bytes)
Q6_K = 14  # GGUF type id (256-element superblocks of 210 bytes)
IQ4_XS = 23  # GGUF type id (256-element superblocks of 136 bytes)
BLOCK_ELEMS = 32
_BLOCK_BYTES = {F16: 64, Q4_0: 18, Q8_0: 34, Q4_K: 18, Q5_K: 22, IQ4_XS: 17}
_SUPER_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, IQ4_XS: 136}
# IQ4_XS's code book, for the encoder's nearest-value search
_IQ4_BOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113], np.float64)


def block_bytes(qtype: int) -> int:
    """Bytes of 32 elements of ``qtype`` (one block; 64 bytes of F16; an
    eighth of a Q4_K superblock)."""
    return _BLOCK_BYTES[qtype]


def row_bytes(qtype: int, k: int) -> int:
    """Bytes of one weight row of ``k`` elements."""
    if qtype in _SUPER_BYTES:
        return k // 256 * _SUPER_BYTES[qtype]
    return k // BLOCK_ELEMS * _BLOCK_BYTES[qtype]


def _round_half_away(v: np.ndarray) -> np.ndarray:
    v = v.astype(np.float64)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def _pack_scale(d32: np.ndarray) -> np.ndarray:
    """fp16 bits of ``d`` (RNE) as two little-endian bytes, shape ``[..., 2]``."""
    bits = d32.astype(np.float16).view(np.uint16)
    return np.stack([(bits & 0xFF).astype(np.uint8), (bits >> 8).astype(np.uint8)], axis=-1)


def quantize_q4_0(w: np.ndarray) -> np.ndarray:
    """Encode an f32 ``[n][k]`` weight (k % 32 == 0) into Q4_0 bytes ``[n][k/32*18]``."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % BLOCK_ELEMS == 0
    blk = w.reshape(n, k // BLOCK_ELEMS, BLOCK_ELEMS)
    idx = np.argmax(np.abs(blk), axis=-1)[..., None]
    m = np.take_along_axis(blk, idx, axis=-1)[..., 0]
    d = (m / np.float32(-8.0)).astype(np.float32)
    safe = np.where(d == 0, np.float32(1.0), d)
    ratio = (blk / safe[..., None]).astype(np.float32)
    q = np.clip(_round_half_away(ratio) + 8, 0, 15).astype(np.uint8)
    q = np.where((d == 0)[..., None], np.uint8(8), q)
    out = np.empty((n, k // BLOCK_ELEMS, 18), dtype=np.uint8)
    out[..., 0:2] = _pack_scale(d)
    out[..., 2:18] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(n, -1)


def quantize_q8_0(w: np.ndarray) -> np.ndarray:
    """Encode an f32 ``[n][k]`` weight (k % 32 == 0) into Q8_0 bytes ``[n][k/32*34]``."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % BLOCK_ELEMS == 0
    blk = w.reshape(n, k // BLOCK_ELEMS, BLOCK_ELEMS)
    amax = np.max(np.abs(blk), axis=-1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(d == 0, np.float32(1.0), d)
    ratio = (blk / safe[..., None]).astype(np.float32)
    q = np.clip(_round_half_away(ratio), -127, 127).astype(np.int8)
    q = np.where((d == 0)[..., None], np.int8(0), q)
    out = np.empty((n, k // BLOCK_ELEMS, 34), dtype=np.uint8)
    out[..., 0:2] = _pack_scale(d)
    out[..., 2:34] = q.view(np.uint8)
    return out.reshape(n, -1)


def quantize_f16(w: np.ndarray) -> np.ndarray:
    """Store an f32 ``[n][k]`` weight as F16 bytes ``[n][2k]`` (RNE, little endian)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    return np.ascontiguousarray(w.astype("<f2")).view(np.uint8).reshape(n, 2 * k)


def _pack_q4_k_scales(sc: np.ndarray, mn: np.ndarray) -> np.ndarray:
    """Eight 6-bit scales and mins ``[..., 8]`` into the 12 packed bytes."""
    out = np.zeros(sc.shape[:-1] + (12,), np.uint8)
    for j in range(4):
        out[..., j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        out[..., j + 4] = (mn[..., j] & 63) | ((mn[..., j + 4] >> 4) << 6)
        out[..., j + 8] = (sc[..., j + 4] & 15) | ((mn[..., j + 4] & 15) << 4)
    return out


def quantize_q4_k(w: np.ndarray) -> np.ndarray:
    """Encode an f32 ``[n][k]`` weight (k % 256 == 0) into Q4_K superblocks
    ``[n][k/256*144]``: per 32-element sub-block the range [lo, hi] (lo <= 0 <=
    hi widened to include 0) gives scale (hi - lo) / 15 and min -lo; d and
    dmin are the largest of them over 63 (stored as fp16), the 6-bit
    sub-scales round(scale / d) and round(min / dmin), and each code
    round((w + dmin m) / (d sc)) clamped to 0..15."""
    return _quantize_k(w, 4)


def quantize_q5_k(w: np.ndarray) -> np.ndarray:
    """Q5_K superblocks ``[n][k/256*176]`` the same way with codes 0..31 (scale
    (hi - lo) / 31): the low four bits as Q4_K's code bytes, the fifth bits in
    the 32 bytes after the scales."""
    return _quantize_k(w, 5)


def quantize_q6_k(w: np.ndarray) -> np.ndarray:
    """Encode an f32 ``[n][k]`` weight (k % 256 == 0) into Q6_K superblocks
    ``[n][k/256*210]``: per 16-element sub-block the signed element m of
    largest magnitude gives the sub-scale m / -32 (m maps to code 0); d is the
    largest |sub-scale| over 127 (fp16), the int8 scales round(sub-scale / d),
    and each code round(w / (d sc)) + 32 clamped to 0..63. Byte placement:
    low nibble of element 128 h + 32 c + l in byte 64 h + 32 (c % 2) + l
    (nibble c / 2), its top two bits at bits 2 c of byte 128 + 32 h + l, the
    scales at bytes 192-207 and d at 208-209."""
    w = np.ascontiguousarray(w, dtype=np.float32).astype(np.float64)
    n, k = w.shape
    nsb = k // 256
    x = w.reshape(n, nsb, 16, 16)
    idx = np.abs(x).argmax(axis=-1)
    m = np.take_along_axis(x, idx[..., None], axis=-1)[..., 0]
    sub = m / -32.0
    d16 = (np.abs(sub).max(axis=-1) / 127.0).astype(np.float16)
    df = d16.astype(np.float64)
    sc = np.where(df[..., None] > 0, np.clip(np.rint(sub / np.where(df > 0, df, 1.0)[..., None]), -127, 127), 0)
    sc = sc.astype(np.int64)
    step = df[..., None] * sc
    q = np.where(step[..., None] != 0, np.rint(x / np.where(step != 0, step, 1.0)[..., None]) + 32, 32)
    q = np.clip(q, 0, 63).astype(np.int64).reshape(n, nsb, 2, 4, 32)  # [half][c][l]
    out = np.zeros((n, nsb, 210), np.uint8)
    low = q & 15
    ql = low[:, :, :, 0:2, :] | (low[:, :, :, 2:4, :] << 4)  # [half][c % 2][l]: quarters c and c + 2
    out[..., 0:128] = ql.reshape(n, nsb, 128).astype(np.uint8)
    qh = np.zeros((n, nsb, 2, 32), np.int64)
    for c in range(4):
        qh |= (q[:, :, :, c, :] >> 4) << (2 * c)
    out[..., 128:192] = qh.reshape(n, nsb, 64).astype(np.uint8)
    out[..., 192:208] = sc.astype(np.int8).view(np.uint8)
    out[..., 208:210] = d16.view(np.uint16)[..., None].view(np.uint8).reshape(n, nsb, 2)
    return out.reshape(n, -1)


def quantize_iq4_xs(w: np.ndarray) -> np.ndarray:
    """Encode an f32 ``[n][k]`` weight (k % 256 == 0) into IQ4_XS superblocks
    ``[n][k/256*136]``: per 32-element sub-block the signed element m of
    largest magnitude gives the sub-scale m / -127 (m maps to the book's
    first entry, -127); d is the largest |sub-scale| over 31 (fp16), the
    six-bit scales ls = round(sub-scale / d) + 32 clamped to 1..63, and each
    element takes the book entry nearest to w / (d (ls - 32)). Byte
    placement: d at bytes 0-1, the scales' top two bits at bits 2 j of the
    little-endian word at bytes 2-3, their low nibbles at nibble j % 2 of
    byte 4 + j / 2, the code of element 32 j + l (l < 16) in the low nibble
    of byte 8 + 16 j + l and that of 32 j + 16 + l in its high nibble."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    if n > 1024:  # row blocks bound the float64 temporaries
        return np.concatenate([quantize_iq4_xs(w[i:i + 1024]) for i in range(0, n, 1024)])
    w = w.astype(np.float64)
    nsb = k // 256
    x = w.reshape(n, nsb, 8, 32)
    idx = np.abs(x).argmax(axis=-1)
    m = np.take_along_axis(x, idx[..., None], axis=-1)[..., 0]
    sub = m / -127.0
    d16 = (np.abs(sub).max(axis=-1) / 31.0).astype(np.float16)
    df = d16.astype(np.float64)
    s = np.where(df[..., None] > 0, np.clip(np.rint(sub / np.where(df > 0, df, 1.0)[..., None]), -31, 31), 0)
    ls = (s + 32).astype(np.int64)
    step = df[..., None] * s
    ratio = np.where(step[..., None] != 0, x / np.where(step != 0, step, 1.0)[..., None], 1.0)
    # the nearest entry (the lower one on a tie) by the midpoints of the sorted book
    code = np.searchsorted((_IQ4_BOOK[1:] + _IQ4_BOOK[:-1]) / 2, ratio, side="left").astype(np.int64)
    out = np.zeros((n, nsb, 136), np.uint8)
    out[..., 0:2] = d16.view(np.uint16)[..., None].view(np.uint8).reshape(n, nsb, 2)
    hi = np.zeros((n, nsb), np.int64)
    for j in range(8):
        hi |= ((ls[..., j] >> 4) & 3) << (2 * j)
        out[..., 4 + j // 2] |= ((ls[..., j] & 15) << (4 * (j % 2))).astype(np.uint8)
    out[..., 2] = (hi & 0xFF).astype(np.uint8)
    out[..., 3] = (hi >> 8).astype(np.uint8)
    qs = code[..., 0:16] | (code[..., 16:32] << 4)                     # [n][nsb][8][16]
    out[..., 8:] = qs.reshape(n, nsb, 128).astype(np.uint8)
    return out.reshape(n, -1)


def _quantize_k(w: np.ndarray, bits: int) -> np.ndarray:
    top = (1 << bits) - 1
    w = np.ascontiguousarray(w, dtype=np.float32).astype(np.float64)
    n, k = w.shape
    x = w.reshape(n, k // 256, 8, 32)
    lo = np.minimum(x.min(axis=-1), 0.0)
    hi = np.maximum(x.max(axis=-1), 0.0)
    scale = (hi - lo) / top
    mins = -lo
    d = scale.max(axis=-1) / 63.0
    dmin = mins.max(axis=-1) / 63.0
    d16 = d.astype(np.float16)
    dmin16 = dmin.astype(np.float16)
    df = d16.astype(np.float64)
    dmf = dmin16.astype(np.float64)
    sc = np.where(df[..., None] > 0, np.clip(np.rint(scale / np.where(df > 0, df, 1.0)[..., None]), 0, 63), 0)
    mn = np.where(dmf[..., None] > 0, np.clip(np.rint(mins / np.where(dmf > 0, dmf, 1.0)[..., None]), 0, 63), 0)
    sc = sc.astype(np.int64)
    mn = mn.astype(np.int64)
    step = df[..., None] * sc
    q = np.where(step[..., None] > 0,
                 np.rint((x + (dmf[..., None] * mn)[..., None]) / np.where(step > 0, step, 1.0)[..., None]), 0)
    q = np.clip(q, 0, top).astype(np.uint8).reshape(n, k // 256, 4, 2, 32)
    qs = ((q[:, :, :, 0, :] & 15) | ((q[:, :, :, 1, :] & 15) << 4)).reshape(n, k // 256, 128)
    out = np.zeros((n, k // 256, 144 if bits == 4 else 176), np.uint8)
    out[..., 0:2] = d16.view(np.uint16)[..., None].view(np.uint8).reshape(n, k // 256, 2)
    out[..., 2:4] = dmin16.view(np.uint16)[..., None].view(np.uint8).reshape(n, k // 256, 2)
    out[..., 4:16] = _pack_q4_k_scales(sc, mn)
    if bits == 4:
        out[..., 16:] = qs
    else:
        qh = np.zeros((n, k // 256, 32), np.uint8)
        for g in range(4):
            qh |= ((q[:, :, g, 0, :] >> 4) << (2 * g)).astype(np.uint8)
            qh |= ((q[:, :, g, 1, :] >> 4) << (2 * g + 1)).astype(np.uint8)
        out[..., 16:48] = qh
        out[..., 48:] = qs
    return out.reshape(n, -1)


def quantize(qtype: int, w: np.ndarray) -> np.ndarray:
    if qtype == F16:
        return quantize_f16(w)
    if qtype == Q4_K:
        return quantize_q4_k(w)
    if qtype == Q5_K:
        return quantize_q5_k(w)
    if qtype == Q6_K:
        return quantize_q6_k(w)
    if qtype == IQ4_XS:
        return quantize_iq4_xs(w)
    if qtype == Q4_0:
        return quantize_q4_0(w)
    if qtype == Q8_0:
        return quantize_q8_0(w)
    raise ValueError(f"unsupported qtype {qtype}")


def weight_f32(n: int, k: int, seed: int, sigma: float = 0.02) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, k)) * sigma).astype(np.float32)


def activations(rows: int, cols: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, cols)) * sigma).astype(np.float32)


# Scale classes of ``random_blocks``: ranges of the fp16 exponent field of d
# (0 = subnormal). Every class draws both signs and random mantissas.
SCALE_CLASSES = {
    "subnormal": (0, 0),      # |d| in [2^-24, 2^-14)
    "small": (1, 5),          # [2^-14, 2^-9)
    "typical": (6, 12),       # [2^-9, 2^-2), where quantized model weights sit
    "large": (16, 30),        # [2, 65504], capped by fp16_range below
    "mixed": (0, 30),         # every finite exponent, block by block
}


def random_blocks(qtype: int, n: int, k: int, seed: int, scale_class: str = "mixed",
                  fp16_range: bool = False) -> np.ndarray:
    """Arbitrary GGUF blocks ``[n][k/32*bytes]``: uniformly random payload bytes
    (every Q4_0 nibble 0..15, every Q8_0 code -128..127) and fp16 scales of both
    signs whose exponent field is uniform over the class's range (random
    mantissa; the subnormal class has a nonzero mantissa). Scales are finite.
    For F16 the elements themselves are drawn that way.

    ``fp16_range``: cap |d| so that |d * q| stays within fp16's largest finite
    value 65504 for every code (|q| <= 8 for Q4_0, 128 for Q8_0): the scale's
    exponent field is at most 27 (Q4_0) or 23 (Q8_0), which with any mantissa
    gives |d| <= 8188 or 511.75.
    """
    lo, hi = SCALE_CLASSES[scale_class]
    if qtype in _SUPER_BYTES:
        # random bytes; d and dmin (Q6_K: d alone, at the end; IQ4_XS: d
        # alone, first) of both signs drawn from the class
        rng = np.random.default_rng(seed)
        raw = rng.integers(0, 256, size=(n, k // 256, _SUPER_BYTES[qtype]), dtype=np.uint8)
        offs = (208,) if qtype == Q6_K else ((0,) if qtype == IQ4_XS else (0, 2))
        for off in offs:
            exp = rng.integers(lo, hi + 1, size=(n, k // 256)).astype(np.uint16)
            # |w| within fp16's range: |d| < 2^5 (63 x 31 x 2^5 < 65504);
            # Q6_K |d| < 16 (128 x 32 x 16), IQ4_XS |d| < 16 (127 x 32 x 16)
            if fp16_range:
                exp = np.minimum(exp, 18 if qtype in (Q6_K, IQ4_XS) else 19)
            man = rng.integers(0, 1024, size=(n, k // 256)).astype(np.uint16)
            man = np.where(exp == 0, np.maximum(man, 1), man)
            sign = rng.integers(0, 2, size=(n, k // 256)).astype(np.uint16)
            bits = (sign << 15) | (exp << 10) | man
            raw[..., off] = (bits & 0xFF).astype(np.uint8)
            raw[..., off + 1] = (bits >> 8).astype(np.uint8)
        return raw.reshape(n, -1)
    if qtype == F16:
        # every element an fp16 value of both signs, exponent field uniform over
        # the class (nonzero mantissa in the subnormal class)
        rng = np.random.default_rng(seed)
        exp = rng.integers(lo, hi + 1, size=(n, k)).astype(np.uint16)
        man = rng.integers(0, 1024, size=(n, k)).astype(np.uint16)
        man = np.where(exp == 0, np.maximum(man, 1), man)
        sign = rng.integers(0, 2, size=(n, k)).astype(np.uint16)
        bits = ((sign << 15) | (exp << 10) | man).astype("<u2")
        return np.ascontiguousarray(bits).view(np.uint8).reshape(n, 2 * k)
    if fp16_range:
        hi = min(hi, 27 if qtype == Q4_0 else 23)
    rng = np.random.default_rng(seed)
    bb = block_bytes(qtype)
    raw = rng.integers(0, 256, size=(n, k // BLOCK_ELEMS, bb), dtype=np.uint8)
    exp = rng.integers(lo, hi + 1, size=(n, k // BLOCK_ELEMS)).astype(np.uint16)
    man = rng.integers(0, 1024, size=(n, k // BLOCK_ELEMS)).astype(np.uint16)
    man = np.where(exp == 0, np.maximum(man, 1), man)
    sign = rng.integers(0, 2, size=(n, k // BLOCK_ELEMS)).astype(np.uint16)
    bits = (sign << 15) | (exp << 10) | man
    raw[..., 0] = (bits & 0xFF).astype(np.uint8)
    raw[..., 1] = (bits >> 8).astype(np.uint8)
    return raw.reshape(n, -1)


def make_case(qtype: int, n: int, k: int, T: int, *, residual: bool = False,
              gate_up: bool = False, seed: int = 0) -> dict:
    """One seeded problem: quantized ``W`` (and ``Wu`` for a gate/up pair), ``X``, ``R``.

    Returns numpy arrays: ``W``/``Wu`` uint8 ``[n][k/32*bytes]``, ``X`` f32
    ``[T][k]``, ``R`` f32 ``[T][n]`` or ``None``.
    """
    case = {"qtype": qtype, "n": n, "k": k, "T": T}
    case["W"] = quantize(qtype, weight_f32(n, k, seed))
    case["Wu"] = quantize(qtype, weight_f32(n, k, seed + 3)) if gate_up else None
    case["X"] = activations(T, k, seed + 1)
    case["R"] = activations(T, n, seed + 2) if residual else None
    return case


def attention_case(T: int, pos0: int, num_heads: int, num_kv_heads: int, head_dim: int = 256,
                   seed: int = 0, cache_rows: int | None = None) -> dict:
    """One seeded prefill-attention problem: ``Q`` f32 ``[T][num_heads * d]``
    (seed), the K and V caches f32 ``[cache_rows][num_kv_heads * d]`` (seed+1,
    seed+2), all ``N(0, 1)``; ``cache_rows`` defaults to ``pos0 + T``."""
    rows = pos0 + T if cache_rows is None else cache_rows
    return {
        "T": T, "pos0": pos0, "num_heads": num_heads, "num_kv_heads": num_kv_heads, "head_dim": head_dim,
        "Q": activations(T, num_heads * head_dim, seed),
        "K": activations(rows, num_kv_heads * head_dim, seed + 1),
        "V": activations(rows, num_kv_heads * head_dim, seed + 2),
    }


# Named workloads: shapes of the prefill projections the pages run, at their
# chunk sizes (512 rows by default, 2048 on a unified-memory box).
WORKLOADS = {
    # Q8_0 GEMM, 256 x 512 weight, 16 tokens (the small reference problem)
    "q8_0_n256_k512_t16": dict(qtype=Q8_0, n=256, k=512, T=16),
    # Q4_0 GEMM + residual, 4096 x 4096, 512 tokens
    "q4_0_n4096_k4096_t512_res": dict(qtype=Q4_0, n=4096, k=4096, T=512, residual=True),
    # fused gate/up SwiGLU, 12288 x 4096 each, then down 4096 x 12288 + residual
    "swiglu_q4_0_n12288_k4096_t512": dict(qtype=Q4_0, n=12288, k=4096, T=512, gate_up=True),
    "down_q4_0_n4096_k12288_t512_res": dict(qtype=Q4_0, n=4096, k=12288, T=512, residual=True),
    "swiglu_q8_0_n12288_k4096_t512": dict(qtype=Q8_0, n=12288, k=4096, T=512, gate_up=True),
    "down_q8_0_n4096_k12288_t512_res": dict(qtype=Q8_0, n=4096, k=12288, T=512, residual=True),
}
