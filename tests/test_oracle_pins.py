"""Pins of the CPU oracle to facts outside itself (no GPU).

* hand-built blocks with values derived from the block definitions
  (``tests/golden/*.txt``, each with its source);
* the fp16 decoder against two independent decoders over all 65,536 bit
  patterns;
* exactly representable fp16 values (the dequant test idea of aprender-serve
  0.70.2 src/cuda/executor/gdn_prefill_ops.rs, ``f16_weight_dequantizes_on_the_device``);
* brute force: exact rational dot products on tiny shapes, with an independent
  block parser (``struct``) and an independent fp16 decoder;
* invariants that any correct implementation satisfies exactly.
"""

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
QTYPES = [synth.Q4_0, synth.Q8_0, synth.F16, synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.IQ4_XS]
KQ = (synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.IQ4_XS)


def _kk(qtype, k):
    """k as given, or widened to whole 256-element superblocks for the K-quants."""
    return max(256, k // 256 * 256) if qtype in KQ else k


def load_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            out[key] = rest.split()
    qtype = int(out["qtype"][0])
    byts = np.array([int(b, 16) for b in out["bytes"]], dtype=np.uint8)
    vals = np.array([float(v) for v in out["values"]], dtype=np.float64)
    return qtype, byts, vals


GOLDEN_FILES = sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt"))


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_golden_block_dequant(name):
    qtype, byts, vals = load_golden(name)
    got64 = oracle.dequant_f64(qtype, byts, 1, 32)[0]
    got32 = oracle.dequant_f32(qtype, byts, 1, 32)[0]
    np.testing.assert_array_equal(got64, vals)
    np.testing.assert_array_equal(got32.astype(np.float64), vals)


def test_golden_files_present():
    assert {"q4_0_zero_block.txt", "q4_0_nibble_order.txt", "q8_0_half_scale.txt",
            "q8_0_subnormal_scale.txt", "q4_0_negative_scale.txt", "f16_exact_values.txt"} <= set(GOLDEN_FILES)


# ---------------------------------------------------------------- F16 weights
def test_f16_weight_page_values_come_back_unchanged():
    # aprender-serve 0.70.2 src/cuda/executor/gdn_prefill_ops.rs,
    # f16_weight_dequantizes_on_the_device: n = 2, k = 64, w = i * 0.5 - 16 for
    # element i in row-major order, stored as little-endian halves
    n, k = 2, 64
    want = np.array([i * 0.5 - 16.0 for i in range(n * k)]).reshape(n, k)
    raw = np.frombuffer(b"".join(struct.pack("<e", v) for v in want.reshape(-1)), np.uint8).reshape(n, 2 * k)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.F16, raw, n, k), want)
    got32 = oracle.dequant_f32(synth.F16, raw, n, k)
    assert got32.dtype == np.float32
    np.testing.assert_array_equal(got32.astype(np.float64), want)
    # the encoder writes exactly those bytes
    np.testing.assert_array_equal(synth.quantize(synth.F16, want.astype(np.float32)), raw)


def test_f16_weight_equals_a_q8_0_weight_with_the_same_values():
    # a Q8_0 block whose values d * q are fp16 values (d = 2^-3, |q| <= 127:
    # at most 7 significant bits), written as F16: every product is the same
    n, k, T = 3, 64, 2
    rng = np.random.default_rng(5)
    blk = np.zeros((n, k // 32, 34), np.uint8)
    blk[..., 0], blk[..., 1] = 0x00, 0x30                    # d = 0x3000 = 2^-3
    codes = rng.integers(-127, 128, size=(n, k // 32, 32)).astype(np.int8)
    blk[..., 2:] = codes.view(np.uint8)
    W8 = blk.reshape(n, -1)
    vals = codes.reshape(n, k).astype(np.float64) / 8.0
    W16 = np.frombuffer(b"".join(struct.pack("<e", v) for v in vals.reshape(-1)), np.uint8).reshape(n, 2 * k)
    X = synth.activations(T, k, 6)
    R = synth.activations(T, n, 7)
    np.testing.assert_array_equal(oracle.qgemm_f64(synth.F16, W16, n, k, X, R), oracle.qgemm_f64(synth.Q8_0, W8, n, k, X, R))
    np.testing.assert_array_equal(oracle.dequant_f32(synth.F16, W16, n, k), oracle.dequant_f32(synth.Q8_0, W8, n, k))


def test_f16_weight_has_no_block_scales_and_needs_its_byte_count():
    raw = np.zeros((2, 128), np.uint8)
    with pytest.raises(ValueError):
        oracle.block_scales_and_codes(synth.F16, raw, 2, 64)
    with pytest.raises(ValueError):
        oracle.dequant_f64(synth.F16, raw[:, :96], 2, 64)
    with pytest.raises(ValueError):
        oracle.dequant_f64(synth.F16, raw.reshape(-1)[:96], 1, 48)  # k % 32 != 0


# ---------------------------------------------------------------- Q4_K (layout read, not printed on the pages)
def _q4_k_superblock(d_bits, dmin_bits, sc, mn, q):
    """Bytes of one Q4_K superblock from d, dmin, 8 scales, 8 mins and 256
    codes in element order, packed by hand from the layout reading."""
    b = bytearray(144)
    b[0:2] = struct.pack("<H", d_bits)
    b[2:4] = struct.pack("<H", dmin_bits)
    for j in range(4):
        b[4 + j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[8 + j] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        b[12 + j] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    for g in range(4):
        for l in range(32):
            b[16 + 32 * g + l] = q[64 * g + l] | (q[64 * g + 32 + l] << 4)
    return bytes(b)


def test_q4_k_equals_q4_0_blocks_with_the_same_codes():
    # d = 2^-9, dmin = 2^-7, sub-scales 16..31 and mins 2 sc: every element is
    # d sc (q - 8), the Q4_0 block of scale d sc with the same code. Scales and
    # mins above 15 use the packing's top bits.
    rng = np.random.default_rng(21)
    n, k = 3, 512
    W4 = np.zeros((n, k // 32, 18), np.uint8)
    WK = bytearray()
    for i in range(n):
        for s_ in range(k // 256):
            sc = [int(v) for v in rng.integers(16, 32, size=8)]
            mn = [2 * v for v in sc]
            q = [int(v) for v in rng.integers(0, 16, size=256)]
            WK += _q4_k_superblock(0x1800, 0x2000, sc, mn, q)
            for j in range(8):
                blk = W4[i, 8 * s_ + j]
                blk[0:2] = np.frombuffer(struct.pack("<e", 2.0 ** -9 * sc[j]), np.uint8)
                for e in range(16):
                    blk[2 + e] = q[32 * j + e] | (q[32 * j + 16 + e] << 4)
    WK = np.frombuffer(bytes(WK), np.uint8).reshape(n, -1)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q4_K, WK, n, k),
                                  oracle.dequant_f64(synth.Q4_0, W4.reshape(n, -1), n, k))


def test_q4_k_sub_block_scales_and_mins_land_on_their_elements():
    # codes 1 everywhere, d = 1, dmin = 1: element e of sub-block j is sc_j - m_j
    sc = [1, 2, 3, 4, 17, 33, 48, 63]
    mn = [0, 1, 2, 3, 16, 40, 5, 62]
    raw = np.frombuffer(_q4_k_superblock(0x3C00, 0x3C00, sc, mn, [1] * 256), np.uint8).reshape(1, 144)
    w = oracle.dequant_f64(synth.Q4_K, raw, 1, 256)[0]
    for j in range(8):
        np.testing.assert_array_equal(w[32 * j:32 * (j + 1)], np.full(32, float(sc[j] - mn[j])))
    got_sc, got_mn = oracle.q4_k_scales_mins(raw[0, 4:16])
    assert list(got_sc) == sc and list(got_mn) == mn


def test_q4_k_codes_in_element_order():
    # d = 1, dmin = 0, unit scales: w = q; element e gets code e mod 16
    q = [e % 16 for e in range(256)]
    raw = np.frombuffer(_q4_k_superblock(0x3C00, 0x0000, [1] * 8, [0] * 8, q), np.uint8).reshape(1, 144)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q4_K, raw, 1, 256)[0], np.array(q, np.float64))


def _q5_k_superblock(d_bits, dmin_bits, sc, mn, q):
    """Q5_K bytes: the Q4_K header and scales, the fifth bits of the codes
    (bit 2 g of byte l for element 64 g + l, bit 2 g + 1 for 64 g + 32 + l),
    then the low four bits as Q4_K's code bytes."""
    k4 = _q4_k_superblock(d_bits, dmin_bits, sc, mn, [v & 15 for v in q])
    qh = bytearray(32)
    for g in range(4):
        for l in range(32):
            qh[l] |= ((q[64 * g + l] >> 4) << (2 * g)) | ((q[64 * g + 32 + l] >> 4) << (2 * g + 1))
    return k4[:16] + bytes(qh) + k4[16:]


def test_q5_k_without_fifth_bits_equals_q4_k():
    rng = np.random.default_rng(23)
    sc = [int(v) for v in rng.integers(0, 64, size=8)]
    mn = [int(v) for v in rng.integers(0, 64, size=8)]
    q = [int(v) for v in rng.integers(0, 16, size=256)]
    k4 = np.frombuffer(_q4_k_superblock(0x2C00, 0x2800, sc, mn, q), np.uint8).reshape(1, 144)
    k5 = np.frombuffer(_q5_k_superblock(0x2C00, 0x2800, sc, mn, q), np.uint8).reshape(1, 176)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q5_K, k5, 1, 256), oracle.dequant_f64(synth.Q4_K, k4, 1, 256))


def test_q5_k_fifth_bits_land_on_their_elements():
    # d = 1, dmin = 0, unit scales, low bits zero: element e is 16 x its fifth bit
    rng = np.random.default_rng(24)
    hb = [int(v) for v in rng.integers(0, 2, size=256)]
    raw = np.frombuffer(_q5_k_superblock(0x3C00, 0x0000, [1] * 8, [0] * 8, [16 * b for b in hb]), np.uint8)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q5_K, raw.reshape(1, 176), 1, 256)[0],
                                  16.0 * np.array(hb, np.float64))
    # and the codes 0 .. 31 in element order
    q = [e % 32 for e in range(256)]
    raw = np.frombuffer(_q5_k_superblock(0x3C00, 0x0000, [1] * 8, [0] * 8, q), np.uint8).reshape(1, 176)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q5_K, raw, 1, 256)[0], np.array(q, np.float64))


def test_q5_k_encoder_round_trip():
    n, k = 16, 512
    w = synth.weight_f32(n, k, seed=4)
    W = synth.quantize(synth.Q5_K, w)
    assert W.shape == (n, k // 256 * 176) and synth.block_bytes(synth.Q5_K) * (k // 32) == W.shape[1]
    err = np.abs(oracle.dequant_f64(synth.Q5_K, W, n, k) - w.astype(np.float64)).reshape(n, k // 256, 8, 32)
    rng_ = w.reshape(n, k // 256, 8, 32)
    step = (np.maximum(rng_.max(-1), 0) - np.minimum(rng_.min(-1), 0)) / 31.0
    assert np.all(err.max(-1) <= 0.75 * step + 0.01 * np.abs(w).max())


def test_q4_k_encoder_round_trip_and_sizes():
    n, k = 16, 512
    w = synth.weight_f32(n, k, seed=4)
    W = synth.quantize(synth.Q4_K, w)
    assert W.shape == (n, k // 256 * 144) and synth.block_bytes(synth.Q4_K) * (k // 32) == W.shape[1]
    err = np.abs(oracle.dequant_f64(synth.Q4_K, W, n, k) - w.astype(np.float64)).reshape(n, k // 256, 8, 32)
    rng_ = w.reshape(n, k // 256, 8, 32)
    step = (np.maximum(rng_.max(-1), 0) - np.minimum(rng_.min(-1), 0)) / 15.0
    assert np.all(err.max(-1) <= 0.75 * step + 0.01 * np.abs(w).max())
    with pytest.raises(ValueError):
        oracle.dequant_f64(synth.Q4_K, W[:, :144], n, 128)


def _q6_k_superblock(d_bits, sc, q):
    """Q6_K bytes from d's fp16 bits, 16 int8 scales and 256 six-bit codes,
    placed one element at a time: element 128 h + 32 c + l keeps its low four
    bits in nibble c // 2 of byte 64 h + 32 (c % 2) + l and its top two at bit
    2 c of byte 128 + 32 h + l; the scales at bytes 192-207, d at 208-209."""
    b = bytearray(210)
    for e in range(256):
        h, c, l = e // 128, (e % 128) // 32, e % 32
        b[64 * h + 32 * (c % 2) + l] |= (q[e] & 15) << (4 * (c // 2))
        b[128 + 32 * h + l] |= (q[e] >> 4) << (2 * c)
    b[192:208] = struct.pack("<16b", *sc)
    b[208:210] = struct.pack("<H", d_bits)
    return bytes(b)


def test_q6_k_with_unit_scales_equals_q8_0_blocks():
    # every scale 1: element e is d (q_e - 32), the Q8_0 block of scale d with
    # code q_e - 32 (-32 .. 31)
    rng = np.random.default_rng(25)
    n, k = 3, 512
    W8 = np.zeros((n, k // 32, 34), np.uint8)
    W6 = bytearray()
    for i in range(n):
        for s_ in range(k // 256):
            d_bits = int(rng.integers(0x0400, 0x7800))
            q = [int(v) for v in rng.integers(0, 64, size=256)]
            W6 += _q6_k_superblock(d_bits, [1] * 16, q)
            for j in range(8):
                blk = W8[i, 8 * s_ + j]
                blk[0:2] = np.frombuffer(struct.pack("<H", d_bits), np.uint8)
                blk[2:34] = np.array([v - 32 for v in q[32 * j:32 * (j + 1)]], np.int8).view(np.uint8)
    W6 = np.frombuffer(bytes(W6), np.uint8).reshape(n, -1)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q6_K, W6, n, k),
                                  oracle.dequant_f64(synth.Q8_0, W8.reshape(n, -1), n, k))


def test_q6_k_scales_land_on_their_sixteen_elements():
    # d = 1, every code 33 (q - 32 = 1): element e is the int8 scale of e // 16
    sc = [1, -1, 2, -128, 127, 0, 5, -7, 64, -64, 3, 33, -100, 99, 11, -2]
    raw = np.frombuffer(_q6_k_superblock(0x3C00, sc, [33] * 256), np.uint8).reshape(1, 210)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q6_K, raw, 1, 256)[0],
                                  np.repeat(np.array(sc, np.float64), 16))


def test_q6_k_codes_in_element_order():
    # d = 1, unit scales: w = q - 32; element e gets code e mod 64, then a
    # code whose top bits alone are set
    q = [e % 64 for e in range(256)]
    raw = np.frombuffer(_q6_k_superblock(0x3C00, [1] * 16, q), np.uint8).reshape(1, 210)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q6_K, raw, 1, 256)[0], np.array(q, np.float64) - 32)
    q = [48 if e == 201 else 32 for e in range(256)]
    raw = np.frombuffer(_q6_k_superblock(0x4000, [1] * 16, q), np.uint8).reshape(1, 210)
    want = np.zeros(256)
    want[201] = 2.0 * 16
    np.testing.assert_array_equal(oracle.dequant_f64(synth.Q6_K, raw, 1, 256)[0], want)


def test_q6_k_encoder_round_trip_and_sizes():
    n, k = 16, 512
    w = synth.weight_f32(n, k, seed=4)
    W = synth.quantize(synth.Q6_K, w)
    assert W.shape == (n, k // 256 * 210) == (n, synth.row_bytes(synth.Q6_K, k))
    err = np.abs(oracle.dequant_f64(synth.Q6_K, W, n, k) - w.astype(np.float64)).reshape(n, k // 256, 16, 16)
    amax = np.abs(w.reshape(n, k // 256, 16, 16)).max(-1)
    # a step of about amax / 32, rounded to nearest; the 8-bit scale and fp16 d
    # add a few hundredths of the largest value
    assert np.all(err.max(-1) <= amax / 64 * 1.1 + 0.02 * np.abs(w).max())
    with pytest.raises(ValueError):
        oracle.dequant_f64(synth.Q6_K, W[:, :210], n, 128)


def test_f16_weights_reach_every_finite_half():
    # the random F16 generator draws every exponent field 0..30 and no inf/NaN;
    # the oracle decodes each element to its binary16 value
    W = synth.random_blocks(synth.F16, 16, 256, seed=3)
    bits = W.view("<u2")
    exp = (bits >> 10) & 0x1F
    assert set(np.unique(exp)) == set(range(31))
    np.testing.assert_array_equal(oracle.dequant_f64(synth.F16, W, 16, 256), bits.view(np.float16).astype(np.float64))


# ---------------------------------------------------------------- fp16 decode
def _struct_half(bits):
    return struct.unpack("<e", struct.pack("<H", int(bits)))[0]


def test_fp16_decode_all_patterns_vs_numpy_and_struct():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.fp16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    # a third, unrelated decoder on a stride of patterns
    for b in range(0, 65536, 97):
        s = _struct_half(b)
        if math.isnan(s):
            assert math.isnan(ours[b])
        else:
            assert ours[b] == s


def test_fp16_exactly_representable_values():
    # i * 0.5 - 16 for i in 0..127: exactly representable, distinct and signed.
    want = [i * 0.5 - 16.0 for i in range(128)]
    bits = [struct.unpack("<H", struct.pack("<e", v))[0] for v in want]
    got = oracle.fp16_bits_to_f64(np.array(bits, dtype=np.uint16))
    assert list(got) == want


def test_fp16_decode_landmarks():
    assert oracle.fp16_bits_to_f64(np.uint16(0x3C00)) == 1.0       # page bytes 0x00, 0x3C
    assert oracle.fp16_bits_to_f64(np.uint16(0x0001)) == 2.0 ** -24
    assert oracle.fp16_bits_to_f64(np.uint16(0x03FF)) == 1023 * 2.0 ** -24
    assert oracle.fp16_bits_to_f64(np.uint16(0x0400)) == 2.0 ** -14
    assert oracle.fp16_bits_to_f64(np.uint16(0x7BFF)) == 65504.0
    assert oracle.fp16_bits_to_f64(np.uint16(0xC000)) == -2.0
    assert oracle.fp16_bits_to_f64(np.uint16(0x7C00)) == np.inf

def _iq4_xs_superblock(d_bits, ls, codes):
    """IQ4_XS bytes from d's fp16 bits, eight six-bit scales and 256 four-bit
    codes, placed one at a time: scale j's low nibble at nibble j % 2 of byte
    4 + j // 2, its top two bits at bits 2 j of the word at bytes 2-3; the code
    of element 32 j + l at nibble l // 16 of byte 8 + 16 j + l % 16."""
    b = bytearray(136)
    b[0:2] = struct.pack("<H", d_bits)
    word = 0
    for j in range(8):
        b[4 + j // 2] |= (ls[j] & 15) << (4 * (j % 2))
        word |= (ls[j] >> 4) << (2 * j)
    b[2:4] = struct.pack("<H", word)
    for e in range(256):
        j, l = e // 32, e % 32
        b[8 + 16 * j + l % 16] |= codes[e] << (4 * (l // 16))
    return bytes(b)


def test_iq4_xs_with_a_linear_book_equals_q4_0_blocks():
    # with the book replaced by c - 8, sub-block j is the Q4_0 block of scale
    # d (ls_j - 32) over the same 16 code bytes (d a power of two, so that
    # scale is an fp16 value)
    rng = np.random.default_rng(31)
    n, k = 3, 512
    W4 = bytearray()
    WX = bytearray()
    for i in range(n):
        for s_ in range(k // 256):
            e = int(rng.integers(-8, 3))
            ls = [int(v) for v in rng.integers(0, 64, size=8)]
            codes = [int(v) for v in rng.integers(0, 16, size=256)]
            sb = _iq4_xs_superblock(struct.unpack("<H", struct.pack("<e", 2.0 ** e))[0], ls, codes)
            WX += sb
            for j in range(8):
                W4 += struct.pack("<e", 2.0 ** e * (ls[j] - 32)) + sb[8 + 16 * j:24 + 16 * j]
    WX = np.frombuffer(bytes(WX), np.uint8).reshape(n, -1)
    W4 = np.frombuffer(bytes(W4), np.uint8).reshape(n, -1)
    lin = tuple(range(-8, 8))
    np.testing.assert_array_equal(oracle.qref._dequant_iq4_xs(WX, n, k, table=lin),
                                  oracle.dequant_f64(synth.Q4_0, W4, n, k))


def test_iq4_xs_scales_land_on_their_sub_blocks():
    # d = 1, every code 8 with the identity book (c stands for c): element e is
    # 8 (ls_{e // 32} - 32); the default book gives entry 8 times ls - 32
    ls = [0, 63, 32, 33, 17, 48, 31, 1]
    raw = np.frombuffer(_iq4_xs_superblock(0x3C00, ls, [8] * 256), np.uint8).reshape(1, 136)
    want = np.repeat(np.array(ls, np.float64) - 32, 32)
    np.testing.assert_array_equal(oracle.qref._dequant_iq4_xs(raw, 1, 256, table=tuple(range(16)))[0], 8 * want)
    np.testing.assert_array_equal(oracle.iq4_xs_scales(raw)[0], np.array(ls) - 32)
    np.testing.assert_array_equal(oracle.dequant_f64(synth.IQ4_XS, raw, 1, 256)[0],
                                  oracle.IQ4_NL_VALUES[8] * want)


def test_iq4_xs_codes_in_element_order():
    # d = 1, every scale 33 (ls - 32 = 1), the identity book: element e is its
    # own code; then one element's code alone set
    codes = [(e * 7 + e // 32) % 16 for e in range(256)]
    raw = np.frombuffer(_iq4_xs_superblock(0x3C00, [33] * 8, codes), np.uint8).reshape(1, 136)
    np.testing.assert_array_equal(oracle.qref._dequant_iq4_xs(raw, 1, 256, table=tuple(range(16)))[0],
                                  np.array(codes, np.float64))
    np.testing.assert_array_equal(oracle.dequant_f64(synth.IQ4_XS, raw, 1, 256)[0],
                                  np.array([oracle.IQ4_NL_VALUES[c] for c in codes], np.float64))


def test_iq4_xs_book_shape():
    # the book's values are taken as given (nothing on the pages fixes them);
    # what the format needs of it: 16 distinct increasing int8 values that
    # reach -127, so that |w| <= 127 |d (ls - 32)| and fp32 holds w exactly
    book = np.array(oracle.IQ4_NL_VALUES)
    assert book.shape == (16,) and np.all(np.diff(book) > 0)
    assert book.min() == -127 and book.max() < 128


def test_iq4_xs_encoder_round_trip_and_sizes():
    n, k = 16, 512
    w = synth.weight_f32(n, k, seed=6)
    W = synth.quantize(synth.IQ4_XS, w)
    assert W.shape == (n, k // 256 * 136) == (n, synth.row_bytes(synth.IQ4_XS, k))
    deq = oracle.dequant_f64(synth.IQ4_XS, W, n, k)
    err = np.abs(deq - w.astype(np.float64)).reshape(n, k // 256, 8, 32)
    amax = np.abs(w.reshape(n, k // 256, 8, 32)).max(-1)
    # the book's widest gap (24 of 127) at a step of amax / 127, the 6-bit
    # scale and fp16 d adding a few hundredths of the largest value
    assert np.all(err.max(-1) <= amax * 12.5 / 127 + 0.04 * np.abs(w).max())
    assert np.linalg.norm(deq - w) / np.linalg.norm(w) < 0.12
    with pytest.raises(ValueError):
        oracle.dequant_f64(synth.IQ4_XS, W[:, :136], n, 128)


# ---------------------------------------------------------------- brute force
def _parse_block_independent(qtype, blk: bytes):
    """(Fraction d, list of 32 int codes) via struct, not the oracle's decoder."""
    if qtype == synth.F16:  # 32 binary16 values, no scale
        return Fraction(1), [Fraction(v) for v in struct.unpack("<32e", blk)]
    d = Fraction(struct.unpack("<e", blk[0:2])[0])
    if qtype == synth.Q4_0:
        lo = [(b & 0xF) - 8 for b in blk[2:18]]
        hi = [(b >> 4) - 8 for b in blk[2:18]]
        return d, lo + hi
    return d, list(struct.unpack("32b", blk[2:34]))


def _random_blocks(rng, qtype, n, k):
    """Random raw bytes with finite scales (exponent field kept below 31); for
    F16 every element is such a half; for Q4_K d and dmin of every superblock."""
    if qtype in KQ:
        sbb = {synth.Q4_K: 144, synth.Q5_K: 176, synth.Q6_K: 210, synth.IQ4_XS: 136}[qtype]
        raw = rng.integers(0, 256, size=(n, k // 256, sbb), dtype=np.uint8)
        for b in {synth.Q6_K: (209,), synth.IQ4_XS: (1,)}.get(qtype, (1, 3)):
            raw[..., b] = np.where((raw[..., b] & 0x7C) == 0x7C, raw[..., b] & 0xBF, raw[..., b])
        return raw.reshape(n, -1)
    bb = synth.block_bytes(qtype)
    raw = rng.integers(0, 256, size=(n, k // 32, bb), dtype=np.uint8)
    hi = raw[..., 1::2] if qtype == synth.F16 else raw[..., 1]
    hi = np.where((hi & 0x7C) == 0x7C, hi & 0xBF, hi)  # clear one exp bit
    if qtype == synth.F16:
        raw[..., 1::2] = hi
    else:
        raw[..., 1] = hi
    return raw.reshape(n, -1)


def _q4_k_row_independent(raw: bytes, k, five=False):
    """Exact values of one Q4_K (Q5_K: five=True) row, element by element with
    struct (the layout read in the oracle's header, written out here as plain
    loops)."""
    out = []
    sbb = 176 if five else 144
    qoff = 48 if five else 16
    for sb in range(k // 256):
        blk = raw[sbb * sb:sbb * (sb + 1)]
        d = Fraction(struct.unpack("<e", blk[0:2])[0])
        dmin = Fraction(struct.unpack("<e", blk[2:4])[0])
        s = blk[4:16]
        vals = [None] * 256
        for j in range(8):
            if j < 4:
                sc, m = s[j] & 63, s[j + 4] & 63
            else:
                sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4)
                m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
            g, hi = j // 2, j % 2
            for l in range(32):
                byte = blk[qoff + 32 * g + l]
                q = (byte >> 4) if hi else (byte & 15)
                if five:
                    q += 16 * ((blk[16 + l] >> (2 * g + hi)) & 1)
                vals[64 * g + 32 * hi + l] = d * sc * q - dmin * m
        out.extend(vals)
    return out


def _q6_k_row_independent(raw: bytes, k):
    """Exact values of one Q6_K row, element by element with struct: element
    128 h + 32 c + l takes nibble c // 2 of byte 64 h + 32 (c % 2) + l, bits
    2 c, 2 c + 1 of byte 128 + 32 h + l, scale byte 192 + (element % 256) // 16
    (int8) and d from bytes 208-209; w = d sc (q - 32)."""
    out = []
    for sb in range(k // 256):
        blk = raw[210 * sb:210 * (sb + 1)]
        d = Fraction(struct.unpack("<e", blk[208:210])[0])
        vals = [None] * 256
        for h in range(2):
            for c in range(4):
                for l in range(32):
                    e = 128 * h + 32 * c + l
                    lo = blk[64 * h + 32 * (c % 2) + l]
                    lo = (lo >> 4) if c >= 2 else (lo & 15)
                    hi = (blk[128 + 32 * h + l] >> (2 * c)) & 3
                    sc = struct.unpack("<b", blk[192 + e // 16:193 + e // 16])[0]
                    vals[e] = d * sc * ((lo | (hi << 4)) - 32)
        out.extend(vals)
    return out


_BOOK = [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113]


def _iq4_xs_row_independent(raw: bytes, k):
    """Exact values of one IQ4_XS row, element by element with struct:
    element 32 j + l takes nibble l // 16 of byte 8 + 16 j + l % 16 as its
    code c, scale ls_j from nibble j % 2 of byte 4 + j // 2 and bits 2 j,
    2 j + 1 of the word at bytes 2-3; w = d (ls_j - 32) book[c]."""
    out = []
    for sb in range(k // 256):
        blk = raw[136 * sb:136 * (sb + 1)]
        d = Fraction(struct.unpack("<e", blk[0:2])[0])
        word = struct.unpack("<H", blk[2:4])[0]
        for e in range(256):
            j, l = e // 32, e % 32
            ls = ((blk[4 + j // 2] >> (4 * (j % 2))) & 15) + 16 * ((word >> (2 * j)) & 3)
            c = (blk[8 + 16 * j + l % 16] >> (4 * (l // 16))) & 15
            out.append(d * (ls - 32) * _BOOK[c])
    return out


def _kq_row_independent(qtype, raw: bytes, k):
    if qtype == synth.IQ4_XS:
        return _iq4_xs_row_independent(raw, k)
    if qtype == synth.Q6_K:
        return _q6_k_row_independent(raw, k)
    return _q4_k_row_independent(raw, k, five=qtype == synth.Q5_K)


def _exact_qgemm(qtype, W, n, k, X, R):
    rows = []
    for i in range(n):
        if qtype in KQ:
            rows.append(_kq_row_independent(qtype, bytes(W[i]), k))
            continue
        bb = synth.block_bytes(qtype)
        wrow = []
        for b in range(k // 32):
            blk = bytes(W[i, b * bb:(b + 1) * bb])
            d, codes = _parse_block_independent(qtype, blk)
            wrow.extend(d * c for c in codes)
        rows.append(wrow)
    T = X.shape[0]
    Y = [[None] * n for _ in range(T)]
    for t in range(T):
        xs = [Fraction(float(v)) for v in X[t]]
        for i in range(n):
            acc = sum(x * w for x, w in zip(xs, rows[i]))
            if R is not None:
                acc += Fraction(float(R[t, i]))
            Y[t][i] = acc
    return Y, rows


def _ulp32(x):
    x = abs(np.float32(x))
    return float(np.spacing(x)) if x != 0 else float(np.spacing(np.float32(0)))


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T,res", [(3, 32, 2, False), (5, 64, 3, True), (2, 96, 1, True)])
def test_brute_force_exact_rationals(qtype, n, k, T, res):
    k = _kk(qtype, k)
    rng = np.random.default_rng(1234 + n + k + T + qtype)
    W = _random_blocks(rng, qtype, n, k)
    X = rng.standard_normal((T, k)).astype(np.float32)
    R = rng.standard_normal((T, n)).astype(np.float32) if res else None
    exact, wrows = _exact_qgemm(qtype, W, n, k, X, R)
    got = oracle.qgemm(qtype, W, n, k, X, R)
    assert got.shape == (T, n) and got.dtype == np.float32
    n_equal = 0
    for t in range(T):
        for i in range(n):
            e = exact[t][i]
            mag = sum(abs(Fraction(float(X[t, j])) * wrows[i][j]) for j in range(k))
            bound = 0.5 * _ulp32(float(e)) + float(mag) * (k + 2) * 2.0 ** -52
            assert abs(float(got[t, i]) - float(e)) <= bound, (t, i)
            n_equal += float(got[t, i]) == float(np.float32(float(e)))
    assert n_equal >= T * n - 1


@pytest.mark.parametrize("qtype", QTYPES)
def test_brute_force_dequant_exact(qtype):
    rng = np.random.default_rng(77 + qtype)
    n, k = 4, _kk(qtype, 64)
    W = _random_blocks(rng, qtype, n, k)
    _, rows = _exact_qgemm(qtype, W, n, k, np.zeros((1, k), np.float32), None)
    got = oracle.dequant_f32(qtype, W, n, k)
    for i in range(n):
        for j in range(k):
            if qtype in (synth.Q4_K, synth.Q5_K):  # d sc q - dmin m may need more than 24 bits: rounded once
                assert abs(Fraction(float(got[i, j])) - rows[i][j]) <= Fraction(_ulp32(float(got[i, j]))) / 2
            else:
                assert Fraction(float(got[i, j])) == rows[i][j]


@pytest.mark.parametrize("qtype", QTYPES)
def test_brute_force_swiglu(qtype):
    rng = np.random.default_rng(99 + qtype)
    n, k, T = 4, _kk(qtype, 64), 3
    Wg = synth.quantize(qtype, (rng.standard_normal((n, k)) * 0.3).astype(np.float32))
    Wu = synth.quantize(qtype, (rng.standard_normal((n, k)) * 0.3).astype(np.float32))
    X = rng.standard_normal((T, k)).astype(np.float32)
    g, _ = _exact_qgemm(qtype, Wg, n, k, X, None)
    u, _ = _exact_qgemm(qtype, Wu, n, k, X, None)
    got = oracle.gate_up_swiglu(qtype, Wg, Wu, n, k, X)
    for t in range(T):
        for i in range(n):
            gf, uf = float(g[t][i]), float(u[t][i])
            want = gf / (1.0 + math.exp(-gf)) * uf
            assert abs(float(got[t, i]) - want) <= _ulp32(want) + 1e-12 * abs(want)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("qtype", QTYPES)
def test_identity_x_returns_dequantized_weight(qtype):
    n, k = 8, _kk(qtype, 64)
    W = synth.quantize(qtype, synth.weight_f32(n, k, seed=5))
    X = np.eye(k, dtype=np.float32)
    Y = oracle.qgemm(qtype, W, n, k, X)
    np.testing.assert_array_equal(Y, oracle.dequant_f32(qtype, W, n, k).T)


@pytest.mark.parametrize("qtype", QTYPES)
def test_scaling_and_permutation(qtype):
    n, k, T = 16, _kk(qtype, 128), 7
    case = synth.make_case(qtype, n, k, T, seed=3)
    Y = oracle.qgemm(qtype, case["W"], n, k, case["X"])
    np.testing.assert_array_equal(oracle.qgemm(qtype, case["W"], n, k, 2 * case["X"]), 2 * Y)
    perm = np.random.default_rng(0).permutation(T)
    np.testing.assert_array_equal(oracle.qgemm(qtype, case["W"], n, k, case["X"][perm]), Y[perm])


def test_q4_block_reencoded_as_q8_dequantizes_identically():
    n, k = 6, 96
    W4 = synth.quantize_q4_0(synth.weight_f32(n, k, seed=11))
    blk = W4.reshape(n, k // 32, 18)
    W8 = np.empty((n, k // 32, 34), dtype=np.uint8)
    W8[..., 0:2] = blk[..., 0:2]
    lo = (blk[..., 2:] & 0xF).astype(np.int16) - 8
    hi = (blk[..., 2:] >> 4).astype(np.int16) - 8
    W8[..., 2:] = np.concatenate([lo, hi], axis=-1).astype(np.int8).view(np.uint8)
    np.testing.assert_array_equal(oracle.dequant_f32(synth.Q4_0, W4, n, k),
                                  oracle.dequant_f32(synth.Q8_0, W8.reshape(n, -1), n, k))


def test_zero_codes_give_residual_and_zero_swiglu():
    n, k, T = 5, 64, 4
    Wz = np.zeros((n, k // 32, 34), np.uint8)
    Wz[..., 1] = 0x3C  # d = 1.0, every q = 0
    Wz = Wz.reshape(n, -1)
    X = synth.activations(T, k, 1)
    R = synth.activations(T, n, 2)
    np.testing.assert_array_equal(oracle.qgemm(synth.Q8_0, Wz, n, k, X, R), R)
    Wu = synth.quantize_q8_0(synth.weight_f32(n, k, 4))
    np.testing.assert_array_equal(oracle.gate_up_swiglu(synth.Q8_0, Wz, Wu, n, k, X),
                                  np.zeros((T, n), np.float32))


def test_residual_is_added_once():
    n, k, T = 8, 64, 3
    case = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=9)
    y0 = oracle.qgemm_f64(synth.Q4_0, case["W"], n, k, case["X"])
    y1 = oracle.qgemm_f64(synth.Q4_0, case["W"], n, k, case["X"], case["R"])
    np.testing.assert_allclose(y1 - y0, case["R"].astype(np.float64), rtol=0, atol=1e-12)


def test_f16_input_mode_rounds_both_operands():
    n, k, T = 4, 64, 2
    case = synth.make_case(synth.Q4_0, n, k, T, seed=21)
    X = case["X"] * np.float32(1.0 + 2.0 ** -20)  # not fp16-representable
    a = oracle.qgemm_f16_inputs_f64(synth.Q4_0, case["W"], n, k, X)
    X16 = X.astype(np.float16).astype(np.float32)
    W16 = oracle.dequant_f32(synth.Q4_0, case["W"], n, k).astype(np.float16).astype(np.float64)
    b = X16.astype(np.float64) @ W16.T
    np.testing.assert_allclose(a, b, rtol=1e-15, atol=0)


# ---------------------------------------------------------------- encoder
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_quantizer_round_trip(qtype):
    n, k = 64, 256
    w = synth.weight_f32(n, k, seed=2)
    W = synth.quantize(qtype, w)
    d_bits, _ = oracle.block_scales_and_codes(qtype, W, n, k)
    d = np.abs(oracle.fp16_bits_to_f64(d_bits))
    err = np.abs(oracle.dequant_f64(qtype, W, n, k) - w.astype(np.float64)).reshape(n, k // 32, 32)
    # Q8_0 rounds to the nearest code; Q4_0 may also clamp 16 -> 15 (one more step).
    # The fp16 rounding of d adds at most 2^-11 relative on top.
    step = 0.5 if qtype == synth.Q8_0 else 1.0
    lim = d[..., None] * (step + 128 * 2.0 ** -11) + 1e-12
    assert np.all(err <= lim)


def test_q4_0_encoder_maps_signed_extreme_to_nibble_zero():
    w = np.zeros((1, 32), np.float32)
    w[0, 5] = 0.8
    w[0, 9] = -0.4
    W = synth.quantize_q4_0(w)
    d_bits, codes = oracle.block_scales_and_codes(synth.Q4_0, W, 1, 32)
    assert oracle.fp16_bits_to_f64(d_bits)[0, 0] == float(np.float16(-0.1))
    assert codes[0, 0, 5] == -8 and codes[0, 0, 9] == 4 and codes[0, 0, 0] == 0


# ------------------------------------------------------------------ FFN sublayer
# The pages run a batched RMSNorm (weight, eps) before the gate/up GEMM and add
# the down projection back into the rows (oxibonsai-kernels 0.1.4,
# encode_q_std_ffn_phase); the norm is read as x / sqrt(mean(x^2) + eps) * w.
def test_rmsnorm_hand_values():
    # [3, 4]: mean of squares 12.5, so 3 / sqrt(12.5) and 4 / sqrt(12.5), weights 1 and 2
    y = oracle.rmsnorm_f64(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(y, [[0.8485281374238571, 2.2627416997969525]], rtol=1e-15)
    # a constant row c with eps: c / sqrt(c^2 + eps); 2 / sqrt(4 + 5) = 2 / 3
    y = oracle.rmsnorm_f64(np.full((1, 4), 2.0), np.ones(4), 5.0)
    np.testing.assert_allclose(y, np.full((1, 4), 2.0 / 3.0), rtol=1e-15)
    # rows are normalised one by one: [1, 1] and [10, 10] both give [1, 1]
    y = oracle.rmsnorm_f64(np.array([[1.0, 1.0], [-10.0, -10.0]]), np.array([1.0, 0.5]), 0.0)
    np.testing.assert_array_equal(y, [[1.0, 0.5], [-1.0, -0.5]])


def test_rmsnorm_scale_invariance():
    X = synth.activations(3, 64, 5).astype(np.float64)
    w = synth.activations(1, 64, 6)[0]
    # scaling a row by 8 (a power of 4 times 2) leaves x / rms(x) unchanged
    # exactly: sqrt(64 m) = 8 sqrt(m) in floating point
    np.testing.assert_array_equal(oracle.rmsnorm_f64(8.0 * X, w, 0.0), oracle.rmsnorm_f64(X, w, 0.0))


def test_ffn_sublayer_special_cases():
    hidden, inter, T = 64, 96, 3
    X = synth.activations(T, hidden, 1)
    w = np.ones(hidden, np.float32)
    Wg = synth.quantize_q8_0(synth.weight_f32(inter, hidden, 2))
    Wu = synth.quantize_q8_0(synth.weight_f32(inter, hidden, 3))
    Wd = synth.quantize_q8_0(synth.weight_f32(hidden, inter, 4))
    # zero norm weight: the normed rows are zero, so is SwiGLU, and X comes back
    y = oracle.ffn_sublayer_f64(synth.Q8_0, X, np.zeros(hidden), 1e-6, Wg, Wu, Wd, hidden, inter)
    np.testing.assert_array_equal(y, X.astype(np.float64))
    # a down weight with every code zero adds nothing
    Wz = np.zeros((hidden, inter // 32, 34), np.uint8)
    Wz[..., 1] = 0x3C
    y = oracle.ffn_sublayer_f64(synth.Q8_0, X, w, 1e-6, Wg, Wu, Wz.reshape(hidden, -1), hidden, inter)
    np.testing.assert_array_equal(y, X.astype(np.float64))


def _block_values(raw, qtype, n, k):
    """Dequantized weight from the raw bytes, by the block rules (struct parse)."""
    if qtype in KQ:
        return np.array([[float(v) for v in _kq_row_independent(qtype, bytes(raw[i]), k)] for i in range(n)])
    if qtype == synth.F16:
        return np.array([struct.unpack("<%de" % k, bytes(raw[i])) for i in range(n)], dtype=np.float64)
    bb = 18 if qtype == synth.Q4_0 else 34
    out = np.zeros((n, k))
    for i in range(n):
        for b in range(k // 32):
            blk = bytes(raw[i, b * bb:(b + 1) * bb])
            d = struct.unpack("<e", blk[:2])[0]
            for j in range(32):
                if qtype == synth.Q4_0:
                    byte = blk[2 + (j % 16)]
                    q = (byte & 0xF if j < 16 else byte >> 4) - 8
                else:
                    q = struct.unpack("<b", blk[2 + j:3 + j])[0]
                out[i, 32 * b + j] = d * q
    return out


@pytest.mark.parametrize("qtype", QTYPES)
def test_ffn_sublayer_brute_force(qtype):
    """Element-by-element loops (struct block parsing, math.sqrt, math.exp)
    against the oracle's array form."""
    hidden, inter, T, eps = _kk(qtype, 32), _kk(qtype, 64), 2, 1e-5
    X = synth.activations(T, hidden, 7).astype(np.float64)
    w = synth.activations(1, hidden, 8)[0].astype(np.float64)
    raw = {}
    for name, (rows, cols, seed) in {"g": (inter, hidden, 9), "u": (inter, hidden, 10), "d": (hidden, inter, 11)}.items():
        raw[name] = synth.quantize(qtype, synth.weight_f32(rows, cols, seed))
    Wg, Wu, Wd = (_block_values(raw[n_], qtype, *s) for n_, s in
                  (("g", (inter, hidden)), ("u", (inter, hidden)), ("d", (hidden, inter))))
    want = np.zeros((T, hidden))
    for t in range(T):
        ms = sum(X[t, c] * X[t, c] for c in range(hidden)) / hidden
        h = [X[t, c] / math.sqrt(ms + eps) * w[c] for c in range(hidden)]
        act = []
        for i in range(inter):
            g = sum(h[c] * Wg[i, c] for c in range(hidden))
            u = sum(h[c] * Wu[i, c] for c in range(hidden))
            act.append(g / (1.0 + math.exp(-g)) * u)
        for o in range(hidden):
            want[t, o] = X[t, o] + sum(act[i] * Wd[o, i] for i in range(inter))
    got = oracle.ffn_sublayer_f64(qtype, X, w, eps, raw["g"], raw["u"], raw["d"], hidden, inter)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("qtype", QTYPES)
def test_normed_projection_reduces_to_projection(qtype):
    """Rows of +-1 have mean square 1, so with eps = 0 and unit weight the norm
    is the identity and the normed projection is the plain one (pinned above
    by brute force); a weight of 2 doubles it."""
    n, k, T = 40, _kk(qtype, 96), 5
    c = synth.make_case(qtype, n, k, T, residual=True, seed=12)
    X = np.where(synth.activations(T, k, 13) >= 0, 1.0, -1.0).astype(np.float32)
    ones = np.ones(k, np.float32)
    np.testing.assert_array_equal(oracle.normed_qgemm_f64(qtype, c["W"], n, k, X, ones, 0.0, c["R"]),
                                  oracle.qgemm_f64(qtype, c["W"], n, k, X, c["R"]))
    np.testing.assert_array_equal(oracle.normed_qgemm_f64(qtype, c["W"], n, k, X, 2 * ones, 0.0),
                                  2 * oracle.qgemm_f64(qtype, c["W"], n, k, X))
    Wu = synth.quantize(qtype, synth.weight_f32(n, k, 14))
    np.testing.assert_array_equal(oracle.normed_qgemm_f64(qtype, c["W"], n, k, X, ones, 0.0, Wu=Wu),
                                  oracle.gate_up_swiglu_f64(qtype, c["W"], Wu, n, k, X))


# ---------------------------------------------------------------- attention
# Causal prefill attention (aprender-serve 0.70.2
# src/cuda/executor/gdn_prefill_ops.rs, qwen35_prefill_attention and
# qwen35_attention_pass): each pin fixes a part of the definition, the
# 1/sqrt(d) scale, the mask j <= pos0 + t, the head grouping
# h / (heads / kv_heads) and the softmax normalisation, from facts the
# definition implies.
def _attn(c, rows=None, **over):
    a = dict(c)
    a.update(over)
    return oracle.prefill_attention_f64(a["Q"], a["K"], a["V"], a["T"], a["pos0"], a["num_heads"],
                                        a["num_kv_heads"], a["head_dim"], rows=rows)


def test_attention_first_position_sees_only_its_own_key():
    # row 0 at position 0 attends to key 0 alone: its weight is exactly 1
    c = synth.attention_case(3, 0, 4, 2, 16, seed=5)
    out = _attn(c)
    V = c["V"].astype(np.float64)
    for h in range(4):
        g = h // 2
        assert np.array_equal(out[0, h * 16:(h + 1) * 16], V[0, g * 16:(g + 1) * 16])


def test_attention_zero_query_is_the_running_mean_of_values():
    # q = 0: every visible score is 0, the weights uniform, the output the mean
    # of the values at positions 0 .. pos0 + t
    T, pos0, d = 6, 5, 8
    c = synth.attention_case(T, pos0, 2, 1, d, seed=6)
    c["Q"] = np.zeros_like(c["Q"])
    out = _attn(c)
    V = c["V"].astype(np.float64)
    running = np.cumsum(V, axis=0) / np.arange(1, len(V) + 1)[:, None]
    for t in range(T):
        for h in range(2):
            np.testing.assert_allclose(out[t, h * d:(h + 1) * d], running[pos0 + t], rtol=0, atol=1e-14)


def test_attention_two_keys_hand_value():
    # d = 4, one head, query at position 1: q = (2,0,0,0), k0 = (1,0,0,0),
    # k1 = 0, so the scores are 2 * 1 / sqrt(4) = 1 and 0, the weights
    # e / (e + 1) and 1 / (e + 1); v0 = (1,2,0,0), v1 = (0,0,3,0)
    e = math.e
    Q = np.array([[2.0, 0, 0, 0]], dtype=np.float32)
    K = np.array([[1.0, 0, 0, 0], [0, 0, 0, 0]], dtype=np.float32)
    V = np.array([[1.0, 2, 0, 0], [0, 0, 3, 0]], dtype=np.float32)
    out = oracle.prefill_attention_f64(Q, K, V, 1, 1, 1, 1, 4)
    want = [e / (e + 1), 2 * e / (e + 1), 3 / (e + 1), 0.0]
    np.testing.assert_allclose(out[0], want, rtol=1e-15, atol=0)


def test_attention_mask_hides_later_positions():
    T, pos0, d = 5, 3, 8
    c = synth.attention_case(T, pos0, 2, 2, d, seed=7)
    base = _attn(c)
    for t in range(T):
        # change every cache row after position pos0 + t: rows <= t keep their output
        K2, V2 = c["K"].copy(), c["V"].copy()
        K2[pos0 + t + 1:] += 1.5
        V2[pos0 + t + 1:] -= 2.0
        out = _attn(c, K=K2, V=V2)
        np.testing.assert_array_equal(out[:t + 1], base[:t + 1])
        if t + 1 < T:
            assert np.abs(out[t + 1:] - base[t + 1:]).max() > 1e-3
        # and the row's own position is visible to it
        V3 = c["V"].copy()
        V3[pos0 + t] += 1.0
        assert np.abs(_attn(c, V=V3)[t] - base[t]).max() > 1e-6


def test_attention_query_heads_share_kv_heads_in_consecutive_groups():
    # 4 query heads over 2 KV heads: heads 0, 1 read KV head 0 and heads 2, 3
    # read KV head 1 (h / 2, not h % 2)
    T, pos0, d = 4, 2, 8
    c = synth.attention_case(T, pos0, 4, 2, d, seed=8)
    base = _attn(c)
    V2 = c["V"].copy()
    V2[:, d:2 * d] *= 2.0  # KV head 1 only (exact in f32: the weights stay, the sums double)
    out = _attn(c, V=V2)
    np.testing.assert_array_equal(out[:, :2 * d], base[:, :2 * d])
    np.testing.assert_array_equal(out[:, 2 * d:], 2.0 * base[:, 2 * d:])


def test_attention_chunk_split_gives_the_same_rows():
    # rows 4..6 of a chunk at pos0 = 2 are the chunk of 3 rows at pos0 = 6 over
    # the same cache: the output of a row depends on its position, not on the chunk
    c = synth.attention_case(7, 2, 2, 1, 16, seed=9)
    whole = _attn(c)
    part = oracle.prefill_attention_f64(c["Q"][4:], c["K"], c["V"], 3, 6, 2, 1, 16)
    np.testing.assert_allclose(part, whole[4:], rtol=0, atol=1e-14)


def test_attention_is_invariant_to_a_shift_of_all_keys_and_to_key_order():
    # adding one vector to every key shifts all scores of a row by the same
    # amount; permuting the visible keys with their values changes nothing
    T, pos0, d = 1, 9, 8
    c = synth.attention_case(T, pos0, 1, 1, d, seed=10)
    # keys on a 1/64 grid and a shift of whole 1/64 steps, so that the shifted
    # keys are exact in f32
    c["K"] = (np.round(c["K"] * 64) / 64).astype(np.float32)
    base = _attn(c)
    shift = (np.arange(d, dtype=np.float32) - 3) / 64
    shifted = _attn(c, K=c["K"] + shift[None, :])
    assert np.array_equal((c["K"] + shift).astype(np.float64), c["K"].astype(np.float64) + shift)
    np.testing.assert_allclose(shifted, base, rtol=1e-12, atol=1e-13)
    perm = np.random.default_rng(0).permutation(pos0 + T)
    np.testing.assert_allclose(_attn(c, K=c["K"][perm], V=c["V"][perm]), base, rtol=1e-12, atol=1e-13)


def test_attention_dominant_key_takes_all_the_weight():
    # one key aligned with the query and far longer than the others: its
    # weight is 1 - O(exp(-200)), so the output is its value
    T, pos0, d = 1, 7, 16
    c = synth.attention_case(T, pos0, 1, 1, d, seed=11)
    K = c["K"] * 0.01
    K[3] = c["Q"][0] / np.linalg.norm(c["Q"][0]) * (200.0 * 4 / np.linalg.norm(c["Q"][0]))
    out = _attn(c, K=K)
    np.testing.assert_allclose(out[0], c["V"][3].astype(np.float64), rtol=0, atol=1e-12)


def test_attention_f16_input_mode_rounds_q_k_and_v():
    c = synth.attention_case(3, 1, 2, 1, 8, seed=12)
    r = lambda a: a.astype(np.float16).astype(np.float32)  # noqa: E731
    np.testing.assert_array_equal(
        oracle.prefill_attention_f16_inputs_f64(c["Q"], c["K"], c["V"], 3, 1, 2, 1, 8),
        oracle.prefill_attention_f64(r(c["Q"]), r(c["K"]), r(c["V"]), 3, 1, 2, 1, 8))


def test_attention_sampled_rows_equal_the_full_result():
    # the full-size GPU tests compare sampled rows: computing only those rows
    # (fewer keys gathered) must give exactly the full computation's rows
    c = synth.attention_case(9, 4, 4, 2, 8, seed=13)
    full = _attn(c)
    rows = np.array([8, 0, 3, 3, 5])
    np.testing.assert_allclose(_attn(c, rows=rows), full[rows], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- fp16-input modes
# The fp16-input modes round X (or q, k, v) and the decoded weight to fp16,
# round to nearest even, then compute exactly. Pinned by hand-rounded values
# (which fix fp16 rather than bf16, and nearest-even rather than truncation),
# and by equality with the float64 oracle when every operand is already an
# fp16 value (the modes may then change nothing).
def _q4_block(d_bits, nibbles):
    """One Q4_0 block, element j's nibble nibbles[j] (j < 32)."""
    b = bytearray(struct.pack("<H", d_bits))
    b += bytes((nibbles[j] & 0xF) | ((nibbles[j + 16] & 0xF) << 4) for j in range(16))
    return np.frombuffer(bytes(b), dtype=np.uint8).reshape(1, 18)


ONE_PLUS = 1.0 + 2.0 ** -11 + 2.0 ** -20   # fp16: 1 + 2^-10 (bf16 and truncation give 1)


@pytest.mark.parametrize("x,want", [
    (ONE_PLUS, 1.0 + 2.0 ** -10),
    (1.0 + 2.0 ** -11, 1.0),                  # tie, the even neighbour is 1
    (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),  # tie, the even neighbour is above
    (-ONE_PLUS, -(1.0 + 2.0 ** -10)),
])
def test_f16_mode_rounds_x_to_nearest_even_fp16(x, want):
    W = _q4_block(0x3C00, [9] + [8] * 31)     # d = 1, w_0 = 1, the rest 0
    X = np.zeros((1, 32), np.float32)
    X[0, 0] = x
    assert oracle.qgemm_f16_inputs_f64(synth.Q4_0, W, 1, 32, X)[0, 0] == want


def test_f16_mode_rounds_the_decoded_weight():
    # d = 1 + 2^-10 (0x3C01), nibble 11 (q' = 3): w = 3 + 3 * 2^-10 lies halfway
    # between the fp16 values 3 + 2^-9 (odd mantissa 513) and 3 + 2^-8 (even,
    # 514); nearest even gives 3 + 2^-8. The residual is added unrounded.
    W = _q4_block(0x3C01, [11] + [8] * 31)
    X = np.zeros((1, 32), np.float32)
    X[0, 0] = 1.0
    R = np.array([[2.0 ** -30]], np.float32)
    assert oracle.qgemm_f16_inputs_f64(synth.Q4_0, W, 1, 32, X)[0, 0] == 3.0 + 2.0 ** -8
    assert oracle.qgemm_f64(synth.Q4_0, W, 1, 32, X)[0, 0] == 3.0 + 3 * 2.0 ** -10
    assert oracle.qgemm_f16_inputs_f64(synth.Q4_0, W, 1, 32, X, R)[0, 0] == 3.0 + 2.0 ** -8 + 2.0 ** -30


def _fp16_exact_case(seed, n, k, T):
    """Q4_0 weights whose decoded values are fp16 values (scales with at most 7
    significant bits times codes of at most 4) and fp16-valued activations."""
    rng = np.random.default_rng(seed)
    raw = rng.integers(0, 256, size=(n, k // 32, 18), dtype=np.uint8)
    man = (rng.integers(0, 8, size=(n, k // 32)) << 7).astype(np.uint16)  # 3 fraction bits
    exp = rng.integers(5, 20, size=(n, k // 32)).astype(np.uint16)
    sign = rng.integers(0, 2, size=(n, k // 32)).astype(np.uint16)
    bits = (sign << 15) | (exp << 10) | man
    raw[..., 0] = (bits & 0xFF).astype(np.uint8)
    raw[..., 1] = (bits >> 8).astype(np.uint8)
    X = synth.activations(T, k, seed + 1).astype(np.float16).astype(np.float32)
    return raw.reshape(n, -1), X


def test_f16_mode_equals_the_exact_oracle_on_fp16_operands():
    n, k, T = 6, 128, 4
    W, X = _fp16_exact_case(31, n, k, T)
    Wf = oracle.dequant_f64(synth.Q4_0, W, n, k)
    assert np.array_equal(Wf, Wf.astype(np.float16).astype(np.float64))  # the case is what it claims
    R = synth.activations(T, n, 33)
    np.testing.assert_array_equal(oracle.qgemm_f16_inputs_f64(synth.Q4_0, W, n, k, X, R),
                                  oracle.qgemm_f64(synth.Q4_0, W, n, k, X, R))
    W2, _ = _fp16_exact_case(32, n, k, T)
    np.testing.assert_array_equal(oracle.gate_up_swiglu_f16_inputs_f64(synth.Q4_0, W, W2, n, k, X),
                                  oracle.gate_up_swiglu_f64(synth.Q4_0, W, W2, n, k, X))
    # and a perturbation below fp16's resolution changes nothing in the mode
    Xp = (X.astype(np.float64) * (1.0 + 2.0 ** -14)).astype(np.float32)
    np.testing.assert_array_equal(oracle.qgemm_f16_inputs_f64(synth.Q4_0, W, n, k, Xp),
                                  oracle.qgemm_f64(synth.Q4_0, W, n, k, X))


def test_f16_swiglu_mode_hand_value():
    # gate and up both w_0 = 1; x_0 rounds to g = u = 1 + 2^-10 in fp16
    W = _q4_block(0x3C00, [9] + [8] * 31)
    X = np.zeros((1, 32), np.float32)
    X[0, 0] = ONE_PLUS
    g = 1.0 + 2.0 ** -10
    want = g / (1.0 + math.exp(-g)) * g
    got = oracle.gate_up_swiglu_f16_inputs_f64(synth.Q4_0, W, W, 1, 32, X)[0, 0]
    assert abs(got - want) <= 1e-15 * want
    x = float(np.float32(ONE_PLUS))
    unrounded = x / (1.0 + math.exp(-x)) * x
    assert abs(got - unrounded) > 1e-4  # the rounding is visible


def test_f16_attention_mode_hand_values():
    d = 4
    # one visible key (position 0): the output is fp16(v_0)
    Q = np.array([[ONE_PLUS, 0, 0, 0]], np.float32)
    K = np.array([[0.5, 0, 0, 0]], np.float32)
    V = np.array([[ONE_PLUS, -ONE_PLUS, 1.0 + 2.0 ** -11, 2.0]], np.float32)
    out = oracle.prefill_attention_f16_inputs_f64(Q, K, V, 1, 0, 1, 1, d)
    np.testing.assert_array_equal(out[0], [1.0 + 2.0 ** -10, -(1.0 + 2.0 ** -10), 1.0, 2.0])
    # two keys: k_0 = 0, k_1 = (2, 0, 0, 0); the score of key 1 is
    # fp16(q_0) * 2 / sqrt(4) = 1 + 2^-10, of key 0 zero; v_0 = 0 and
    # v_1 = (1 + 3 * 2^-11) -> 1 + 2^-9
    Q = np.array([[ONE_PLUS, 0, 0, 0]], np.float32)
    K = np.array([[0, 0, 0, 0], [2, 0, 0, 0]], np.float32)
    V = np.array([[0, 0, 0, 0], [1.0 + 3 * 2.0 ** -11, 0, 0, 0]], np.float32)
    out = oracle.prefill_attention_f16_inputs_f64(Q, K, V, 1, 1, 1, 1, d)
    s = 1.0 + 2.0 ** -10
    want = math.exp(s) / (1.0 + math.exp(s)) * (1.0 + 2.0 ** -9)
    assert abs(out[0, 0] - want) <= 1e-15 * want
    np.testing.assert_array_equal(out[0, 1:], [0.0, 0.0, 0.0])


def test_f16_attention_mode_equals_the_exact_oracle_on_fp16_operands():
    c = synth.attention_case(5, 3, 4, 2, 8, seed=14)
    r = {key: c[key].astype(np.float16).astype(np.float32) for key in ("Q", "K", "V")}
    np.testing.assert_array_equal(oracle.prefill_attention_f16_inputs_f64(r["Q"], r["K"], r["V"], 5, 3, 4, 2, 8),
                                  oracle.prefill_attention_f64(r["Q"], r["K"], r["V"], 5, 3, 4, 2, 8))


# ---------------------------------------------------------------- prefill layer
# Pinned by composition identities (zero output or down weights leave one
# sublayer), by the cache rows it must write, and by chunk splitting (a layer
# over T rows equals the same layer over two consecutive chunks, the second
# reading the cache rows the first wrote): a property of causal attention.
_LD = dict(hidden=64, inter=96, num_heads=4, num_kv_heads=2, head_dim=8)


def _layer_case(seed, T, pos0, zero_o=False, zero_d=False, qtype=synth.Q4_0):
    h, i, H, KV, d = (_LD[k] for k in ("hidden", "inter", "num_heads", "num_kv_heads", "head_dim"))
    w = lambda r, c, s, z: synth.quantize(qtype, np.zeros((r, c), np.float32) if z else  # noqa: E731
                                          synth.weight_f32(r, c, s, sigma=0.1))
    c = dict(
        X=synth.activations(T, h, seed), an=(1 + 0.3 * synth.activations(1, h, seed + 1)[0]).astype(np.float32),
        fn=(1 + 0.3 * synth.activations(1, h, seed + 2)[0]).astype(np.float32),
        Wqkv=w((H + 2 * KV) * d, h, seed + 3, False), Wo=w(h, H * d, seed + 4, zero_o),
        Wg=w(i, h, seed + 5, False), Wu=w(i, h, seed + 6, False), Wd=w(h, i, seed + 7, zero_d),
        K=synth.activations(pos0 + T + 2, KV * d, seed + 8), V=synth.activations(pos0 + T + 2, KV * d, seed + 9))
    return c


def _layer(qtype, c, pos0, X=None, K=None, V=None):
    return oracle.prefill_layer_f64(qtype, c["X"] if X is None else X, c["an"], c["fn"], 1e-5, c["Wqkv"], c["Wo"],
                                    c["Wg"], c["Wu"], c["Wd"], _LD["hidden"], _LD["inter"], _LD["num_heads"],
                                    _LD["num_kv_heads"], _LD["head_dim"], c["K"] if K is None else K,
                                    c["V"] if V is None else V, pos0)


def test_layer_with_zero_output_and_down_weights_leaves_x_and_writes_the_cache():
    T, pos0 = 5, 3
    c = _layer_case(1, T, pos0, zero_o=True, zero_d=True)
    X2, K, V = _layer(synth.Q4_0, c, pos0)
    np.testing.assert_array_equal(X2, c["X"].astype(np.float64))
    h, H, KV, d = _LD["hidden"], _LD["num_heads"], _LD["num_kv_heads"], _LD["head_dim"]
    rb = h // 32 * 18
    Wk = c["Wqkv"].reshape(-1)[H * d * rb:(H + KV) * d * rb]
    Wv = c["Wqkv"].reshape(-1)[(H + KV) * d * rb:(H + 2 * KV) * d * rb]
    k = oracle.normed_qgemm_f64(synth.Q4_0, Wk, KV * d, h, c["X"], c["an"], 1e-5)
    v = oracle.normed_qgemm_f64(synth.Q4_0, Wv, KV * d, h, c["X"], c["an"], 1e-5)
    np.testing.assert_allclose(K[pos0:pos0 + T], k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(V[pos0:pos0 + T], v, rtol=1e-12, atol=1e-12)
    # rows outside the chunk stay as they were
    np.testing.assert_array_equal(K[:pos0], c["K"][:pos0].astype(np.float64))
    np.testing.assert_array_equal(K[pos0 + T:], c["K"][pos0 + T:].astype(np.float64))
    np.testing.assert_array_equal(V[pos0 + T:], c["V"][pos0 + T:].astype(np.float64))


def test_layer_with_zero_output_weight_is_the_ffn_sublayer():
    T, pos0 = 6, 2
    c = _layer_case(2, T, pos0, zero_o=True)
    X2, _, _ = _layer(synth.Q4_0, c, pos0)
    ffn = oracle.ffn_sublayer_f64(synth.Q4_0, c["X"], c["fn"], 1e-5, c["Wg"], c["Wu"], c["Wd"], _LD["hidden"],
                                  _LD["inter"])
    np.testing.assert_allclose(X2, ffn, rtol=1e-12, atol=1e-12)


def test_layer_with_zero_down_weight_is_the_attention_sublayer():
    T, pos0 = 4, 5
    c = _layer_case(3, T, pos0, zero_d=True)
    X2, K, V = _layer(synth.Q4_0, c, pos0)
    h, H, KV, d = _LD["hidden"], _LD["num_heads"], _LD["num_kv_heads"], _LD["head_dim"]
    rb = h // 32 * 18
    q = oracle.normed_qgemm_f64(synth.Q4_0, c["Wqkv"].reshape(-1)[:H * d * rb], H * d, h, c["X"], c["an"], 1e-5)
    a = oracle.prefill_attention_f64(q, K, V, T, pos0, H, KV, d)
    want = c["X"].astype(np.float64) + a @ oracle.dequant_f64(synth.Q4_0, c["Wo"], h, H * d).T
    # prefill_attention_f64 rounds its inputs to float32 first: agreement to float32 level
    np.testing.assert_allclose(X2, want, rtol=1e-6, atol=1e-6)


def test_layer_over_two_chunks_equals_one_chunk():
    T, pos0, T1 = 7, 2, 3
    c = _layer_case(4, T, pos0)
    X_all, K_all, V_all = _layer(synth.Q4_0, c, pos0)
    X_a, K_a, V_a = _layer(synth.Q4_0, c, pos0, X=c["X"][:T1])
    X_b, K_b, V_b = _layer(synth.Q4_0, c, pos0 + T1, X=c["X"][T1:], K=K_a, V=V_a)
    np.testing.assert_allclose(np.concatenate([X_a, X_b]), X_all, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(K_b, K_all, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(V_b, V_all, rtol=1e-12, atol=1e-12)
    # and the order matters: the second chunk first (it would see stale cache rows) differs
    X_w, _, _ = _layer(synth.Q4_0, c, pos0 + T1, X=c["X"][T1:])
    assert np.max(np.abs(X_w - X_all[T1:])) > 1e-3
