"""GPU parity of the 256-element superblock weights on every route, against
the float64 oracle: Q4_K and Q5_K (fp16 d and dmin, 6-bit sub-block scales
and mins, 4-bit codes, and for Q5_K a fifth code bit per element), Q6_K
(6-bit codes, an int8 scale per 16 elements, fp16 d; rows take k % 2048 ==
0) and IQ4_XS (fp16 d, 6-bit scales per 32 elements, 4-bit codes standing for
the entries of a 16-value code book; rows take k % 512 == 0); the layouts are
those read in the oracle.

Bars:
* dequant: bit exact (d sc q - dmin m rounded once to f32 on both sides;
  Q6_K's d sc (q - 32) and IQ4_XS's d (ls - 32) book[c] are exact);
* fp16 leg: against the oracle fed fp16-rounded X and weights, each element
  within 3e-5 of the sum of its terms' magnitudes, and the whole output within
  the fp16-leg bar against the float64 oracle (the kernel rounds the fp32 value
  of a weight to fp16, the oracle its exact value; they differ only where the
  fp32 value lands on an fp16 tie the exact value is not on);
* exact routes (GEMV, the exact leg's GEMM): within 1e-5 of the sum of the
  terms' magnitudes elementwise and the exact-leg bar overall.
Inputs: the seeded N(0, 0.02) weight encoded in the format, and random superblocks
(random bytes, d and dmin of both signs from one exponent class).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu



@pytest.fixture(params=[synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.IQ4_XS], ids=["q4_k", "q5_k", "q6_k", "iq4_xs"])
def qk(request):
    return request.param


def _k(qk, k):
    """k as given, or raised to a multiple of the format's row unit (Q6_K
    2048, IQ4_XS 512)."""
    unit = {synth.Q6_K: 2048, synth.IQ4_XS: 512}.get(qk, 256)
    return max(unit, -(-k // unit) * unit)

CLASSES = ["subnormal", "small", "typical", "large", "mixed"]


def _scale(qk, W, n, k, X, R=None, f16=False):
    Wf = oracle.dequant_f64(qk, W, n, k)
    Xf = np.asarray(X, np.float32)
    if f16:
        Wf = Wf.astype(np.float16).astype(np.float64)
        Xf = Xf.astype(np.float16)
    s = np.abs(Xf.astype(np.float64)) @ np.abs(Wf).T
    if R is not None:
        s = s + np.abs(np.asarray(R, np.float64))
    return s


def _elementwise(y, ref, s, tol):
    y = np.asarray(y, np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    bad = np.abs(y - ref) > tol * s
    if np.any(bad):
        t, i = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} elements past {tol} x sum|terms|; first at (t={t}, i={i}): "
                             f"y={y[t, i]!r} ref={ref[t, i]!r} scale={s[t, i]!r}")


def _check_exact(qk, W, n, k, X, R, y):
    ref = oracle.qgemm_f64(qk, W, n, k, X, R)
    _elementwise(y, ref, _scale(qk, W, n, k, X, R), 1e-5)
    assert_exact_leg(y, ref)


def _check_f16(qk, W, n, k, X, R, y, f64_bar=True):
    ref16 = oracle.qgemm_f16_inputs_f64(qk, W, n, k, X, R)
    _elementwise(y, ref16, _scale(qk, W, n, k, X, R, f16=True), 3e-5)
    if f64_bar:
        assert_f16_leg(y, oracle.qgemm_f64(qk, W, n, k, X, R))


def _synthetic(qk, n, k, T, seed, residual=False):
    c = synth.make_case(qk, n, k, T, residual=residual, seed=seed)
    return c["W"], c["X"], c["R"]


def _call(q, qk, W, n, k, X, T, R=None, leg=0, path=0, Wu=None):
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(qk, dev(W), n, k, dev(X), T, Y, residual=None if R is None else dev(R),
                   Wu=None if Wu is None else dev(Wu), leg=leg, path=path)
    q.apr_stream_status()
    check_guards(buf, T, n)
    return Y.cpu().numpy()


# ------------------------------------------------------------------ dequant
@pytest.mark.parametrize("cls", CLASSES)
@pytest.mark.parametrize("n,k", [(1, 256), (37, 768), (130, 4096)])
def test_dequant_bit_exact_random_superblocks(q, qk, cls, n, k):
    k = _k(qk, k)
    W = synth.random_blocks(qk, n, k, seed=n + k, scale_class=cls)
    out = torch.full((n, k), float("nan"), device="cuda")
    q.apr_dequant(qk, dev(W), n, k, out)
    q.apr_stream_status()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32),
                                  oracle.dequant_f32(qk, W, n, k).view(np.uint32))


def test_dequant_hand_superblocks(q, qk):
    import test_oracle_pins as pins

    if qk == synth.Q6_K:  # row 0: the int8 scales on their 16 elements; row 1: codes in element order
        sc = [1, -1, 2, -128, 127, 0, 5, -7, 64, -64, 3, 33, -100, 99, 11, -2]
        W = np.frombuffer(pins._q6_k_superblock(0x3C00, sc, [33] * 256) * 8 +
                          pins._q6_k_superblock(0x3C00, [1] * 16, [e % 64 for e in range(256)]) * 8,
                          np.uint8).reshape(2, 8 * 210).copy()
        out = torch.empty((2, 2048), device="cuda")
        q.apr_dequant(qk, dev(W), 2, 2048, out)
        q.apr_stream_status()
        got = out.cpu().numpy()
        np.testing.assert_array_equal(got[0], np.tile(np.repeat(np.array(sc, np.float32), 16), 8))
        np.testing.assert_array_equal(got[1], np.tile(np.array([e % 64 - 32 for e in range(256)], np.float32), 8))
        return
    if qk == synth.IQ4_XS:  # row 0: the scales on their sub-blocks (code 8: book 1); row 1: the book in order
        ls = [0, 63, 32, 33, 17, 48, 31, 1]
        W = np.frombuffer(pins._iq4_xs_superblock(0x3C00, ls, [8] * 256) * 2 +
                          pins._iq4_xs_superblock(0x3C00, [33] * 8, [e % 16 for e in range(256)]) * 2,
                          np.uint8).reshape(2, 2 * 136).copy()
        out = torch.empty((2, 512), device="cuda")
        q.apr_dequant(qk, dev(W), 2, 512, out)
        q.apr_stream_status()
        got = out.cpu().numpy()
        book = np.array(oracle.IQ4_NL_VALUES, np.float32)
        np.testing.assert_array_equal(got[0], np.tile(np.repeat(np.array(ls, np.float32) - 32, 32), 2))
        np.testing.assert_array_equal(got[1], np.tile(book[np.arange(256) % 16], 2))
        return
    five = qk == synth.Q5_K
    build, qmax, sbb = (pins._q5_k_superblock, 32, 176) if five else (pins._q4_k_superblock, 16, 144)
    sc = [1, 2, 3, 4, 17, 33, 48, 63]
    mn = [0, 1, 2, 3, 16, 40, 5, 62]
    a = build(0x3C00, 0x3C00, sc, mn, [1] * 256)
    b = build(0x3C00, 0x0000, [1] * 8, [0] * 8, [e % qmax for e in range(256)])
    W = np.frombuffer(a + b, np.uint8).reshape(2, sbb).copy()
    out = torch.empty((2, 256), device="cuda")
    q.apr_dequant(qk, dev(W), 2, 256, out)
    q.apr_stream_status()
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got[0], np.repeat(np.array(sc) - np.array(mn), 32).astype(np.float32))
    np.testing.assert_array_equal(got[1], np.array([e % qmax for e in range(256)], np.float32))


# ------------------------------------------------------------------ fp16-leg GEMM
@pytest.mark.parametrize("n,k,T,res", [(300, 768, 200, True), (4096, 4096, 512, True), (128, 256, 9, False),
                                       (1000, 1024, 130, False), (256, 512, 100, True)])
def test_gemm_synthetic(q, qk, n, k, T, res):
    k = _k(qk, k)
    W, X, R = _synthetic(qk, n, k, T, seed=n + T, residual=res)
    y = _call(q, qk, W, n, k, X, T, R, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    _check_f16(qk, W, n, k, X, R, y)


@pytest.mark.parametrize("cls", ["small", "typical", "large", "mixed"])
def test_gemm_random_superblocks(q, qk, cls):
    n, k, T = 300, 1024, 150
    k = _k(qk, k)
    W = synth.random_blocks(qk, n, k, 60, cls, fp16_range=True)
    X = synth.activations(T, k, 61)
    R = synth.activations(T, n, 62)
    y = _call(q, qk, W, n, k, X, T, R, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    _check_f16(qk, W, n, k, X, R, y)


def test_gate_up_swiglu(q, qk):
    n, k, T = 384, 1024, 200
    k = _k(qk, k)
    Wg = synth.quantize(qk, synth.weight_f32(n, k, 5))
    Wu = synth.quantize(qk, synth.weight_f32(n, k, 6))
    X = synth.activations(T, k, 7)
    buf, Y = guarded(T, n)
    q.apr_qgemm_gate_up_swiglu(qk, dev(Wg), dev(Wu), n, k, dev(X), T, Y)
    q.apr_stream_status()
    check_guards(buf, T, n)
    y = Y.cpu().numpy()
    ref16 = oracle.gate_up_swiglu_f16_inputs_f64(qk, Wg, Wu, n, k, X)
    assert float(np.linalg.norm(y - ref16) / np.linalg.norm(ref16)) <= 2e-5
    assert_f16_leg(y, oracle.gate_up_swiglu_f64(qk, Wg, Wu, n, k, X))


def test_f16_input_entry_and_noalloc(q, qk):
    n, k, T = 300, 512, 64
    k = _k(qk, k)
    W, X, R = _synthetic(qk, n, k, T, seed=9, residual=True)
    X16 = torch.empty((T, k), dtype=torch.float16, device="cuda")
    q.apr_convert_f32_to_f16(dev(X), T * k, X16)
    buf, Y = guarded(T, n)
    q.apr_qgemm_f16_in(qk, dev(W), n, k, X16, T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_f16(qk, W, n, k, X, R, Y.cpu().numpy())
    buf, Y = guarded(T, n)
    q.apr_qgemm_noalloc(qk, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_f16(qk, W, n, k, X, R, Y.cpu().numpy())


# ------------------------------------------------------------------ exact routes
@pytest.mark.parametrize("cls", CLASSES)
@pytest.mark.parametrize("n,k,T,res", [(130, 1024, 129, True), (200, 512, 40, False)])
def test_exact_gemm(q, qk, cls, n, k, T, res):
    k = _k(qk, k)
    W = synth.random_blocks(qk, n, k, 7 * n + T, cls)
    X = synth.activations(T, k, 8)
    R = synth.activations(T, n, 9) if res else None
    y = _call(q, qk, W, n, k, X, T, R, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM)
    _check_exact(qk, W, n, k, X, R, y)


def test_exact_gate_up(q, qk):
    n, k, T = 200, 512, 40
    k = _k(qk, k)
    Wg = synth.random_blocks(qk, n, k, 15, "typical")
    Wu = synth.random_blocks(qk, n, k, 16, "typical")
    X = synth.activations(T, k, 17)
    y = _call(q, qk, Wg, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(qk, Wg, Wu, n, k, X))


# T <= 8: the Q4_K GEMV; T = 13: the exact tensor-core GEMM
@pytest.mark.parametrize("cls", ["subnormal", "typical", "large", "mixed"])
@pytest.mark.parametrize("n,k,T", [(300, 512, 1), (300, 512, 2), (300, 1024, 4), (300, 512, 8), (300, 512, 13),
                                   (77, 256, 1), (64, 12288, 3),
                                   (77, 512, 3), (1, 256, 5)])
def test_gemv(q, qk, cls, n, k, T):
    k = _k(qk, k)
    W = synth.random_blocks(qk, n, k, 3 * n + k + T, cls)
    X = synth.activations(T, k, 5)
    R = synth.activations(T, n, 6)
    buf, Y = guarded(T, n)
    q.apr_qgemv(qk, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_exact(qk, W, n, k, X, R, Y.cpu().numpy())


@pytest.mark.parametrize("n,k", [(300, 12288), (20000, 2048), (40000, 1024)])
def test_one_token_gemv_large_shapes(q, qk, n, k):
    """T = 1 with long rows (one Q6_K row a stage at k = 12288), a gate/up
    pair, and many rows a CTA on two CTAs an SM (20000 x 2048 and 40000 x
    1024: over 16 MiB of weight in every format)."""
    k = _k(qk, k)
    W = synth.random_blocks(qk, n, k, 11 + n, "typical")
    X = synth.activations(1, k, 12)
    R = synth.activations(1, n, 13)
    buf, Y = guarded(1, n)
    q.apr_qgemv(qk, dev(W), n, k, dev(X), 1, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, 1, n)
    _check_exact(qk, W, n, k, X, R, Y.cpu().numpy())
    if n <= 300:
        Wu = synth.random_blocks(qk, n, k, 17 + n, "typical")
        y = _call(q, qk, W, n, k, X, 1, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMV, Wu=Wu)
        assert_exact_leg(y, oracle.gate_up_swiglu_f64(qk, W, Wu, n, k, X))


@pytest.mark.parametrize("T", [2, 3, 6])
def test_gemv_gate_up_odd_rows(q, qk, T):
    """Gate/up on the GEMV path with an odd row count: the last warp's second
    row lies past n (its loads repeat row n - 1, nothing is stored for it)."""
    n, k = 77, _k(qk, 512)
    Wg = synth.random_blocks(qk, n, k, 21 + T, "typical")
    Wu = synth.random_blocks(qk, n, k, 22 + T, "typical")
    X = synth.activations(T, k, 23)
    y = _call(q, qk, Wg, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMV, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(qk, Wg, Wu, n, k, X))


@pytest.mark.parametrize("T", [1, 4, 7])
def test_auto_rule_and_gemv_gate_up(q, qk, T):
    n, k = 4096, 4096
    W, X, R = _synthetic(qk, n, k, T, seed=T, residual=True)
    buf, Y = guarded(T, n)
    q.apr_qgemm(qk, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    (_check_exact if T <= q.APR_AUTO_GEMV_MAX_T else _check_f16)(qk, W, n, k, X, R, Y.cpu().numpy())
    Wu = synth.quantize(qk, synth.weight_f32(n, k, 100 + T))
    y = _call(q, qk, W, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMV, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(qk, W, Wu, n, k, X))


# ------------------------------------------------------------------ composites
@pytest.mark.parametrize("leg,T", [(0, 40), (1, 40), (0, 3), (1, 3)])
def test_ffn_sublayer(q, qk, leg, T):
    hidden, inter = _k(qk, 256), _k(qk, 512)
    Ws = [synth.quantize(qk, synth.weight_f32(r, c, 30 + i))
          for i, (r, c) in enumerate(((inter, hidden), (inter, hidden), (hidden, inter)))]
    X = synth.activations(T, hidden, 33)
    w = (1.0 + 0.5 * synth.activations(1, hidden, 34)[0]).astype(np.float32)
    Xd = dev(X)
    q.apr_ffn_sublayer(qk, *[dev(Wi) for Wi in Ws], hidden, inter, T, dev(w), 1e-6, Xd, leg=leg)
    q.apr_stream_status()
    ref = oracle.ffn_sublayer_f64(qk, X, w, 1e-6, Ws[0], Ws[1], Ws[2], hidden, inter)
    x0 = X.astype(np.float64)
    (assert_f16_leg if leg == 0 else assert_exact_leg)(Xd.cpu().numpy() - x0, ref - x0)


def test_normed_projection(q, qk):
    n, k, T = 300, 512, 50
    k = _k(qk, k)
    W = synth.random_blocks(qk, n, k, 41, "typical")
    X = synth.activations(T, k, 42)
    w = (1.0 + 0.5 * synth.activations(1, k, 43)[0]).astype(np.float32)
    buf, Y = guarded(T, n)
    q.apr_qgemm_rmsnorm(qk, dev(W), n, k, dev(X), T, Y, dev(w), 1e-6)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.normed_qgemm_f64(qk, W, n, k, X, w, 1e-6))


@pytest.mark.parametrize("leg", [0, 1])
def test_prefill_layer(q, qk, leg):
    import test_gpu_layer as lay

    if qk == synth.Q6_K:  # hidden, inter and 8 heads x 256 multiples of 2048
        c = lay._case(qk, 2048, 2048, 8, 2, 100, 37, seed=71)
    else:
        c = lay._case(qk, 512, 1024, 4, 2, 200, 37, seed=71)
    lay._check(c, lay._run(q, c, leg=leg, chunk=128), leg)
