"""GPU parity of F16 weights (each weight its own little-endian IEEE binary16
value) on every route, against the float64 oracle.

The format is the F16 arm of aprender-serve 0.70.2
src/cuda/executor/gdn_prefill_ops.rs (``qwen35_dequant_f32``) and its test
``f16_weight_dequantizes_on_the_device``. Bars:

* dequant: bit exact (every finite half widens exactly to f32);
* fp16 leg: the weights enter the tensor cores unrounded, only X is rounded to
  fp16, so against the oracle fed the fp16-rounded X each element is within
  3e-5 of the sum of its terms' magnitudes (only the fp32 accumulation
  differs), and the whole output within the fp16-leg bar against the float64
  oracle;
* exact routes (GEMV, the exact leg's GEMMs, the FFMA GEMM): within 1e-5 of
  the sum of the terms' magnitudes elementwise and the exact-leg bar overall.

Inputs: the seeded N(0, 0.02) weight rounded to F16 (``synth.quantize_f16``),
and random finite halves of every exponent class (``synth.random_blocks``).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu

F16 = synth.F16
CLASSES = ["subnormal", "small", "typical", "large", "mixed"]


def _scale(W, n, k, X, R=None, f16=False):
    Wf = oracle.dequant_f64(F16, W, n, k)
    Xf = np.asarray(X, np.float32)
    if f16:
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


def _check_exact(W, n, k, X, R, y):
    ref = oracle.qgemm_f64(F16, W, n, k, X, R)
    _elementwise(y, ref, _scale(W, n, k, X, R), 1e-5)
    assert_exact_leg(y, ref)


def _check_f16(W, n, k, X, R, y):
    ref16 = oracle.qgemm_f16_inputs_f64(F16, W, n, k, X, R)
    _elementwise(y, ref16, _scale(W, n, k, X, R, f16=True), 3e-5)
    assert_f16_leg(y, oracle.qgemm_f64(F16, W, n, k, X, R))


def _synthetic(n, k, T, seed, residual=False):
    c = synth.make_case(F16, n, k, T, residual=residual, seed=seed)
    return c["W"], c["X"], c["R"]


def _call(q, W, n, k, X, T, R=None, leg=0, path=0, Wu=None):
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(F16, dev(W), n, k, dev(X), T, Y, residual=None if R is None else dev(R),
                   Wu=None if Wu is None else dev(Wu), leg=leg, path=path)
    q.apr_stream_status()
    check_guards(buf, T, n)
    return Y.cpu().numpy()


# ------------------------------------------------------------------ dequant
def test_dequant_the_pages_values(q):
    n, k = 2, 64
    want = np.array([i * 0.5 - 16.0 for i in range(n * k)], np.float32).reshape(n, k)
    W = synth.quantize_f16(want)
    out = torch.full((n, k), float("nan"), device="cuda")
    q.apr_dequant(F16, dev(W), n, k, out)
    q.apr_stream_status()
    np.testing.assert_array_equal(out.cpu().numpy(), want)


def test_dequant_every_finite_half(q):
    # all 63,488 finite bit patterns (exponent field 0 .. 30), as 62 rows of 1024
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 10) & 0x1F) != 31]
    n, k = 62, 1024
    W = np.ascontiguousarray(bits.astype("<u2")).view(np.uint8).reshape(n, 2 * k)
    out = torch.full((n, k), float("nan"), device="cuda")
    q.apr_dequant(F16, dev(W), n, k, out)
    q.apr_stream_status()
    got = out.cpu().numpy()
    want = oracle.dequant_f32(F16, W, n, k)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequant_at_an_odd_two_byte_offset(q):
    # the standalone dequant takes any 2-byte aligned F16 weight
    n, k = 5, 96
    W = synth.random_blocks(F16, n, k, seed=4)
    buf = torch.zeros(W.size + 16, dtype=torch.uint8, device="cuda")
    buf[2:2 + W.size] = dev(W.reshape(-1))
    out = torch.empty((n, k), device="cuda")
    q.apr_dequant(F16, buf[2:], n, k, out)
    q.apr_stream_status()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32),
                                  oracle.dequant_f32(F16, W, n, k).view(np.uint32))


# ------------------------------------------------------------------ fp16-leg GEMM
# (300, 768, 200): three row tiles (the last ragged), three 256-k chunks, two
# token tiles (the last ragged); (4096, 4096, 512): the full-size projection;
# (128, 256, 9): one tile, one chunk
@pytest.mark.parametrize("n,k,T,res", [(300, 768, 200, True), (4096, 4096, 512, True), (128, 256, 9, False),
                                       (1000, 1024, 130, False)])
def test_gemm_synthetic(q, n, k, T, res):
    W, X, R = _synthetic(n, k, T, seed=n + T, residual=res)
    y = _call(q, W, n, k, X, T, R, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    _check_f16(W, n, k, X, R, y)


@pytest.mark.parametrize("cls", CLASSES)
def test_gemm_random_halves(q, cls):
    n, k, T = 300, 1024, 150
    W = synth.random_blocks(F16, n, k, 60, cls)
    X = synth.activations(T, k, 61)
    R = synth.activations(T, n, 62)
    y = _call(q, W, n, k, X, T, R, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    _check_f16(W, n, k, X, R, y)


def test_gemm_auto_rule_and_accumulate(q):
    # T = 8 on AUTO takes the fp16-leg GEMM; Y == residual accumulates
    n, k, T = 256, 512, 8
    W, X, R = _synthetic(n, k, T, seed=3, residual=True)
    Y = dev(R)
    q.apr_qgemm(F16, dev(W), n, k, dev(X), T, Y, Y)
    q.apr_stream_status()
    _check_f16(W, n, k, X, R, Y.cpu().numpy())


@pytest.mark.parametrize("n,k,T", [(384, 1024, 200), (12288, 4096, 64)])
def test_gate_up_swiglu(q, n, k, T):
    Wg = synth.quantize_f16(synth.weight_f32(n, k, 5))
    Wu = synth.quantize_f16(synth.weight_f32(n, k, 6))
    X = synth.activations(T, k, 7)
    buf, Y = guarded(T, n)
    q.apr_qgemm_gate_up_swiglu(F16, dev(Wg), dev(Wu), n, k, dev(X), T, Y)
    q.apr_stream_status()
    check_guards(buf, T, n)
    y = Y.cpu().numpy()
    ref16 = oracle.gate_up_swiglu_f16_inputs_f64(F16, Wg, Wu, n, k, X)
    assert float(np.linalg.norm(y - ref16) / np.linalg.norm(ref16)) <= 2e-5
    assert_f16_leg(y, oracle.gate_up_swiglu_f64(F16, Wg, Wu, n, k, X))


def test_f16_input_entry_and_noalloc(q):
    n, k, T = 300, 512, 64
    W, X, R = _synthetic(n, k, T, seed=9, residual=True)
    X16 = torch.empty((T, k), dtype=torch.float16, device="cuda")
    q.apr_convert_f32_to_f16(dev(X), T * k, X16)
    buf, Y = guarded(T, n)
    q.apr_qgemm_f16_in(F16, dev(W), n, k, X16, T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_f16(W, n, k, X, R, Y.cpu().numpy())
    buf, Y = guarded(T, n)
    q.apr_qgemm_noalloc(F16, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_f16(W, n, k, X, R, Y.cpu().numpy())


# ------------------------------------------------------------------ exact routes
# (130, 1024, 129): the exact leg on the tensor cores (ragged tiles);
# (200, 288, 70): k % 256 != 0, the FFMA GEMM
@pytest.mark.parametrize("cls", CLASSES)
@pytest.mark.parametrize("n,k,T,res", [(130, 1024, 129, True), (200, 288, 70, False)])
def test_exact_gemm(q, cls, n, k, T, res):
    W = synth.random_blocks(F16, n, k, 7 * n + T, cls)
    X = synth.activations(T, k, 8)
    R = synth.activations(T, n, 9) if res else None
    y = _call(q, W, n, k, X, T, R, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM)
    _check_exact(W, n, k, X, R, y)


def test_exact_gemm_full_size(q):
    n, k, T = 4096, 4096, 512
    W, X, R = _synthetic(n, k, T, seed=0, residual=True)
    y = _call(q, W, n, k, X, T, R, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM)
    assert_exact_leg(y, oracle.qgemm_f64(F16, W, n, k, X, R))


def test_exact_gate_up(q):
    n, k, T = 200, 512, 40
    Wg = synth.random_blocks(F16, n, k, 15, "typical")
    Wu = synth.random_blocks(F16, n, k, 16, "typical")
    X = synth.activations(T, k, 17)
    y = _call(q, Wg, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(F16, Wg, Wu, n, k, X))


# T <= 8: the staged CUDA-core GEMV; 9 <= T <= 16 at k % 256 == 0: the exact
# tensor-core GEMM; k = 288: the staged GEMV at every T
@pytest.mark.parametrize("cls", ["subnormal", "typical", "large", "mixed"])
@pytest.mark.parametrize("n,k,T", [(300, 512, 1), (300, 512, 2), (300, 1024, 4), (300, 512, 8), (300, 512, 13),
                                   (77, 288, 1), (77, 288, 16), (77, 512, 3), (1, 256, 5)])
def test_gemv(q, cls, n, k, T):
    W = synth.random_blocks(F16, n, k, 3 * n + k + T, cls)
    X = synth.activations(T, k, 5)
    R = synth.activations(T, n, 6)
    buf, Y = guarded(T, n)
    q.apr_qgemv(F16, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_exact(W, n, k, X, R, Y.cpu().numpy())


@pytest.mark.parametrize("T", [2, 3, 6])
def test_gemv_gate_up_odd_rows(q, T):
    """Gate/up on the streaming GEMV with an odd row count: the last warp's
    second row lies past n (its loads repeat row n - 1, nothing is stored for it)."""
    n, k = 77, 512
    Wg = synth.random_blocks(F16, n, k, 21 + T, "typical")
    Wu = synth.random_blocks(F16, n, k, 22 + T, "typical")
    X = synth.activations(T, k, 23)
    y = _call(q, Wg, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMV, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(F16, Wg, Wu, n, k, X))


@pytest.mark.parametrize("T", [1, 3, 4, 7])
def test_auto_rule_and_gemv_gate_up(q, T):
    # AUTO: the exact GEMV up to APR_AUTO_GEMV_MAX_T tokens, the fp16-leg GEMM above
    n, k = 4096, 4096
    W, X, R = _synthetic(n, k, T, seed=T, residual=True)
    buf, Y = guarded(T, n)
    q.apr_qgemm(F16, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    (_check_exact if T <= q.APR_AUTO_GEMV_MAX_T else _check_f16)(W, n, k, X, R, Y.cpu().numpy())
    Wu = synth.quantize_f16(synth.weight_f32(n, k, 100 + T))
    y = _call(q, W, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMV, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(F16, W, Wu, n, k, X))


# ------------------------------------------------------------------ composites
@pytest.mark.parametrize("leg,T", [(0, 40), (1, 40), (0, 3), (1, 3)])
def test_ffn_sublayer(q, leg, T):
    hidden, inter = 256, 512
    Ws = [synth.quantize_f16(synth.weight_f32(r, c, 30 + i))
          for i, (r, c) in enumerate(((inter, hidden), (inter, hidden), (hidden, inter)))]
    X = synth.activations(T, hidden, 33)
    w = (1.0 + 0.5 * synth.activations(1, hidden, 34)[0]).astype(np.float32)
    Xd = dev(X)
    q.apr_ffn_sublayer(F16, *[dev(Wi) for Wi in Ws], hidden, inter, T, dev(w), 1e-6, Xd, leg=leg)
    q.apr_stream_status()
    ref = oracle.ffn_sublayer_f64(F16, X, w, 1e-6, Ws[0], Ws[1], Ws[2], hidden, inter)
    got = Xd.cpu().numpy()
    x0 = X.astype(np.float64)
    (assert_f16_leg if leg == 0 else assert_exact_leg)(got - x0, ref - x0)


def test_normed_projection(q):
    n, k, T = 300, 512, 50
    W = synth.random_blocks(F16, n, k, 41, "typical")
    X = synth.activations(T, k, 42)
    w = (1.0 + 0.5 * synth.activations(1, k, 43)[0]).astype(np.float32)
    buf, Y = guarded(T, n)
    q.apr_qgemm_rmsnorm(F16, dev(W), n, k, dev(X), T, Y, dev(w), 1e-6)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.normed_qgemm_f64(F16, W, n, k, X, w, 1e-6))


@pytest.mark.parametrize("leg", [0, 1])
def test_prefill_layer(q, leg):
    import test_gpu_layer as lay

    c = lay._case(F16, 512, 1024, 4, 2, 200, 37, seed=71)
    lay._check(c, lay._run(q, c, leg=leg, chunk=128), leg)
