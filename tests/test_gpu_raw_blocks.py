"""GPU parity on arbitrary GGUF blocks, every route against the float64 oracle.

The quantizer of ``synth`` only ever writes Q8_0 codes in [-127, 127] and small
positive-or-negative scales near 1e-3; GGUF files may hold any code and any
finite fp16 scale. Here the weights are ``synth.random_blocks``: uniformly
random payload bytes (Q8_0 codes -128..127, every Q4_0 nibble) and scales of
both signs drawn from one exponent class per case (fp16 subnormal, small
normal, the typical range of quantized weights, large, or every exponent
mixed block by block).

Checks, per output element y[t][i] with the scale s[t][i] = sum_j |x[t][j]
w[i][j]| (+ |r[t][i]|), the sum of the magnitudes of its terms:

* exact-fp32 routes (FFMA GEMM, every GEMV kernel, the exact FFN): against the
  float64 oracle, |y - ref| <= 1e-5 s elementwise, and the whole output within
  the exact-leg bar (relative Frobenius 1e-5);
* the fp16 leg (tensor-core GEMM, gate/up, normed projection, the allocation-
  free entry): against the oracle fed the same fp16-rounded operands,
  |y - ref16| <= 3e-5 s16 elementwise (only the fp32 accumulation differs),
  and, where the decoded weights lie in fp16's normal range, the whole output
  within the fp16-leg bar against the float64 oracle. Subnormal-scale blocks
  decode to fp16 subnormals (|d q| < 2^-14), which carry fewer significant
  bits: by the definition of the fp16 leg its result then differs from the
  exact one by more than the fp16 bar, so those cases are held to the
  fp16-input oracle only. On the fp16 leg |d q| must stay within fp16's range
  (<= 65504), so the scales there are capped (``fp16_range``).

An element-wise bound scaled by the terms' magnitudes is what an fp32
accumulation guarantees for any data: it checks rows with tiny scales as
strictly as rows with large ones, which a bar on the whole output cannot.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]
CLASSES = ["subnormal", "small", "typical", "large", "mixed"]


def _scale(qtype, W, n, k, X, R=None, f16=False):
    """s[t][i] = sum_j |x w| (+ |r|), the operands rounded to fp16 if f16."""
    Wf = oracle.dequant_f32(qtype, W, n, k)
    Xf = np.asarray(X, np.float32)
    if f16:
        Wf = Wf.astype(np.float16)
        Xf = Xf.astype(np.float16)
    s = np.abs(Xf.astype(np.float64)) @ np.abs(Wf.astype(np.float64)).T
    if R is not None:
        s = s + np.abs(np.asarray(R, np.float64))
    return s


def _elementwise(y, ref, s, tol):
    y = np.asarray(y, np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    err = np.abs(y - ref)
    bad = err > tol * s
    if np.any(bad):
        t, i = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} elements past {tol} x sum|terms|; first at (t={t}, i={i}): "
                             f"y={y[t, i]!r} ref={ref[t, i]!r} scale={s[t, i]!r}")


def _check_exact(qtype, W, n, k, X, R, y):
    ref = oracle.qgemm_f64(qtype, W, n, k, X, R)
    _elementwise(y, ref, _scale(qtype, W, n, k, X, R), 1e-5)
    assert_exact_leg(y, ref)


def _check_f16(qtype, W, n, k, X, R, y, cls):
    ref16 = oracle.qgemm_f16_inputs_f64(qtype, W, n, k, X, R)
    _elementwise(y, ref16, _scale(qtype, W, n, k, X, R, f16=True), 3e-5)
    if cls != "subnormal":
        assert_f16_leg(y, oracle.qgemm_f64(qtype, W, n, k, X, R))


def _case(qtype, n, k, T, cls, seed, residual=False, fp16_range=False):
    W = synth.random_blocks(qtype, n, k, seed, cls, fp16_range=fp16_range)
    X = synth.activations(T, k, seed + 1)
    R = synth.activations(T, n, seed + 2) if residual else None
    return W, X, R


def _call(q, qtype, W, n, k, X, T, R=None, leg=0, path=0, Wu=None):
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(qtype, dev(W), n, k, dev(X), T, Y, residual=None if R is None else dev(R),
                   Wu=None if Wu is None else dev(Wu), leg=leg, path=path)
    q.apr_stream_status()
    check_guards(buf, T, n)
    return Y.cpu().numpy()


# ------------------------------------------------------------------ fp16-leg GEMM
# (256, 512, 100): 256-token tiles split over k by a 2-CTA cluster;
# (1000, 1024, 130): several row tiles, ragged tokens
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", CLASSES)
@pytest.mark.parametrize("n,k,T,res", [(256, 512, 100, True), (1000, 1024, 130, False)])
def test_tensor_core_gemm(q, qtype, cls, n, k, T, res):
    W, X, R = _case(qtype, n, k, T, cls, seed=11 * n + T, residual=res, fp16_range=True)
    y = _call(q, qtype, W, n, k, X, T, R, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    _check_f16(qtype, W, n, k, X, R, y, cls)


# the two other tile plans: 128-token tiles (80 row tiles) and unsplit
# 256-token tiles (37 x 5 tiles)
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", ["typical", "mixed"])
@pytest.mark.parametrize("n,k,T,res", [(10240, 256, 200, True), (4736, 512, 1030, False)])
def test_tensor_core_gemm_other_plans(q, qtype, cls, n, k, T, res):
    W, X, R = _case(qtype, n, k, T, cls, seed=n + T, residual=res, fp16_range=True)
    y = _call(q, qtype, W, n, k, X, T, R, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    _check_f16(qtype, W, n, k, X, R, y, cls)


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", ["subnormal", "small", "typical"])
def test_tensor_core_gate_up(q, qtype, cls):
    # gate/up values must stay in range for silu and the product; the large
    # classes would only test overflow of the SwiGLU product
    n, k, T = 384, 1024, 200
    Wg = synth.random_blocks(qtype, n, k, 5, cls, fp16_range=True)
    Wu = synth.random_blocks(qtype, n, k, 6, cls, fp16_range=True)
    X = synth.activations(T, k, 7)
    y = _call(q, qtype, Wg, n, k, X, T, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM, Wu=Wu)
    ref16 = oracle.gate_up_swiglu_f16_inputs_f64(qtype, Wg, Wu, n, k, X)
    rel16 = float(np.linalg.norm(y - ref16) / np.linalg.norm(ref16))
    assert rel16 <= 2e-5, rel16
    if cls != "subnormal":
        assert_f16_leg(y, oracle.gate_up_swiglu_f64(qtype, Wg, Wu, n, k, X))


# ------------------------------------------------------------------ exact leg
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", CLASSES)
@pytest.mark.parametrize("n,k,T,res", [(200, 288, 70, True), (130, 1024, 129, False)])
def test_exact_gemm(q, qtype, cls, n, k, T, res):
    W, X, R = _case(qtype, n, k, T, cls, seed=7 * n + T, residual=res)
    y = _call(q, qtype, W, n, k, X, T, R, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM)
    _check_exact(qtype, W, n, k, X, R, y)


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", ["small", "typical", "mixed"])
def test_exact_gate_up(q, qtype, cls):
    n, k, T = 200, 512, 40
    Wg = synth.random_blocks(qtype, n, k, 15, cls)
    Wu = synth.random_blocks(qtype, n, k, 16, cls)
    X = synth.activations(T, k, 17)
    y = _call(q, qtype, Wg, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(qtype, Wg, Wu, n, k, X))


# ------------------------------------------------------------------ GEMV routes
# T = 1, 2 at k % 256 == 0: the integer-dot kernel (Q8_0 at T = 2 on this
# small weight: the bulk kernel); T = 5, 8: bulk kernel;
# T = 3, 4: tensor cores; T = 13: staged fallback; k = 288: the staged
# fallback at every T
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", CLASSES)
@pytest.mark.parametrize("n,k,T", [(300, 512, 1), (300, 512, 2), (300, 1024, 3), (300, 1024, 4), (300, 512, 5),
                                   (300, 512, 8), (300, 512, 13), (77, 288, 1), (77, 288, 16)])
def test_gemv_routes(q, qtype, cls, n, k, T):
    W, X, R = _case(qtype, n, k, T, cls, seed=3 * n + k + T, residual=True)
    buf, Y = guarded(T, n)
    q.apr_qgemv(qtype, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_exact(qtype, W, n, k, X, R, Y.cpu().numpy())


# T = 2 on a weight of 2^25 elements: the integer-dot kernel's two-token
# form (one CTA an SM), 54 rows a CTA
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", ["subnormal", "mixed"])
def test_gemv_tensor_core_two_tokens(q, qtype, cls):
    n, k, T = 8192, 4096, 2
    W, X, R = _case(qtype, n, k, T, cls, seed=91, residual=False)
    buf, Y = guarded(T, n)
    q.apr_qgemv(qtype, dev(W), n, k, dev(X), T, Y)
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_exact(qtype, W, n, k, X, None, Y.cpu().numpy())


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("cls", ["small", "typical", "mixed"])
@pytest.mark.parametrize("T", [1, 3, 6])
def test_gemv_gate_up(q, qtype, cls, T):
    n, k = 300, 512
    Wg = synth.random_blocks(qtype, n, k, 21, cls)
    Wu = synth.random_blocks(qtype, n, k, 22, cls)
    X = synth.activations(T, k, 23)
    y = _call(q, qtype, Wg, n, k, X, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMV, Wu=Wu)
    assert_exact_leg(y, oracle.gate_up_swiglu_f64(qtype, Wg, Wu, n, k, X))


# ------------------------------------------------------------------ composites
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("leg,cls", [(0, "small"), (0, "typical"), (1, "typical"), (1, "mixed")])
def test_ffn_sublayer(q, qtype, leg, cls):
    hidden, inter, T = 256, 512, 40
    Ws = [synth.random_blocks(qtype, r, c, 30 + i, cls, fp16_range=leg == 0)
          for i, (r, c) in enumerate(((inter, hidden), (inter, hidden), (hidden, inter)))]
    X = synth.activations(T, hidden, 33)
    # on the fp16 leg the SwiGLU output is rounded to fp16 for the down
    # projection: a small norm weight keeps it inside fp16's range
    w = ((0.02 if leg == 0 else 1.0) * (1.0 + 0.5 * synth.activations(1, hidden, 34)[0])).astype(np.float32)
    Xd = dev(X)
    q.apr_ffn_sublayer(qtype, *[dev(Wi) for Wi in Ws], hidden, inter, T, dev(w), 1e-6, Xd, leg=leg)
    q.apr_stream_status()
    ref = oracle.ffn_sublayer_f64(qtype, X, w, 1e-6, Ws[0], Ws[1], Ws[2], hidden, inter)
    (assert_f16_leg if leg == 0 else assert_exact_leg)(Xd.cpu().numpy(), ref)


@pytest.mark.parametrize("qtype", QTYPES)
def test_normed_projection(q, qtype):
    n, k, T = 300, 512, 50
    W = synth.random_blocks(qtype, n, k, 41, "mixed", fp16_range=True)
    X = synth.activations(T, k, 42)
    w = (1.0 + 0.5 * synth.activations(1, k, 43)[0]).astype(np.float32)
    buf, Y = guarded(T, n)
    q.apr_qgemm_rmsnorm(qtype, dev(W), n, k, dev(X), T, Y, dev(w), 1e-6)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.normed_qgemm_f64(qtype, W, n, k, X, w, 1e-6))


@pytest.mark.parametrize("qtype", QTYPES)
def test_noalloc_entry(q, qtype):
    n, k, T = 300, 512, 64
    W, X, R = _case(qtype, n, k, T, "mixed", seed=51, residual=True, fp16_range=True)
    buf, Y = guarded(T, n)
    q.apr_qgemm_noalloc(qtype, dev(W), n, k, dev(X), T, Y, dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    _check_f16(qtype, W, n, k, X, R, Y.cpu().numpy(), "mixed")
