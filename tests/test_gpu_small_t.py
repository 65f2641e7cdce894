"""GPU parity of the small-T routes around the T rule.

* The tensor-core GEMM at T < 16: the library pads its fp16 copy of X to 16
  rows (a TMA tile over a tensor of fewer rows is slow); rows past T feed
  only output columns that are never stored. Checked through every entry
  that converts X itself (apr_qgemm_ex on both legs, the normed projection,
  the FFN sublayer, the allocation-free entry), with outputs guarded by
  canaries so that a stored padding column would show.
* The GEMV path: Q8_0 at T = 8 on k = 4096 (the bulk kernel's two-stage ring),
  and shapes no streaming GEMV kernel takes (long rows with T >= 3), which run
  on the exact leg's tensor-core GEMM.
Bars as everywhere: fp16 leg rel-Frobenius <= 2e-3 and max|err| <= 1e-2 rms,
exact routes rel-Frobenius <= 1e-5, against the float64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]


def _ex(q, qtype, c, n, k, T, **kw):
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, residual=None if c["R"] is None else dev(c["R"]),
                   **kw)
    q.apr_stream_status()
    check_guards(buf, T, n)
    return Y.cpu().numpy()


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [1, 2, 5, 9, 15, 16])
def test_tensor_core_gemm_below_sixteen_rows(q, qtype, T):
    n, k = 384, 1024
    c = synth.make_case(qtype, n, k, T, residual=True, seed=T)
    y = _ex(q, qtype, c, n, k, T, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    assert_f16_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))
    y = _ex(q, qtype, c, n, k, T, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM)
    assert_exact_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("T", [3, 12])
def test_gate_up_below_sixteen_rows(q, T):
    n, k = 256, 512
    c = synth.make_case(synth.Q4_0, n, k, T, gate_up=True, seed=40 + T)
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, Wu=dev(c["Wu"]), path=q.APR_PATH_GEMM)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.gate_up_swiglu_f64(synth.Q4_0, c["W"], c["Wu"], n, k, c["X"]))


@pytest.mark.parametrize("T", [5, 11])
def test_normed_projection_and_ffn_below_sixteen_rows(q, T):
    # above APR_AUTO_GEMV_MAX_T the normed projection and the FFN take the
    # tensor-core route with the norm writing fp16 rows (padded to 16)
    n, k = 300, 512
    c = synth.make_case(synth.Q8_0, n, k, T, residual=True, seed=50 + T)
    w = (1.0 + 0.5 * synth.activations(1, k, 51)[0]).astype(np.float32)
    buf, Y = guarded(T, n)
    q.apr_qgemm_rmsnorm(synth.Q8_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(w), 1e-6, residual=dev(c["R"]))
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.normed_qgemm_f64(synth.Q8_0, c["W"], n, k, c["X"], w, 1e-6, c["R"]))
    hidden, inter = 256, 512
    Ws = [synth.quantize(synth.Q4_0, synth.weight_f32(r, cc, 60 + i))
          for i, (r, cc) in enumerate(((inter, hidden), (inter, hidden), (hidden, inter)))]
    X = synth.activations(T, hidden, 63)
    wn = (1.0 + 0.5 * synth.activations(1, hidden, 64)[0]).astype(np.float32)
    Xd = dev(X)
    q.apr_ffn_sublayer(synth.Q4_0, *[dev(Wi) for Wi in Ws], hidden, inter, T, dev(wn), 1e-6, Xd)
    q.apr_stream_status()
    ref = oracle.ffn_sublayer_f64(synth.Q4_0, X, wn, 1e-6, Ws[0], Ws[1], Ws[2], hidden, inter)
    x0 = X.astype(np.float64)
    assert_f16_leg(Xd.cpu().numpy() - x0, ref - x0)


@pytest.mark.parametrize("T", [1, 7])
def test_noalloc_below_sixteen_rows(q, T):
    n, k = 300, 512
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=70 + T)
    buf, Y = guarded(T, n)
    q.apr_qgemm_noalloc(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]))
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T", [(4096, 4096, 8), (1000, 4096, 7), (300, 12288, 5), (300, 12288, 3),
                                   (200, 16384, 2)])
def test_gemv_path_shapes(q, qtype, n, k, T):
    # (4096, 4096, 8): the bulk kernel with eight tokens (Q8_0: two-stage
    # ring); k = 12288 with T = 5: no streaming kernel takes the X table, the
    # exact tensor-core GEMM runs; T = 3 there: the tensor-core GEMV
    c = synth.make_case(qtype, n, k, T, residual=True, seed=n + T)
    buf, Y = guarded(T, n)
    q.apr_qgemv(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]))
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_exact_leg(Y.cpu().numpy(), oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))
