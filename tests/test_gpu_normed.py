"""GPU parity of the normed projection (apr_qgemm_rmsnorm) against the
float64 oracle: apr_qgemm_ex on RMSNorm(X), on every route (the fp16 leg's
tensor-core GEMM reading the fp16 rows the norm writes, the GEMV, the exact
leg), with a residual, the gate/up form, a strided Y and two chunks of rows."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, dev

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]
EPS = 1e-5


def norm_weight(k, seed):
    return (1.0 + 0.1 * synth.activations(1, k, seed)[0]).astype(np.float32)


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T,leg", [(1000, 2048, 300, 0), (256, 512, 3, 0), (384, 768, 40, 1)])
def test_normed_projection(q, qtype, n, k, T, leg):
    c = synth.make_case(qtype, n, k, T, residual=True, seed=n + T)
    w = norm_weight(k, T)
    Y = torch.full((T, n), float("nan"), device="cuda")
    q.apr_qgemm_rmsnorm(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(w), EPS, residual=dev(c["R"]), leg=leg)
    q.apr_stream_status()
    ref = oracle.normed_qgemm_f64(qtype, c["W"], n, k, c["X"], w, EPS, c["R"])
    if leg == 0 and T > q.APR_AUTO_GEMV_MAX_T:
        assert_f16_leg(Y.cpu().numpy(), ref)
    else:
        assert_exact_leg(Y.cpu().numpy(), ref)


@pytest.mark.parametrize("qtype", QTYPES)
def test_normed_gate_up(q, qtype):
    n, k, T = 768, 1024, 129
    c = synth.make_case(qtype, n, k, T, gate_up=True, seed=3)
    w = norm_weight(k, 4)
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm_rmsnorm(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(w), EPS, Wu=dev(c["Wu"]))
    q.apr_stream_status()
    assert_f16_leg(Y.cpu().numpy(), oracle.normed_qgemm_f64(qtype, c["W"], n, k, c["X"], w, EPS, Wu=c["Wu"]))


def test_normed_strided_output(q):
    n, k, T, ldy = 512, 1024, 200, 520
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=5)
    w = norm_weight(k, 6)
    buf = torch.full((T, ldy), -7.0, device="cuda")
    rbuf = torch.zeros((T, ldy), device="cuda")
    rbuf[:, :n] = dev(c["R"])
    q.apr_qgemm_rmsnorm(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), T, buf[:, :n], dev(w), EPS,
                        residual=rbuf[:, :n], ldy=ldy)
    q.apr_stream_status()
    out = buf.cpu().numpy()
    assert np.all(out[:, n:] == -7.0)
    assert_f16_leg(out[:, :n], oracle.normed_qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"], w, EPS, c["R"]))


def test_normed_two_chunks(q):
    n, k = 256, 256
    T = q.APR_FFN_CHUNK_ROWS + 5
    c = synth.make_case(synth.Q8_0, n, k, T, seed=7)
    w = norm_weight(k, 8)
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm_rmsnorm(synth.Q8_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(w), EPS)
    q.apr_stream_status()
    assert_f16_leg(Y.cpu().numpy(), oracle.normed_qgemm_f64(synth.Q8_0, c["W"], n, k, c["X"], w, EPS))
