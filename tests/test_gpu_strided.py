"""GPU parity of the strided-output form (ldy) on every kernel path.

Row t of Y (and of the residual) sits ldy floats after row t - 1, so Y can be
a column slice of a wider buffer: a fused QKV output, or the gate half of a
gate/up buffer. Each case fills the whole buffer with a canary, runs one path
through apr_qgemm_ex, checks the written columns against the float64 oracle
and checks that the ldy - n columns between rows, and the guard after the last
row, still hold the canary.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import CANARY_BITS, assert_exact_leg, assert_f16_leg, dev

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]
TAIL = 64  # canary floats after the last row's n outputs


def strided(T, n, ldy, fill=None):
    """A canary-filled [T][ldy] buffer (plus a tail) and its [T][n] view."""
    buf = torch.full((T * ldy + TAIL,), CANARY_BITS, dtype=torch.int32, device="cuda")
    view = buf[:T * ldy].view(torch.float32).view(T, ldy)[:, :n]
    if fill is not None:
        view.copy_(torch.from_numpy(np.ascontiguousarray(fill)).cuda())
    return buf, view


def check_gaps(buf, T, n, ldy):
    b = buf.cpu().numpy()
    rows = b[:T * ldy].reshape(T, ldy)
    assert np.all(rows[:, n:] == CANARY_BITS), "write between rows"
    assert np.all(b[T * ldy:] == CANARY_BITS), "write after the last row"


def run(q, qtype, c, n, k, T, ldy, *, leg, path, residual=False, swiglu=False, accumulate=False):
    X = dev(c["X"])
    W = dev(c["W"])
    Wu = dev(c["Wu"]) if swiglu else None
    R = c["R"] if residual else None
    rbuf = rview = None
    if accumulate:
        buf, Y = strided(T, n, ldy, fill=R)
        rview = Y
    else:
        buf, Y = strided(T, n, ldy)
        if residual:
            rbuf, rview = strided(T, n, ldy, fill=R)
    q.apr_qgemm_ex(qtype, W, n, k, X, T, Y, residual=rview, Wu=Wu, leg=leg, path=path, ldy=ldy)
    q.apr_stream_status()
    check_gaps(buf, T, n, ldy)
    if rbuf is not None:
        check_gaps(rbuf, T, n, ldy)  # the residual is read only
        np.testing.assert_array_equal(rview.cpu().numpy(), R)
    y = Y.cpu().numpy()
    if swiglu:
        ref = oracle.gate_up_swiglu_f64(qtype, c["W"], c["Wu"], n, k, c["X"])
    else:
        ref = oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], R)
    return y, ref


# ------------------------------------------------------------------ tensor-core GEMM
# (n, k, T, ldy): TMA stores need n and ldy multiples of 4, else the epilogue
# stores directly; (512, 2048, 300) takes the split-K cluster plan
GEMM_CASES = [
    (256, 512, 200, 260),     # TMA store, two token tiles
    (256, 512, 200, 257),     # direct store, odd row stride
    (300, 768, 129, 306),     # TMA store, ragged 128-row tile
    (302, 768, 129, 305),     # n % 4 != 0: direct store
    (512, 2048, 300, 520),    # split K, TMA store
    (512, 2048, 300, 517),    # split K, direct store
]


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T,ldy", GEMM_CASES)
@pytest.mark.parametrize("residual", [False, True])
def test_gemm_strided(q, qtype, n, k, T, ldy, residual):
    c = synth.make_case(qtype, n, k, T, residual=residual, seed=n + ldy + T)
    y, ref = run(q, qtype, c, n, k, T, ldy, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM, residual=residual)
    assert_f16_leg(y, ref)


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("ldy", [264, 259])
def test_gemm_swiglu_strided(q, qtype, ldy):
    n, k, T = 256, 512, 140
    c = synth.make_case(qtype, n, k, T, gate_up=True, seed=ldy)
    y, ref = run(q, qtype, c, n, k, T, ldy, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM, swiglu=True)
    assert_f16_leg(y, ref)


@pytest.mark.parametrize("ldy", [520, 517])
def test_gemm_strided_accumulate(q, ldy):
    """Y == residual, both strided: Y[t] += X[t] W^T in place."""
    n, k, T = 512, 2048, 300
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=ldy)
    y, ref = run(q, synth.Q4_0, c, n, k, T, ldy, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM, residual=True,
                 accumulate=True)
    assert_f16_leg(y, ref)


# ------------------------------------------------------------------ GEMV (exact fp32)
# T = 1, 2 at k % 256 == 0: the integer-dot kernel; T = 5 and 13: chunked
# bulk kernel (up to 8) and the staged kernel (k = 288, or T > 8)
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T,ldy", [(300, 512, 1, 301), (300, 512, 2, 307), (300, 512, 5, 303), (77, 288, 5, 80),
                                       (10, 2304, 13, 17)])
def test_gemv_strided(q, qtype, n, k, T, ldy):
    c = synth.make_case(qtype, n, k, T, residual=True, seed=T + ldy)
    y, ref = run(q, qtype, c, n, k, T, ldy, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMV, residual=True)
    assert_exact_leg(y, ref)


@pytest.mark.parametrize("T", [1, 2, 3])
def test_gemv_swiglu_strided(q, T):
    n, k = 300, 1024
    c = synth.make_case(synth.Q8_0, n, k, T, gate_up=True, seed=T)
    y, ref = run(q, synth.Q8_0, c, n, k, T, 2 * n, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMV, swiglu=True)
    assert_exact_leg(y, ref)


@pytest.mark.parametrize("T", [2, 4])
def test_gemv_strided_accumulate(q, T):
    n, k = 300, 512
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=5)
    y, ref = run(q, synth.Q4_0, c, n, k, T, 333, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMV, residual=True,
                 accumulate=True)
    assert_exact_leg(y, ref)


# ------------------------------------------------------------------ exact-fp32 GEMM
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("swiglu", [False, True])
def test_exact_gemm_strided(q, qtype, swiglu):
    n, k, T, ldy = 200, 768, 70, 211
    c = synth.make_case(qtype, n, k, T, residual=not swiglu, gate_up=swiglu, seed=7)
    y, ref = run(q, qtype, c, n, k, T, ldy, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM, residual=not swiglu,
                 swiglu=swiglu)
    assert_exact_leg(y, ref)


def test_ldy_equal_n_matches_contiguous(q):
    """ldy == n is the contiguous layout: bit-identical to ldy = 0."""
    n, k, T = 256, 512, 200
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=3)
    Y0 = torch.empty((T, n), device="cuda")
    Y1 = torch.empty((T, n), device="cuda")
    for Y, ldy in ((Y0, 0), (Y1, n)):
        q.apr_qgemm_ex(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, residual=dev(c["R"]), ldy=ldy)
    q.apr_stream_status()
    assert torch.equal(Y0.view(torch.int32), Y1.view(torch.int32))
