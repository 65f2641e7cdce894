"""GPU parity of the FFN sublayer (apr_ffn_sublayer) against the float64 oracle.

X += down(silu(h . Wg^T) * (h . Wu^T)), h = RMSNorm(X) (the pages' batched FFN
phase). Every route is covered: the fp16 leg on the tensor cores (the norm
written as fp16 in the same pass), the small-T GEMV route, the exact-fp32 leg,
sizes that take the FFMA kernels, and T that spans two chunks of rows. The
tolerance is the one of the leg, on the whole updated X.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, dev

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]
EPS = 1e-6


def case(qtype, hidden, inter, T, seed):
    X = synth.activations(T, hidden, seed)
    w = (1.0 + 0.1 * synth.activations(1, hidden, seed + 1)[0]).astype(np.float32)
    Wg = synth.quantize(qtype, synth.weight_f32(inter, hidden, seed + 2))
    Wu = synth.quantize(qtype, synth.weight_f32(inter, hidden, seed + 3))
    Wd = synth.quantize(qtype, synth.weight_f32(hidden, inter, seed + 4))
    return X, w, Wg, Wu, Wd


def run(q, qtype, hidden, inter, T, leg, seed):
    X, w, Wg, Wu, Wd = case(qtype, hidden, inter, T, seed)
    Xd = dev(X)
    q.apr_ffn_sublayer(qtype, dev(Wg), dev(Wu), dev(Wd), hidden, inter, T, dev(w), EPS, Xd, leg=leg)
    q.apr_stream_status()
    ref = oracle.ffn_sublayer_f64(qtype, X, w, EPS, Wg, Wu, Wd, hidden, inter)
    return Xd.cpu().numpy(), ref, X


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [17, 300, 512])
def test_ffn_f16_tensor_cores(q, qtype, T):
    y, ref, X = run(q, qtype, 1024, 2816, T, q.APR_LEG_F16, seed=T)
    assert_f16_leg(y, ref)
    # the update alone, as a diagnostic bar: twice the leg's relative bound
    d, dref = y.astype(np.float64) - X, ref - X
    assert np.linalg.norm(d - dref) / np.linalg.norm(dref) <= 4e-3


@pytest.mark.parametrize("qtype", QTYPES)
def test_ffn_small_T_runs_exact(q, qtype):
    # T <= 16 takes the GEMV, which is exact to fp32 level on either leg
    y, ref, _ = run(q, qtype, 1024, 2816, 3, q.APR_LEG_F16, seed=5)
    assert_exact_leg(y, ref)


@pytest.mark.parametrize("qtype", QTYPES)
def test_ffn_exact_leg(q, qtype):
    y, ref, _ = run(q, qtype, 512, 768, 40, q.APR_LEG_EXACT_F32, seed=6)
    assert_exact_leg(y, ref)


def test_ffn_sizes_off_the_tensor_core_grid(q):
    # hidden and inter not multiples of 256: the FFMA GEMM, exact
    y, ref, _ = run(q, synth.Q4_0, 288, 544, 50, q.APR_LEG_F16, seed=7)
    assert_exact_leg(y, ref)


def test_ffn_two_chunks(q):
    T = q.APR_FFN_CHUNK_ROWS + 37
    y, ref, _ = run(q, synth.Q8_0, 256, 512, T, q.APR_LEG_F16, seed=8)
    assert_f16_leg(y, ref)


def test_ffn_9b_shape_t512(q):
    """The 9B-class FFN (hidden 4096, intermediate 12288, Q4_0) at T = 512."""
    y, ref, _ = run(q, synth.Q4_0, 4096, 12288, 512, q.APR_LEG_F16, seed=9)
    assert_f16_leg(y, ref)


def test_ffn_zero_norm_weight_leaves_x(q):
    hidden, inter, T = 512, 1024, 64
    X, _, Wg, Wu, Wd = case(synth.Q4_0, hidden, inter, T, 10)
    Xd = dev(X)
    q.apr_ffn_sublayer(synth.Q4_0, dev(Wg), dev(Wu), dev(Wd), hidden, inter, T,
                       torch.zeros(hidden, device="cuda"), EPS, Xd)
    q.apr_stream_status()
    np.testing.assert_array_equal(Xd.cpu().numpy(), X)
