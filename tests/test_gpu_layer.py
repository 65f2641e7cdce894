"""GPU parity of the chunked prefill layer (apr_prefill_layer) against the
float64 oracle's layer (norm, q/k/v with k and v written into the cache,
causal attention, output projection + residual, FFN sublayer).

Bars: the layer's update of X (X_out - X) and the cache rows it writes are held
to the fp16-leg bar (relative Frobenius 2e-3, max |err| <= 1e-2 rms) on the
fp16 leg; on the exact leg the cache rows (plain projections) to the exact bar
and the update of X to the fp16 bar, since the attention takes fp16 inputs on
both legs. Cache rows outside the chunk must be untouched, bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, dev

pytestmark = pytest.mark.gpu


def _case(qtype, hidden, inter, H, KV, T, pos0, seed, extra=3):
    d = 256
    r = np.random.default_rng(seed)
    return dict(
        qtype=qtype, hidden=hidden, inter=inter, H=H, KV=KV, T=T, pos0=pos0,
        Wqkv=synth.quantize(qtype, synth.weight_f32((H + 2 * KV) * d, hidden, seed)),
        Wo=synth.quantize(qtype, synth.weight_f32(hidden, H * d, seed + 1)),
        Wg=synth.quantize(qtype, synth.weight_f32(inter, hidden, seed + 2)),
        Wu=synth.quantize(qtype, synth.weight_f32(inter, hidden, seed + 3)),
        Wd=synth.quantize(qtype, synth.weight_f32(hidden, inter, seed + 4)),
        X=synth.activations(T, hidden, seed + 5),
        an=(1.0 + 0.2 * r.standard_normal(hidden)).astype(np.float32),
        fn=(1.0 + 0.2 * r.standard_normal(hidden)).astype(np.float32),
        K=synth.activations(pos0 + T + extra, KV * d, seed + 6),
        V=synth.activations(pos0 + T + extra, KV * d, seed + 7))


def _run(q, c, leg=0, chunk=0):
    X, K, V = dev(c["X"]), dev(c["K"]), dev(c["V"])
    q.apr_prefill_layer(c["qtype"], dev(c["Wqkv"]), dev(c["Wo"]), dev(c["Wg"]), dev(c["Wu"]), dev(c["Wd"]),
                        c["hidden"], c["inter"], c["H"], c["KV"], c["T"], c["pos0"], dev(c["an"]), dev(c["fn"]),
                        1e-6, X, K, V, leg=leg, chunk=chunk)
    q.apr_stream_status()
    return X.cpu().numpy(), K.cpu().numpy(), V.cpu().numpy()


def _ref(c):
    return oracle.prefill_layer_f64(c["qtype"], c["X"], c["an"], c["fn"], 1e-6, c["Wqkv"], c["Wo"], c["Wg"],
                                    c["Wu"], c["Wd"], c["hidden"], c["inter"], c["H"], c["KV"], 256, c["K"], c["V"],
                                    c["pos0"])


def _check(c, got, leg):
    X, K, V = got
    rX, rK, rV = _ref(c)
    p0, T = c["pos0"], c["T"]
    x0 = c["X"].astype(np.float64)
    assert_f16_leg(X - x0, rX - x0)
    cache_bar = assert_f16_leg if leg == 0 else assert_exact_leg
    cache_bar(K[p0:p0 + T], rK[p0:p0 + T])
    cache_bar(V[p0:p0 + T], rV[p0:p0 + T])
    for got_c, given in ((K, c["K"]), (V, c["V"])):
        np.testing.assert_array_equal(got_c[:p0], given[:p0])
        np.testing.assert_array_equal(got_c[p0 + T:], given[p0 + T:])


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("leg", [0, 1])
def test_layer_small_chunks(q, qtype, leg):
    # chunks of 16, 16 and 8 rows: the small-T routes (GEMV) for every projection
    c = _case(qtype, 256, 512, 2, 1, 40, 7, seed=1)
    _check(c, _run(q, c, leg=leg, chunk=16), leg)


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("leg", [0, 1])
def test_layer_one_chunk(q, qtype, leg):
    # one chunk of 200 rows: the tensor-core routes on the fp16 leg
    c = _case(qtype, 512, 768, 4, 2, 200, 0, seed=2)
    _check(c, _run(q, c, leg=leg), leg)


def test_layer_chunking_agrees(q):
    c = _case(synth.Q4_0, 512, 768, 4, 2, 300, 33, seed=3)
    a = _run(q, c, chunk=0)
    b = _run(q, c, chunk=128)  # 128, 128, 44 rows
    _check(c, b, 0)
    x0 = c["X"].astype(np.float64)
    assert_f16_leg(b[0] - x0, a[0].astype(np.float64) - x0)


def test_layer_qkv_on_192_token_tiles(q):
    # 16 query heads over 4 KV heads (a 6144-row fused qkv weight) at 512
    # rows: the qkv GEMM takes 192-token tiles and its epilogue sends the q,
    # k and v rows to their places by row range
    c = _case(synth.Q4_0, 512, 1024, 16, 4, 512, 0, seed=5)
    _check(c, _run(q, c), 0)


def test_layer_nine_b_shape(q):
    # hidden 4096, intermediate 12288, 16 query heads over 4 KV heads, 128 rows
    # after 64 cached positions
    c = _case(synth.Q4_0, 4096, 12288, 16, 4, 128, 64, seed=4)
    _check(c, _run(q, c), 0)


def test_layer_empty_chunk_writes_nothing(q):
    c = _case(synth.Q4_0, 256, 512, 2, 1, 8, 4, seed=5)
    c0 = dict(c, T=0)
    X, K, V = dev(c["X"]), dev(c["K"]), dev(c["V"])
    q.apr_prefill_layer(c["qtype"], dev(c["Wqkv"]), dev(c["Wo"]), dev(c["Wg"]), dev(c["Wu"]), dev(c["Wd"]),
                        c0["hidden"], c0["inter"], c0["H"], c0["KV"], 0, c0["pos0"], dev(c["an"]), dev(c["fn"]),
                        1e-6, X, K, V)
    q.apr_stream_status()
    np.testing.assert_array_equal(X.cpu().numpy(), c["X"])
    np.testing.assert_array_equal(K.cpu().numpy(), c["K"])
