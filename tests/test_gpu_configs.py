"""Parity at the full sizes of the benchmarked workloads, in the launch
configuration the bench uses, against the float64 oracle (full outputs: the
oracle's matrix product is a BLAS call, so every element is checked).

Workloads: the Q8_0 256 x 512 problem with 16 tokens; the Q4_0 4096 x 4096
GEMM + residual at T = 512; the fused gate/up SwiGLU 12288 x 4096 then the
down projection 4096 x 12288 + residual at T = 512 (Q4_0 and Q8_0); the
small-T GEMV sweep; and the projections of a 9B-class layer at T = 512 and
2048 on both legs.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, check_guards, dev, errors, guarded

pytestmark = pytest.mark.gpu


def run(q, case, *, leg=0, path=0, Wu=None):
    n, k, T = case["n"], case["k"], case["T"]
    buf, Y = guarded(T, n)
    R = dev(case["R"]) if case.get("R") is not None else None
    q.apr_qgemm_ex(case["qtype"], dev(case["W"]), n, k, dev(case["X"]), T, Y, residual=R,
                   Wu=dev(Wu) if Wu is not None else None, leg=leg, path=path)
    q.apr_stream_status()
    check_guards(buf, T, n)
    return Y


def test_q8_0_256x512_t16(q):
    c = synth.make_case(synth.Q8_0, 256, 512, 16, seed=0)
    ref = oracle.qgemm_f64(synth.Q8_0, c["W"], 256, 512, c["X"])
    assert_f16_leg(run(q, c).cpu().numpy(), ref)                         # T rule: the fp16 GEMM from T = 8
    assert_exact_leg(run(q, c, path=q.APR_PATH_GEMV).cpu().numpy(), ref)  # the GEMV path (exact)
    assert_f16_leg(run(q, c, path=q.APR_PATH_GEMM).cpu().numpy(), ref)     # forced tcgen05 GEMM
    assert_exact_leg(run(q, c, leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM).cpu().numpy(), ref)


def test_q4_0_4096x4096_t512_residual(q):
    c = synth.make_case(synth.Q4_0, 4096, 4096, 512, residual=True, seed=0)
    ref = oracle.qgemm_f64(synth.Q4_0, c["W"], 4096, 4096, c["X"], c["R"])
    y = run(q, c).cpu().numpy()
    rel, mx = assert_f16_leg(y, ref)
    rel16, _, _ = errors(y, oracle.qgemm_f16_inputs_f64(synth.Q4_0, c["W"], 4096, 4096, c["X"], c["R"]))
    assert rel16 <= 2e-5
    print(f"q4_0 4096^2 T=512 +R: rel {rel:.2e} max/rms {mx:.2e} vs fp16-input oracle {rel16:.2e}")


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_swiglu_then_down_t512(q, qtype):
    T = 512
    up = synth.make_case(qtype, 12288, 4096, T, gate_up=True, seed=0)
    g_ref = oracle.gate_up_swiglu_f64(qtype, up["W"], up["Wu"], 12288, 4096, up["X"])
    h_gpu = run(q, up, Wu=up["Wu"])
    rel, mx = assert_f16_leg(h_gpu.cpu().numpy(), g_ref)
    print(f"swiglu qtype {qtype}: rel {rel:.2e} max/rms {mx:.2e}")
    # down projection + residual, fed (a) the GPU's SwiGLU output, (b) the oracle's
    Wd = synth.quantize(qtype, synth.weight_f32(4096, 12288, seed=4))
    R = synth.activations(T, 4096, 2)
    for name, h in (("gpu", h_gpu.cpu().numpy()), ("oracle", g_ref.astype(np.float32))):
        case = dict(qtype=qtype, n=4096, k=12288, T=T, W=Wd, X=h, R=R)
        y = run(q, case).cpu().numpy()
        rel, mx = assert_f16_leg(y, oracle.qgemm_f64(qtype, Wd, 4096, 12288, h, R))
        print(f"down qtype {qtype} fed by {name}: rel {rel:.2e} max/rms {mx:.2e}")
    # chained end-to-end error of the pair (reported)
    chain_ref = oracle.qgemm_f64(qtype, Wd, 4096, 12288, g_ref.astype(np.float32), R)
    y = run(q, dict(qtype=qtype, n=4096, k=12288, T=T, W=Wd, X=h_gpu.cpu().numpy(), R=R)).cpu().numpy()
    rel, mx, _ = errors(y, chain_ref)
    print(f"chained swiglu->down qtype {qtype}: rel {rel:.2e}")
    assert rel <= 2 * 2e-3


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("n,k", [(4096, 4096), (12288, 4096)])
def test_gemv_sweep(q, qtype, n, k):
    W = synth.quantize(qtype, synth.weight_f32(n, k, seed=0))
    for T in (1, 2, 4, 8, 16):
        X = synth.activations(T, k, 1)
        case = dict(qtype=qtype, n=n, k=k, T=T, W=W, X=X)
        y = run(q, case, path=q.APR_PATH_GEMV).cpu().numpy()
        assert_exact_leg(y, oracle.qgemm_f64(qtype, W, n, k, X))


LAYER = [("qkv", 6144, 4096, False), ("out", 4096, 4096, True), ("gate_up", 12288, 4096, None),
         ("down", 4096, 12288, True)]


@pytest.mark.parametrize("T", [512, 2048])
@pytest.mark.parametrize("leg", [0, 1])
def test_9b_class_layer(q, T, leg):
    for i, (name, n, k, res) in enumerate(LAYER):
        c = synth.make_case(synth.Q4_0, n, k, T, residual=bool(res), gate_up=res is None, seed=10 * i)
        if res is None:
            ref = oracle.gate_up_swiglu_f64(synth.Q4_0, c["W"], c["Wu"], n, k, c["X"])
            y = run(q, c, leg=leg, Wu=c["Wu"]).cpu().numpy()
        else:
            ref = oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"], c["R"])
            y = run(q, c, leg=leg).cpu().numpy()
        if leg == 0:
            rel, mx = assert_f16_leg(y, ref)
        else:
            rel = assert_exact_leg(y, ref)
        print(f"layer T={T} leg={leg} {name}: rel {rel:.2e}")
