"""GPU parity of the CUDA-core kernels against the float64 oracle.

Standalone dequant (bit exact), small-T GEMV (exact fp32) and the exact-fp32
FFMA GEMM, on seeded inputs spanning several tiles with ragged tails.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]


def _random_blocks(rng, qtype, n, k):
    bb = synth.block_bytes(qtype)
    raw = rng.integers(0, 256, size=(n, k // 32, bb), dtype=np.uint8)
    hi = raw[..., 1]
    raw[..., 1] = np.where((hi & 0x7C) == 0x7C, hi & 0xBF, hi)  # finite scales only
    return raw.reshape(n, -1)


# ------------------------------------------------------------------ dequant
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (256, 512), (130, 4096)])
def test_dequant_bit_exact_random_bytes(q, qtype, n, k):
    rng = np.random.default_rng(n * 7 + k + qtype)
    W = _random_blocks(rng, qtype, n, k)  # covers subnormal, negative and large scales
    out = torch.full((n, k), float("nan"), device="cuda")
    q.apr_dequant(qtype, dev(W), n, k, out)
    q.apr_stream_status()
    got = out.cpu().numpy()
    want = oracle.dequant_f32(qtype, W, n, k)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("qtype", QTYPES)
def test_dequant_bit_exact_synthetic_weight(q, qtype):
    n, k = 512, 4096
    W = synth.quantize(qtype, synth.weight_f32(n, k, seed=0))
    out = torch.empty((n, k), device="cuda")
    q.apr_dequant(qtype, dev(W), n, k, out)
    q.apr_stream_status()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32),
                                  oracle.dequant_f32(qtype, W, n, k).view(np.uint32))


def test_dequant_golden_blocks(q):
    import os

    import test_oracle_pins as pins

    for name in pins.GOLDEN_FILES:
        qtype, byts, vals = pins.load_golden(name)
        out = torch.empty((1, 32), device="cuda")
        q.apr_dequant(qtype, dev(byts), 1, 32, out)
        q.apr_stream_status()
        np.testing.assert_array_equal(out.cpu().numpy()[0].astype(np.float64), vals, err_msg=name)


# ------------------------------------------------------------------ GEMV
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 9, 13, 16])
# (300, 512): ragged 16-row groups; (10, 2304): one partial group and a partial
# 2048-column chunk; (77, 288): rows not 16-byte multiples (staged kernel)
@pytest.mark.parametrize("n,k", [(300, 512), (10, 2304), (77, 288)])
def test_gemv_exact(q, qtype, T, n, k):
    c = synth.make_case(qtype, n, k, T, residual=True, seed=T)
    buf, Y = guarded(T, n)
    q.apr_qgemv(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]))
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_exact_leg(Y.cpu().numpy(), oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("n,k", [(20000, 512), (40000, 1024)])
def test_one_token_gemv_many_rows_a_cta(q, qtype, swiglu, n, k):
    """Many rows a CTA of the one-token kernel (its row sums and residuals
    sized by that count): 20000 x 512 (under 16 MiB of weight) on one CTA an
    SM, 132 rows each; 40000 x 1024 (over) on two CTAs an SM, 132 rows each."""
    c = synth.make_case(qtype, n, k, 1, residual=not swiglu, gate_up=swiglu, seed=41)
    buf, Y = guarded(1, n)
    if swiglu:
        q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), 1, Y, Wu=dev(c["Wu"]), leg=q.APR_LEG_EXACT_F32,
                       path=q.APR_PATH_GEMV)
        ref = oracle.gate_up_swiglu_f64(qtype, c["W"], c["Wu"], n, k, c["X"])
    else:
        q.apr_qgemv(qtype, dev(c["W"]), n, k, dev(c["X"]), 1, Y, dev(c["R"]))
        ref = oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"])
    q.apr_stream_status()
    check_guards(buf, 1, n)
    assert_exact_leg(Y.cpu().numpy(), ref)


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [1, 6, 16])
def test_gemv_swiglu_exact(q, qtype, T):
    n, k = 200, 1024
    c = synth.make_case(qtype, n, k, T, gate_up=True, seed=40 + T)
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, Wu=dev(c["Wu"]), path=q.APR_PATH_GEMV)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_exact_leg(Y.cpu().numpy(), oracle.gate_up_swiglu_f64(qtype, c["W"], c["Wu"], n, k, c["X"]))


# Rows longer than a 16 KB stage of the row-streaming kernel (Q8_0 k = 16384,
# and gate/up pairs of Q4_0 rows at k = 16384) go to the chunked bulk kernel.
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [1, 5])
@pytest.mark.parametrize("swiglu", [False, True])
def test_gemv_long_rows(q, qtype, T, swiglu):
    n, k = 40, 16384
    c = synth.make_case(qtype, n, k, T, residual=not swiglu, gate_up=swiglu, seed=90 + T)
    buf, Y = guarded(T, n)
    if swiglu:
        q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, Wu=dev(c["Wu"]), path=q.APR_PATH_GEMV)
        ref = oracle.gate_up_swiglu_f64(qtype, c["W"], c["Wu"], n, k, c["X"])
    else:
        q.apr_qgemv(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]))
        ref = oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"])
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_exact_leg(Y.cpu().numpy(), ref)


# Back-to-back GEMVs on one stream, each reading the previous output as X and
# as its residual: the next call starts before the previous one finishes and
# streams its weight early, but must read X and R only after it.
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [1, 2])
def test_gemv_chain_reads_previous_output(q, qtype, T):
    n = k = 1024
    steps = 6
    cases = [synth.make_case(qtype, n, k, T, seed=300 + i) for i in range(steps)]
    Ws = [dev(c["W"]) for c in cases]
    Ys = [dev(cases[0]["X"])] + [torch.empty((T, n), device="cuda") for _ in range(steps)]
    for i in range(steps):
        q.apr_qgemv(qtype, Ws[i], n, k, Ys[i], T, Ys[i + 1], Ys[i])
    q.apr_stream_status()
    ys = [y.cpu().numpy() for y in Ys]
    for i in range(steps):
        ref = oracle.qgemm_f64(qtype, cases[i]["W"], n, k, ys[i], ys[i])
        assert_exact_leg(ys[i + 1], ref)


def test_gemv_residual_alias_accumulates(q):
    n, k, T = 256, 512, 4
    c = synth.make_case(synth.Q8_0, n, k, T, residual=True, seed=5)
    Y = dev(c["R"])
    q.apr_qgemv(synth.Q8_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, Y)   # Y += X . W^T
    q.apr_stream_status()
    assert_exact_leg(Y.cpu().numpy(), oracle.qgemm_f64(synth.Q8_0, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("T", [1, 2, 4])
def test_auto_rule_small_T_is_exact(q, T):
    # T <= APR_AUTO_GEMV_MAX_T (4) takes the GEMV, whose error is fp32-level even on the fp16 leg
    assert T <= q.APR_AUTO_GEMV_MAX_T
    n, k = 256, 512
    c = synth.make_case(synth.Q8_0, n, k, T, seed=0)
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm(synth.Q8_0, dev(c["W"]), n, k, dev(c["X"]), T, Y)
    q.apr_stream_status()
    assert_exact_leg(Y.cpu().numpy(), oracle.qgemm_f64(synth.Q8_0, c["W"], n, k, c["X"]))


# ------------------------------------------------------------------ exact GEMM
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T", [(256, 512, 17), (200, 288, 70), (130, 1024, 129)])
@pytest.mark.parametrize("res", [False, True])
def test_exact_gemm(q, qtype, n, k, T, res):
    c = synth.make_case(qtype, n, k, T, residual=res, seed=n + T)
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, residual=dev(c["R"]) if res else None,
                   leg=q.APR_LEG_EXACT_F32, path=q.APR_PATH_GEMM)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_exact_leg(Y.cpu().numpy(), oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("qtype", QTYPES)
def test_exact_gemm_swiglu(q, qtype):
    n, k, T = 192, 512, 100
    c = synth.make_case(qtype, n, k, T, gate_up=True, seed=3)
    buf, Y = guarded(T, n)
    q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, Wu=dev(c["Wu"]), leg=q.APR_LEG_EXACT_F32)
    q.apr_stream_status()
    check_guards(buf, T, n)
    assert_exact_leg(Y.cpu().numpy(), oracle.gate_up_swiglu_f64(qtype, c["W"], c["Wu"], n, k, c["X"]))


def test_f16_leg_with_k_not_multiple_of_256_runs_exact(q):
    n, k, T = 96, 288, 40
    c = synth.make_case(synth.Q4_0, n, k, T, seed=8)
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), T, Y)
    q.apr_stream_status()
    assert_exact_leg(Y.cpu().numpy(), oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"]))


def test_empty_batch_leaves_output(q):
    n, k = 64, 256
    c = synth.make_case(synth.Q4_0, n, k, 1, seed=1)
    Y = torch.full((1, n), 7.0, device="cuda")
    q.apr_qgemm(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), 0, Y)
    q.apr_qgemm(synth.Q4_0, dev(c["W"]), 0, k, dev(c["X"]), 1, Y)
    q.apr_stream_status()
    assert torch.all(Y == 7.0)


@pytest.mark.parametrize("nbytes", [16, 16400, 9437184, 28311552 + 48])
def test_read_stream_reads_and_changes_nothing(q, nbytes):
    # the GEMV's data movement alone: it runs to completion and writes nothing
    src = torch.arange(nbytes // 4, dtype=torch.int32, device="cuda")
    before = src.clone()
    q.apr_read_stream(src, nbytes)
    assert q.apr_stream_status() == q.APR_OK
    assert torch.equal(src, before)
