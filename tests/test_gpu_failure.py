"""Failure detection on the GPU, without a fault.

Every wait of the library's kernels on an mbarrier is bounded: when it runs
out, the kernel records a timeout in the device status word, leaves its loops,
drains its own copies and MMAs and returns. apr_test_bounded_wait makes such a
wait run out on purpose (a barrier nothing arrives on, a 2 ms limit); the test
checks that the status reads APR_E_TIMEOUT once, that the kernel really waited
for its limit, and that the library's calls on the same stream are correct
afterwards: the tensor-core GEMV (whose ticket counters are cleared after a
reported timeout), the tensor-core GEMM and the whole-row GEMV.
"""

import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, dev

pytestmark = pytest.mark.gpu


def _checks_after(q, s):
    n, k = 512, 1024
    for T, exact in ((3, True), (1, True), (100, False)):
        c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=90 + T)
        Y = torch.full((T, n), float("nan"), device="cuda")
        q.apr_qgemm(synth.Q4_0, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]), stream=s)
        assert q.apr_stream_status(s) == q.APR_OK
        ref = oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"], c["R"])
        (assert_exact_leg if exact else assert_f16_leg)(Y.cpu().numpy(), ref)


def test_bounded_wait_runs_out_and_the_stream_recovers(q):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _checks_after(q, s)  # the stream's scratch exists before the timeout
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        q.apr_test_bounded_wait(2000, stream=s)
        b.record(s)
        with pytest.raises(q.AprError) as err:
            q.apr_stream_status(s)
        assert err.value.status == q.APR_E_TIMEOUT
        assert a.elapsed_time(b) >= 1.5  # ms: the wait ran to its limit
        assert q.apr_stream_status(s) == q.APR_OK  # reported once, then cleared
        _checks_after(q, s)


def test_timeout_on_one_stream_leaves_another_correct(q):
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    q.apr_test_bounded_wait(1000, stream=s1)
    with pytest.raises(q.AprError) as err:
        q.apr_stream_status(s1)
    assert err.value.status == q.APR_E_TIMEOUT
    with torch.cuda.stream(s2):
        _checks_after(q, s2)


def test_weights_written_by_another_kernel_just_before_are_read_new(q):
    """The library's kernels read the weights before the preceding kernel on
    the stream has finished only when that kernel is the library's own; a
    weight written by any other kernel directly before the call is complete
    first. Here torch overwrites W on the stream right before each call."""
    n, k = 4096, 4096
    cases = [synth.make_case(synth.Q4_0, n, k, T, seed=95 + T) for T in (1, 4, 200)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Wd = torch.empty_like(dev(cases[0]["W"]))
        for c in cases:
            T = c["T"]
            src, X = dev(c["W"]), dev(c["X"])
            Y = torch.empty((T, n), device="cuda")
            Wd.zero_()
            Wd.copy_(src)  # a torch kernel on the stream, immediately before the call
            q.apr_qgemm(synth.Q4_0, Wd, n, k, X, T, Y, stream=s)
            q.apr_stream_status(s)
            ref = oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"])
            (assert_exact_leg if T <= 16 else assert_f16_leg)(Y.cpu().numpy(), ref)
