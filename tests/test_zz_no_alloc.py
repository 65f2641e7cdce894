"""The allocation-free GEMM entry point, apr_qgemm_noalloc, on the GPU.

Some callers cannot allocate device memory once they run (a server that has
reserved nearly all HBM for weights and its KV-cache arena, or a runtime that
allocates only at start-up). For them apr_qgemm_noalloc runs the same
tensor-core GEMM as apr_qgemm, with its fp16 copy of the activations in a
fixed scratch array instead of a pooled allocation. This file is collected
last: it checks two calls in a row against the pooled entry point (and the
float64 oracle), through the C ABI, and the size limit.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_f16_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu


def _noalloc(q, qtype, W, n, k, X, T, Y, R):
    stream = torch.cuda.current_stream().cuda_stream
    return q.library().apr_qgemm_noalloc(qtype, W.data_ptr(), n, k, X.data_ptr(), T, Y.data_ptr(),
                                         R.data_ptr() if R is not None else None, stream)


def test_noalloc_matches_pooled_entry_on_two_calls_in_a_row(q):
    n, k, T = 384, 1024, 200
    cases = [synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=71),
             synth.make_case(synth.Q8_0, n, k, T - 37, residual=False, seed=72)]
    for c in cases:
        Tc = c["T"]
        W, X = dev(c["W"]), dev(c["X"])
        R = dev(c["R"]) if c["R"] is not None else None
        buf, Y = guarded(Tc, n)
        assert _noalloc(q, c["qtype"], W, n, k, X, Tc, Y, R) == 0, q.apr_last_error()
        q.apr_stream_status()
        check_guards(buf, Tc, n)
        Yp = torch.empty((Tc, n), device="cuda")
        q.apr_qgemm_ex(c["qtype"], W, n, k, X, Tc, Yp, residual=R, path=q.APR_PATH_GEMM)
        q.apr_stream_status()
        y = Y.cpu().numpy()
        assert_f16_leg(y, Yp.cpu().numpy().astype(np.float64))
        assert_f16_leg(y, oracle.qgemm_f64(c["qtype"], c["W"], n, k, c["X"], c["R"]))


def test_noalloc_allocates_nothing_on_a_new_stream(q):
    """On a stream the library has not seen, a call of the pooled entry point
    with 4096 x 8192 activations allocates its 64 MiB fp16 scratch (free
    device memory drops: the measurement sees an allocation; small ones may
    come from memory the driver already holds), while apr_qgemm_noalloc leaves
    free memory as it was, on its first call on a new stream and on the next."""
    n, k, T = 256, 1024, 200
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=73)
    W, X, R = dev(c["W"]), dev(c["X"]), dev(c["R"])
    Y = torch.empty((T, n), device="cuda")
    cb = synth.make_case(synth.Q4_0, 128, 8192, 4096, seed=75)
    Wb, Xb = dev(cb["W"]), dev(cb["X"])
    Yb = torch.empty((4096, 128), device="cuda")
    # the kernels' modules are loaded by a first call (lazy module loading)
    assert _noalloc(q, synth.Q4_0, W, n, k, X, T, Y, R) == 0, q.apr_last_error()
    q.apr_qgemm(synth.Q4_0, Wb, 128, 8192, Xb, 4096, Yb)
    q.apr_stream_status()
    s_pooled, s_fixed = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s_pooled):
        q.apr_qgemm(synth.Q4_0, Wb, 128, 8192, Xb, 4096, Yb, stream=s_pooled)
    q.apr_stream_status(s_pooled)
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 <= free0 - 64 * 2**20, "the pooled call on a new stream should have allocated its scratch"
    with torch.cuda.stream(s_fixed):
        for _ in range(2):
            assert _noalloc(q, synth.Q4_0, W, n, k, X, T, Y, R) == 0, q.apr_last_error()
    q.apr_stream_status(s_fixed)
    assert torch.cuda.mem_get_info()[0] == free1
    assert_f16_leg(Y.cpu().numpy(), oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"], c["R"]))


def test_noalloc_at_its_size_limit(q):
    """T * k exactly APR_NOALLOC_MAX_TK: every element of the fixed array is used."""
    n, k = 256, 4096
    T = q.APR_NOALLOC_MAX_TK // k
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=74)
    W, X, R = dev(c["W"]), dev(c["X"]), dev(c["R"])
    buf, Y = guarded(T, n)
    assert _noalloc(q, synth.Q4_0, W, n, k, X, T, Y, R) == 0, q.apr_last_error()
    q.apr_stream_status()
    check_guards(buf, T, n)
    Yp = torch.empty((T, n), device="cuda")
    q.apr_qgemm_ex(synth.Q4_0, W, n, k, X, T, Yp, residual=R, path=q.APR_PATH_GEMM)
    q.apr_stream_status()
    y = Y.cpu().numpy()
    assert_f16_leg(y, Yp.cpu().numpy().astype(np.float64))
    assert_f16_leg(y, oracle.qgemm_f64(synth.Q4_0, c["W"], n, k, c["X"], c["R"]))


def test_noalloc_rejects_sizes_beyond_its_scratch(q):
    k = 4096
    T = q.APR_NOALLOC_MAX_TK // k + 1
    lib = q.library()
    A = 1 << 20  # never dereferenced: the size check comes first
    assert lib.apr_qgemm_noalloc(2, A, 64, k, 2 * A, T, 64 * A, None, None) == q.APR_E_INVAL
    assert "fixed scratch" in q.apr_last_error()
    assert lib.apr_qgemm_noalloc(2, A, 64, 288, 2 * A, 16, 64 * A, None, None) == q.APR_E_INVAL
