"""Streams and graphs: the library's per-stream scratch.

Calls on different streams use different scratch buffers, so they may run
concurrently; a graph may be captured from a stream the library has never
seen (its scratch is allocated during the capture) and replayed.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, assert_f16_leg, dev

pytestmark = pytest.mark.gpu


def _cases():
    gemm = synth.make_case(synth.Q4_0, 1024, 2048, 300, residual=True, seed=21)
    gemv = synth.make_case(synth.Q8_0, 4096, 2048, 3, residual=True, seed=22)
    return gemm, gemv


def _refs(gemm, gemv):
    return (oracle.qgemm_f64(synth.Q4_0, gemm["W"], 1024, 2048, gemm["X"], gemm["R"]),
            oracle.qgemm_f64(synth.Q8_0, gemv["W"], 4096, 2048, gemv["X"], gemv["R"]))


def test_two_streams_run_concurrently(q):
    gemm, gemv = _cases()
    ref_gemm, ref_gemv = _refs(gemm, gemv)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for s in streams:
        with torch.cuda.stream(s):
            ins = {name: (dev(c["W"]), dev(c["X"]), dev(c["R"])) for name, c in (("gemm", gemm), ("gemv", gemv))}
            Yg = torch.empty((300, 1024), device="cuda")
            Yv = torch.empty((3, 4096), device="cuda")
            outs.append((s, ins, Yg, Yv))
    torch.cuda.synchronize()
    # interleave launches on the two streams, several rounds each
    for rnd in range(4):
        for s, ins, Yg, Yv in outs:
            W, X, R = ins["gemm"]
            q.apr_qgemm(synth.Q4_0, W, 1024, 2048, X, 300, Yg, R, stream=s)
            W, X, R = ins["gemv"]
            q.apr_qgemv(synth.Q8_0, W, 4096, 2048, X, 3, Yv, R, stream=s)
    for s, _, Yg, Yv in outs:
        q.apr_stream_status(s)
        assert_f16_leg(Yg.cpu().numpy(), ref_gemm)
        assert_exact_leg(Yv.cpu().numpy(), ref_gemv)


def test_graph_captured_on_a_new_stream(q):
    gemm, gemv = _cases()
    ref_gemm, ref_gemv = _refs(gemm, gemv)
    Wg, Xg, Rg = dev(gemm["W"]), dev(gemm["X"]), dev(gemm["R"])
    Wv, Xv, Rv = dev(gemv["W"]), dev(gemv["X"]), dev(gemv["R"])
    Yg = torch.full((300, 1024), float("nan"), device="cuda")
    Yv = torch.full((3, 4096), float("nan"), device="cuda")
    s = torch.cuda.Stream()  # no library call has used it yet
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        q.apr_qgemm(synth.Q4_0, Wg, 1024, 2048, Xg, 300, Yg, Rg, stream=s)
        q.apr_qgemv(synth.Q8_0, Wv, 4096, 2048, Xv, 3, Yv, Rv, stream=s)
    for _ in range(2):
        Yg.fill_(float("nan"))
        Yv.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_f16_leg(Yg.cpu().numpy(), ref_gemm)
        assert_exact_leg(Yv.cpu().numpy(), ref_gemv)
    q.apr_stream_status(s)


@pytest.mark.parametrize("T", [1, 64])
def test_weight_written_by_another_kernel_just_before_is_read_fresh(q, T):
    # The library's kernels read their weights before the preceding kernel on
    # the stream has finished only when that kernel is the library's own (it
    # lets them launch early); a kernel of other code (here a torch XOR that
    # turns weight A into weight B in place) always completes first, so the
    # call sees B. T = 1 runs the one-token GEMV, T = 64 the tensor-core GEMM.
    n, k = 1024, 2048
    a = synth.make_case(synth.Q4_0, n, k, T, seed=31)
    b = synth.make_case(synth.Q4_0, n, k, T, seed=32)
    W = dev(a["W"])
    flip = dev(np.bitwise_xor(a["W"], b["W"]))
    X = dev(b["X"])
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm(synth.Q4_0, W, n, k, X, T, Y)   # reads A
    W.bitwise_xor_(flip)                         # A -> B on the same stream
    q.apr_qgemm(synth.Q4_0, W, n, k, X, T, Y)   # must read B
    q.apr_stream_status()
    ref = oracle.qgemm_f64(synth.Q4_0, b["W"], n, k, b["X"])
    if T == 1:
        assert_exact_leg(Y.cpu().numpy(), ref)
    else:
        assert_f16_leg(Y.cpu().numpy(), ref)
