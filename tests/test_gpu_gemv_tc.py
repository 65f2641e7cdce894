"""GPU parity of the tensor-core GEMV against the float64 oracle.

The library takes it for T = 3 and 4, and for T = 2 on weights of at least
2^25 elements (k % 256 == 0, no gate/up); the other small-T calls run the
CUDA-core kernels, which the CUDA-core tests cover.

The kernel multiplies exact fp16 integer codes by three fp16 pieces of X,
scaled by a power of two per token and 256 columns, so its error must stay at
fp32 level (the exact-leg bar) whatever the magnitudes of X. The cases cover
tiles shared by many CTAs (long rows), grids smaller than the SM count, ragged
row tiles, activations far outside the fp16 range, all-zero chunks and tokens,
and bitwise repeatability of the fixed-order combination of partial sums.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_exact_leg, check_guards, dev, guarded

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]


def gemv(q, qtype, c, n, k, T, R=None):
    buf, Y = guarded(T, n)
    q.apr_qgemv(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, None if R is None else dev(R))
    q.apr_stream_status()
    check_guards(buf, T, n)
    return Y.cpu().numpy()


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [3, 4])
# (4096, 4096): 512 chunks over the SMs, tiles shared by 4-5 CTAs;
# (1000, 12288): ragged last tile, 48 chunks a tile; (129, 2304): one row in
# the second tile; (1, 256): a one-chunk grid; (12288, 1024): more tiles
# than SMs, several whole tiles per CTA
@pytest.mark.parametrize("n,k", [(4096, 4096), (1000, 12288), (129, 2304), (1, 256), (12288, 1024)])
def test_gemv_tc(q, qtype, T, n, k):
    c = synth.make_case(qtype, n, k, T, residual=True, seed=n + k + T)
    y = gemv(q, qtype, c, n, k, T, c["R"])
    assert_exact_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))
    # the product alone (without R) is held to the same bar
    assert_exact_leg(y - c["R"], oracle.qgemm_f64(qtype, c["W"], n, k, c["X"]))


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("T", [3, 4])
def test_gemv_tc_activation_range(q, qtype, T):
    """Chunks of X at 1e4 (past the fp16 range), 1e-6 (below its normal
    range), all zero, a single nonzero value, and one token all zero."""
    n, k = 512, 2048
    c = synth.make_case(qtype, n, k, T, seed=77 + T)
    X = c["X"].copy()
    X[:, 0:256] *= 1.0e4
    X[:, 256:512] *= 1.0e-6
    X[:, 512:768] = 0.0
    X[:, 768:1024] = 0.0
    X[:, 800] = -3.0e5
    X[:, 1024:1280] *= 1.0e-30
    X[:, 1280:1344] = 1.0e-39     # subnormal floats
    X[1, :] = 0.0
    c["X"] = X
    y = gemv(q, qtype, c, n, k, T)
    ref = oracle.qgemm_f64(qtype, c["W"], n, k, X)
    assert_exact_leg(y, ref)
    assert np.all(y[1] == 0.0)


@pytest.mark.parametrize("qtype", QTYPES)
def test_gemv_tc_repeats_bitwise(q, qtype):
    n, k, T = 4096, 4096, 3
    c = synth.make_case(qtype, n, k, T, residual=True, seed=5)
    W, X, R = dev(c["W"]), dev(c["X"]), dev(c["R"])
    outs = []
    for _ in range(4):
        Y = torch.empty((T, n), device="cuda")
        q.apr_qgemv(qtype, W, n, k, X, T, Y, R)
        outs.append(Y)
    q.apr_stream_status()
    for Y in outs[1:]:
        assert torch.equal(Y.view(torch.int32), outs[0].view(torch.int32))


@pytest.mark.parametrize("qtype", QTYPES)
def test_gemv_tc_two_tokens_large_weight(q, qtype):
    """T = 2 takes the tensor-core GEMV from 2^25 weight elements on."""
    n, k, T = 8192, 4096, 2
    c = synth.make_case(qtype, n, k, T, residual=True, seed=9)
    y = gemv(q, qtype, c, n, k, T, c["R"])
    assert_exact_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


def test_gemv_tc_full_size_sampled_rows(q):
    """The 12288 x 4096 Q4_0 projection at T = 3, checked on 1024 sampled
    rows (the oracle runs on those rows of W only)."""
    n, k, T = 12288, 4096, 3
    c = synth.make_case(synth.Q4_0, n, k, T, seed=0)
    y = gemv(q, synth.Q4_0, c, n, k, T)
    rows = np.random.default_rng(1).choice(n, size=1024, replace=False)
    ref = oracle.qgemm_f64(synth.Q4_0, c["W"][rows], len(rows), k, c["X"])
    assert_exact_leg(y[:, rows], ref)
