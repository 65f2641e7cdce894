"""GPU parity of the tcgen05 fp16-input GEMM against the float64 oracle.

Shapes span several 128-row tiles and 128-token tiles with ragged tails; the
epilogues are plain, residual (also Y == residual, the accumulate form) and
fused gate/up SwiGLU; invariants that hold exactly are checked bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_f16_leg, check_guards, dev, errors, guarded

pytestmark = pytest.mark.gpu

QTYPES = [synth.Q4_0, synth.Q8_0]
SHAPES = [(256, 512, 17), (128, 256, 128), (384, 1024, 200), (300, 768, 129), (1000, 2048, 513)]


def gemm(q, qtype, W, n, k, X, T, Y, R=None, Wu=None):
    q.apr_qgemm_ex(qtype, W, n, k, X, T, Y, residual=R, Wu=Wu, leg=q.APR_LEG_F16, path=q.APR_PATH_GEMM)
    q.apr_stream_status()


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T", SHAPES)
def test_plain(q, qtype, n, k, T):
    c = synth.make_case(qtype, n, k, T, seed=n + k + T)
    buf, Y = guarded(T, n)
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y)
    check_guards(buf, T, n)
    y = Y.cpu().numpy()
    assert_f16_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"]))
    # tighter: against the oracle fed the same fp16-rounded operands, only the
    # fp32 accumulation differs
    rel, _, _ = errors(y, oracle.qgemm_f16_inputs_f64(qtype, c["W"], n, k, c["X"]))
    assert rel <= 2e-5, rel


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T", SHAPES[::2])
def test_residual(q, qtype, n, k, T):
    c = synth.make_case(qtype, n, k, T, residual=True, seed=n * T)
    buf, Y = guarded(T, n)
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]))
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("qtype", QTYPES)
def test_residual_alias_accumulates(q, qtype):
    n, k, T = 256, 512, 64
    c = synth.make_case(qtype, n, k, T, residual=True, seed=11)
    Y = dev(c["R"])
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, Y)
    assert_f16_leg(Y.cpu().numpy(), oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T", [(256, 512, 17), (384, 1024, 200), (200, 768, 129)])
def test_swiglu(q, qtype, n, k, T):
    c = synth.make_case(qtype, n, k, T, gate_up=True, seed=n + T)
    buf, Y = guarded(T, n)
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, Wu=dev(c["Wu"]))
    check_guards(buf, T, n)
    y = Y.cpu().numpy()
    assert_f16_leg(y, oracle.gate_up_swiglu_f64(qtype, c["W"], c["Wu"], n, k, c["X"]))
    rel, _, _ = errors(y, oracle.gate_up_swiglu_f16_inputs_f64(qtype, c["W"], c["Wu"], n, k, c["X"]))
    assert rel <= 2e-5, rel


def test_public_swiglu_entry(q):
    n, k, T = 256, 512, 40
    c = synth.make_case(synth.Q4_0, n, k, T, gate_up=True, seed=2)
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm_gate_up_swiglu(synth.Q4_0, dev(c["W"]), dev(c["Wu"]), n, k, dev(c["X"]), T, Y)
    q.apr_stream_status()
    assert_f16_leg(Y.cpu().numpy(), oracle.gate_up_swiglu_f64(synth.Q4_0, c["W"], c["Wu"], n, k, c["X"]))


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("qtype", QTYPES)
def test_zero_codes_give_residual_exactly(q, qtype):
    n, k, T = 256, 512, 50
    bb = synth.block_bytes(qtype)
    Wz = np.zeros((n, k // 32, bb), np.uint8)
    Wz[..., 1] = 0x3C                          # d = 1.0
    if qtype == synth.Q4_0:
        Wz[..., 2:] = 0x88                     # every nibble 8 -> weight 0
    Wz = Wz.reshape(n, -1)
    X = synth.activations(T, k, 1)
    R = synth.activations(T, n, 2)
    Y = torch.empty((T, n), device="cuda")
    gemm(q, qtype, dev(Wz), n, k, dev(X), T, Y, dev(R))
    np.testing.assert_array_equal(Y.cpu().numpy(), R)


def test_zero_gate_gives_zero_swiglu(q):
    n, k, T = 128, 256, 33
    Wz = np.zeros((n, k // 32, 34), np.uint8).reshape(n, -1)
    c = synth.make_case(synth.Q8_0, n, k, T, gate_up=True, seed=4)
    Y = torch.empty((T, n), device="cuda")
    gemm(q, synth.Q8_0, dev(Wz), n, k, dev(c["X"]), T, Y, Wu=dev(c["Wu"]))
    assert torch.all(Y == 0)


@pytest.mark.parametrize("qtype", QTYPES)
def test_identity_x_returns_fp16_weight(q, qtype):
    n, k = 200, 256
    W = synth.quantize(qtype, synth.weight_f32(n, k, seed=6))
    X = np.eye(k, dtype=np.float32)
    Y = torch.empty((k, n), device="cuda")
    gemm(q, qtype, dev(W), n, k, dev(X), k, Y)
    want = oracle.dequant_f32(qtype, W, n, k).astype(np.float16).astype(np.float32).T
    np.testing.assert_array_equal(Y.cpu().numpy(), want)


def test_scaling_x_by_two_doubles_y(q):
    # fp16(2x) == 2 fp16(x) needs x outside fp16's subnormal range (|x| >= 2^-14),
    # so the few draws below it are zeroed; then every product and partial sum
    # doubles exactly.
    n, k, T = 256, 1024, 150
    c = synth.make_case(synth.Q4_0, n, k, T, seed=12)
    X = np.where(np.abs(c["X"]) < 2.0 ** -13, np.float32(0), c["X"])
    Y1 = torch.empty((T, n), device="cuda")
    Y2 = torch.empty((T, n), device="cuda")
    gemm(q, synth.Q4_0, dev(c["W"]), n, k, dev(X), T, Y1)
    gemm(q, synth.Q4_0, dev(c["W"]), n, k, dev(2 * X), T, Y2)
    np.testing.assert_array_equal(Y2.cpu().numpy(), 2 * Y1.cpu().numpy())


def test_permuting_tokens_permutes_rows(q):
    n, k, T = 256, 512, 300
    c = synth.make_case(synth.Q8_0, n, k, T, seed=13)
    perm = np.random.default_rng(0).permutation(T)
    Y1 = torch.empty((T, n), device="cuda")
    Y2 = torch.empty((T, n), device="cuda")
    gemm(q, synth.Q8_0, dev(c["W"]), n, k, dev(c["X"]), T, Y1)
    gemm(q, synth.Q8_0, dev(c["W"]), n, k, dev(c["X"][perm]), T, Y2)
    np.testing.assert_array_equal(Y2.cpu().numpy(), Y1.cpu().numpy()[perm])


@pytest.mark.parametrize("qtype", QTYPES)
def test_gemv_and_gemm_agree_for_small_T(q, qtype):
    n, k = 384, 1024
    for T in range(1, 17):
        c = synth.make_case(qtype, n, k, T, residual=True, seed=100 + T)
        Yv = torch.empty((T, n), device="cuda")
        Ym = torch.empty((T, n), device="cuda")
        q.apr_qgemm_ex(qtype, dev(c["W"]), n, k, dev(c["X"]), T, Yv, residual=dev(c["R"]), path=q.APR_PATH_GEMV)
        gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Ym, dev(c["R"]))
        assert_f16_leg(Ym.cpu().numpy(), Yv.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("T", [5, 8, 15, 17])
def test_auto_rule_large_T_takes_the_fp16_gemm(q, T):
    # T >= 5 is above the GEMV limit: the fp16 leg's error shows (it is not fp32-exact)
    assert T > q.APR_AUTO_GEMV_MAX_T
    n, k = 256, 512
    c = synth.make_case(synth.Q8_0, n, k, T, seed=0)
    Y = torch.empty((T, n), device="cuda")
    q.apr_qgemm(synth.Q8_0, dev(c["W"]), n, k, dev(c["X"]), T, Y)
    q.apr_stream_status()
    ref = oracle.qgemm_f64(synth.Q8_0, c["W"], n, k, c["X"])
    rel, _ = assert_f16_leg(Y.cpu().numpy(), ref)
    assert rel > 1e-5


# ------------------------------------------------------------------ 256-token tiles
# The GEMM takes 256-token tiles when they still give every SM a tile (here
# 37 x 5 = 185 tiles); ragged rows and tokens, residual through the operand
# ring (n % 4 == 0) and straight from memory (n % 4 != 0).
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,res", [(4736, False), (4736, True), (4738, True)])
def test_wide_tiles(q, qtype, n, res):
    k, T = 512, 1030
    c = synth.make_case(qtype, n, k, T, residual=res, seed=n + qtype)
    buf, Y = guarded(T, n)
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]) if res else None)
    check_guards(buf, T, n)
    assert_f16_leg(Y.cpu().numpy(), oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))


# ------------------------------------------------------------------ tile plans
# Small grids run 256-token tiles split over k between the two CTAs of a
# cluster (each finalizes half the tile's tokens); with T = 100 or 300 some of
# a CTA's 64-token pieces hold no token. 80 row tiles of 256 tokens are too
# many to split and too few for 256-token tiles, so they take 128-token tiles.
# Both with and without a residual, and with rows that are not a multiple of 4
# (residual and output through direct loads and stores instead of TMA).
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("n,k,T,res", [(298, 512, 100, True), (296, 512, 100, True), (296, 512, 100, False),
                                       (512, 2048, 300, True), (512, 2048, 300, False), (10240, 256, 200, False),
                                       (10240, 256, 200, True), (10238, 256, 130, True)])
def test_tile_plans(q, qtype, n, k, T, res):
    c = synth.make_case(qtype, n, k, T, residual=res, seed=3 * n + T)
    buf, Y = guarded(T, n)
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, dev(c["R"]) if res else None)
    check_guards(buf, T, n)
    y = Y.cpu().numpy()
    assert_f16_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"]))
    rel, _, _ = errors(y, oracle.qgemm_f16_inputs_f64(qtype, c["W"], n, k, c["X"], c["R"]))
    assert rel <= 2e-5, rel


# Gate/up at a size with several waves of CTAs: the output must repeat bit for
# bit. (An odd raw ring once let a warpgroup read the other weight's chunk
# now and then: a race that only repetition shows.)
@pytest.mark.parametrize("qtype", QTYPES)
def test_gate_up_repeats_bitwise(q, qtype):
    n, k, T = 12288, 4096, 512
    c = synth.make_case(qtype, n, k, T, gate_up=True, seed=61)
    W, Wu, X = dev(c["W"]), dev(c["Wu"]), dev(c["X"])
    Y0 = torch.empty((T, n), device="cuda")
    q.apr_qgemm_ex(qtype, W, n, k, X, T, Y0, Wu=Wu, path=q.APR_PATH_GEMM)
    q.apr_stream_status()
    Y = torch.empty((T, n), device="cuda")
    for _ in range(24):
        q.apr_qgemm_ex(qtype, W, n, k, X, T, Y, Wu=Wu, path=q.APR_PATH_GEMM)
        q.apr_stream_status()
        assert torch.equal(Y, Y0)
    # and one row block against the oracle
    rows = slice(0, 256)
    ref = oracle.gate_up_swiglu_f64(qtype, c["W"][rows], c["Wu"][rows], 256, k, c["X"])
    assert_f16_leg(Y0[:, rows].cpu().numpy(), ref)


def test_split_k_is_deterministic(q):
    # the split partials are added in split order whichever CTA finishes first
    n, k, T = 512, 4096, 512
    c = synth.make_case(synth.Q4_0, n, k, T, residual=True, seed=77)
    W, X, R = dev(c["W"]), dev(c["X"]), dev(c["R"])
    outs = []
    for _ in range(3):
        Y = torch.empty((T, n), device="cuda")
        gemm(q, synth.Q4_0, W, n, k, X, T, Y, R)
        outs.append(Y.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


# 192-token tiles: 6144 rows take them at T = 300, 400 and 512 (their waves
# cost less than those of 256-token tiles, see plan_gemm_tc); ragged last
# token tiles (300 = 192 + 108: two of its three
# 64-token pieces hold tokens; 400 = 2 x 192 + 16: one), plain and residual
# epilogues, a block format and a superblock format
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q4_K])
@pytest.mark.parametrize("T,res", [(300, True), (512, False), (400, True)])
def test_192_token_tiles(q, qtype, T, res):
    n, k = 6144, 512
    c = synth.make_case(qtype, n, k, T, residual=res, seed=T + res)
    buf, Y = guarded(T, n)
    gemm(q, qtype, dev(c["W"]), n, k, dev(c["X"]), T, Y, R=dev(c["R"]) if res else None)
    check_guards(buf, T, n)
    y = Y.cpu().numpy()
    assert_f16_leg(y, oracle.qgemm_f64(qtype, c["W"], n, k, c["X"], c["R"] if res else None))
    rel, _, _ = errors(y, oracle.qgemm_f16_inputs_f64(qtype, c["W"], n, k, c["X"], c["R"] if res else None))
    assert rel <= 2e-5, rel
