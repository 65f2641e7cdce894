"""The C-ABI library on the host (no GPU needed, no kernel launched).

* it builds, loads and exports every symbol include/apr_qgemm.h declares;
* the header and the binding agree on names and constants;
* argument errors come back as the documented status codes before anything
  touches the device (pointer checks as in aprender-serve 0.70.2
  src/cuda/executor/gdn_prefill_ops.rs qp_launch; empty batch = success as in
  oxibonsai-kernels 0.1.4 try_cuda_prefill_q_std).
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "apr_qgemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(apr_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(q):
    names = declared_functions()
    assert len(names) == 17, names
    lib = q.library()
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(q.EXPORTS) == names


def test_header_constants_match_binding(q):
    text = open(HEADER).read()
    for name in ["APR_F16", "APR_Q4_0", "APR_Q8_0", "APR_Q4_K", "APR_Q5_K", "APR_Q6_K", "APR_IQ4_XS", "APR_LEG_F16", "APR_LEG_EXACT_F32", "APR_PATH_AUTO", "APR_PATH_GEMV",
                 "APR_PATH_GEMM", "APR_OK", "APR_E_INVAL", "APR_E_QTYPE", "APR_E_ALIGN", "APR_E_ALIAS",
                 "APR_E_DEVICE", "APR_E_LAUNCH", "APR_E_TIMEOUT", "APR_E_NOMEM"]:
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m, name
        assert int(m.group(1)) == getattr(q, name), name
    assert q.library().apr_gemv_max_T() == q.APR_GEMV_MAX_T == 16
    m = re.search(r"#define APR_AUTO_GEMV_MAX_T (\d+)", text)
    assert m and int(m.group(1)) == q.APR_AUTO_GEMV_MAX_T == 4
    m = re.search(r"#define APR_FFN_CHUNK_ROWS (\d+)", text)
    assert m and int(m.group(1)) == q.APR_FFN_CHUNK_ROWS


# Raw calls through ctypes with fake (never dereferenced) addresses: every
# case fails on the host before any CUDA call, except the last ones, which
# pass the checks and then find no usable device here (or no-op).
A = 1 << 20  # a 16-byte aligned fake address


def call(q, *args):
    return q.library().apr_qgemm(*args)


@pytest.mark.parametrize("args,code,needle", [
    ((5, A, 64, 64, 2 * A, 8, 3 * A, None, None), -2, "qtype"),
    ((2, A, 64, 33, 2 * A, 8, 3 * A, None, None), -1, "k"),
    ((2, A, 64, 0, 2 * A, 8, 3 * A, None, None), -1, "k"),
    ((2, A, -1, 64, 2 * A, 8, 3 * A, None, None), -1, "n="),
    ((2, A, 64, 64, 2 * A, -3, 3 * A, None, None), -1, "T="),
    ((2, None, 64, 64, 2 * A, 8, 3 * A, None, None), -1, "null"),
    ((2, A, 64, 64, None, 8, 3 * A, None, None), -1, "null"),
    ((2, A, 64, 64, 2 * A, 8, None, None, None), -1, "null"),
    ((2, A + 4, 64, 64, 2 * A, 8, 3 * A, None, None), -3, "aligned"),
    ((2, A, 64, 64, 2 * A + 8, 8, 3 * A, None, None), -3, "aligned"),
    ((2, A, 64, 64, 2 * A, 8, 3 * A + 2, None, None), -3, "aligned"),
    ((2, A, 64, 64, 2 * A, 8, 3 * A, 4 * A + 4, None), -3, "aligned"),
    ((2, A, 64, 64, 2 * A, 8, 2 * A + 16, None, None), -4, "X"),
    ((2, A, 64, 64, 2 * A, 8, A + 32, None, None), -4, "W"),
    ((2, A, 64, 64, 2 * A, 8, 3 * A, 3 * A + 16, None), -4, "residual"),
    ((0, A, 64, 64, 2 * A, 8, 3 * A, None, None), -2, "qtype"),
    ((3, A, 64, 64, 2 * A, 8, 3 * A, None, None), -2, "qtype"),
    ((1, A, 64, 48, 2 * A, 8, 3 * A, None, None), -1, "k"),
    ((12, A, 64, 128, 2 * A, 8, 3 * A, None, None), -1, "256"),   # Q4_K takes whole superblocks
    ((13, A, 64, 128, 2 * A, 8, 3 * A, None, None), -1, "256"),   # so does Q5_K
    # a Q5_K weight spans 22 bytes per 32 weights: 64 x 256 -> 11264 bytes from A
    ((13, A, 64, 256, 2 * A, 8, A + 11264 - 16, None, None), -4, "W"),
    ((14, A, 64, 1024, 2 * A, 8, 3 * A, None, None), -1, "2048"),  # Q6_K rows on 16-byte boundaries
    # a Q6_K weight spans 210 bytes per 256 weights: 64 x 2048 -> 107520 bytes from A
    ((14, A, 64, 2048, 2 * A, 8, A + 107520 - 16, None, None), -4, "W"),
    ((23, A, 64, 256, 2 * A, 8, 3 * A, None, None), -1, "512"),  # IQ4_XS rows on 16-byte boundaries
    # an IQ4_XS weight spans 136 bytes per 256 weights: 64 x 512 -> 17408 bytes from A
    ((23, A, 64, 512, 2 * A, 8, A + 17408 - 16, None, None), -4, "W"),
    # an F16 weight spans 2 bytes a weight: 64 x 64 -> 8192 bytes from A
    ((1, A, 64, 64, 2 * A, 8, A + 8192 - 16, None, None), -4, "W"),
    ((2, A, (1 << 24) + 1, 64, 2 * A, 8, 3 * A, None, None), -1, "limits"),
    ((2, A, 64, (1 << 20) + 32, 2 * A, 8, 3 * A, None, None), -1, "limits"),
])
def test_argument_errors(q, args, code, needle):
    assert call(q, *args) == code
    assert needle in q.apr_last_error()


def test_empty_batch_is_success_without_device(q):
    assert call(q, 2, A, 64, 64, 2 * A, 0, 3 * A, None, None) == 0
    assert call(q, 8, A, 0, 64, 2 * A, 5, 3 * A, None, None) == 0
    assert call(q, 2, None, 64, 64, None, 0, None, None, None) == 0


def test_swiglu_and_gemv_specific_errors(q):
    lib = q.library()
    assert lib.apr_qgemm_gate_up_swiglu(2, A, None, 64, 64, 2 * A, 8, 3 * A, None) == -1
    assert lib.apr_qgemv(2, A, 64, 64, 2 * A, 17, 3 * A, None, None) == -1
    assert "T <= 16" in q.apr_last_error()
    args = q.capi._Args(2, 0, 0, A, 5 * A, 64, 64, 8, 2 * A, 4 * A, 3 * A, None)
    assert lib.apr_qgemm_ex(ctypes.byref(args)) == -1       # SwiGLU with a residual
    args = q.capi._Args(2, 7, 0, A, None, 64, 64, 8, 2 * A, None, 3 * A, None)
    assert lib.apr_qgemm_ex(ctypes.byref(args)) == -1       # unknown leg
    args = q.capi._Args(2, 0, 9, A, None, 64, 64, 8, 2 * A, None, 3 * A, None)
    assert lib.apr_qgemm_ex(ctypes.byref(args)) == -1       # unknown path
    assert lib.apr_qgemm_ex(None) == -1
    for ldy in (-1, 63, (1 << 28) + 1):                      # strided output: 0 or n <= ldy <= 2^28
        args = q.capi._Args(2, 0, 0, A, None, 64, 64, 8, 2 * A, None, 3 * A, None, ldy)
        assert lib.apr_qgemm_ex(ctypes.byref(args)) == -1, ldy
        assert "ldy" in q.apr_last_error()
    # a strided Y reaching over X is an alias even when its first rows are not
    args = q.capi._Args(2, 0, 0, A, None, 64, 64, 8, 3 * A, None, A + 4096, None, 1 << 20)
    assert lib.apr_qgemm_ex(ctypes.byref(args)) == -4
    assert lib.apr_dequant(3, A, 4, 64, 2 * A, None) == -2
    assert lib.apr_dequant(2, A, 4, 48, 2 * A, None) == -1
    assert lib.apr_dequant(2, A, 4, 64, A + 16, None) == -4
    assert lib.apr_dequant(1, A + 1, 4, 64, 2 * A, None) == -3          # F16 needs 2-byte alignment
    assert lib.apr_dequant(1, A, 4, 64, A + 4 * 64 * 2 - 4, None) == -4  # F16: 512 bytes of W


def test_valid_call_without_gpu_reports_device(q):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # Y == residual exactly is allowed (accumulate form)
    assert call(q, 2, A, 64, 64, 2 * A, 8, 3 * A, 3 * A, None) == -5
    assert "device" in q.apr_last_error()
    # F16 passes the checks too; a Q4_0 weight of this shape ends before Y
    assert call(q, 1, A, 64, 64, 2 * A, 8, 3 * A, None, None) == -5
    assert call(q, 2, A, 64, 64, 2 * A, 8, A + 8192 - 16, None, None) == -5
    assert q.library().apr_stream_status(None) == -5


def test_bounded_wait_test_entry_checks_its_limit(q):
    import torch

    lib = q.library()
    assert lib.apr_test_bounded_wait(0, None) == q.APR_E_INVAL
    assert lib.apr_test_bounded_wait(1000001, None) == q.APR_E_INVAL
    assert "limit_us" in q.apr_last_error()
    if not torch.cuda.is_available():
        assert lib.apr_test_bounded_wait(1000, None) == q.APR_E_DEVICE


def test_binding_rejects_host_tensors(q):
    import torch

    W = torch.zeros(64 * 2 * 18, dtype=torch.uint8)
    X = torch.zeros(8, 64)
    Y = torch.zeros(8, 64)
    with pytest.raises(ValueError, match="device memory"):
        q.apr_qgemm(q.APR_Q4_0, W, 64, 64, X, 8, Y, stream=0)


def test_ffn_sublayer_argument_errors(q):
    """Every argument fault of apr_ffn_sublayer is caught on the host, before
    any device work (fake, never dereferenced, aligned addresses)."""
    lib = q.library()
    B = 1 << 24

    def args(**kw):
        a = dict(qtype=2, leg=0, Wg=B, Wu=2 * B, Wd=3 * B, hidden=256, inter=512, T=4, norm_weight=4 * B, eps=1e-5,
                 X=5 * B, stream=None)
        a.update(kw)
        return q.capi._FfnArgs(*[a[f] for f, _ in q.capi._FfnArgs._fields_])

    def rc(**kw):
        return lib.apr_ffn_sublayer(ctypes.byref(args(**kw)))

    assert lib.apr_ffn_sublayer(None) == -1
    assert rc(qtype=3) == -2
    assert rc(leg=7) == -1
    assert rc(hidden=100) == -1 and "hidden" in q.apr_last_error()
    assert rc(inter=48) == -1
    assert rc(T=-1) == -1
    assert rc(eps=-1.0) == -1 and "eps" in q.apr_last_error()
    assert rc(eps=float("nan")) == -1
    assert rc(eps=float("inf")) == -1
    assert rc(T=0) == 0                      # no-op, nothing checked further
    assert rc(Wd=None) == -1
    assert rc(norm_weight=None) == -1
    assert rc(X=5 * B + 4) == -3             # misaligned
    assert rc(X=B + 64) == -4                # X over the gate weight
    assert rc(X=4 * B - 256) == -4           # X over the norm weight


def test_normed_projection_argument_errors(q):
    lib = q.library()
    B = 1 << 24
    args = q.capi._Args(2, 0, 0, B, None, 256, 512, 8, 2 * B, None, 3 * B, None, 0)
    w = 4 * B
    assert lib.apr_qgemm_rmsnorm(None, w, 1e-5) == -1
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(args), None, 1e-5) == -1
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(args), w, -1.0) == -1
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(args), w, float("nan")) == -1
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(args), w + 4, 1e-5) == -3
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(args), 3 * B + 64, 1e-5) == -4   # Y over the norm weight
    bad = q.capi._Args(3, 0, 0, B, None, 256, 512, 8, 2 * B, None, 3 * B, None, 0)
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(bad), w, 1e-5) == -2            # the projection's own checks
    empty = q.capi._Args(2, 0, 0, B, None, 256, 512, 0, 2 * B, None, 3 * B, None, 0)
    assert lib.apr_qgemm_rmsnorm(ctypes.byref(empty), None, -1.0) == 0        # T == 0: nothing to do


def test_prefill_attention_argument_errors(q):
    lib = q.library()
    B = 1 << 26
    Qp, Kp, Vp, Op = B, 2 * B, 3 * B, 4 * B   # 64 MB apart: no overlap at these sizes

    def rc(Q=Qp, K=Kp, V=Vp, O=Op, T=8, pos0=16, nh=16, nkv=4, d=256):
        return lib.apr_prefill_attention(Q, K, V, O, T, pos0, nh, nkv, d, None)

    assert rc(T=-1) == -1
    assert rc(pos0=-1) == -1
    assert rc(nh=0) == -1
    assert rc(nkv=0) == -1
    assert rc(nh=6, nkv=4) == -1             # not a multiple
    assert rc(d=128) == -1                   # the fused form takes head_dim 256
    assert rc(pos0=(1 << 30)) == -1          # past the supported positions
    assert rc(T=1, nh=16384, nkv=16384) == -1  # cache rows wider than the transpose grid takes
    assert rc(Q=None) == -1
    assert rc(O=None) == -1
    assert rc(K=Kp + 4) == -3                # misaligned
    assert rc(O=Qp + 256) == -4              # out over Q
    assert rc(O=Vp + 1024) == -4             # out over the V cache
    assert rc(O=Kp - 4096) == -4             # out runs into the K cache
    assert rc(T=0, Q=None, K=None, V=None, O=None) == 0   # T == 0: nothing to do
    assert "head_dim" in (lib.apr_prefill_attention(Qp, Kp, Vp, Op, 1, 0, 1, 1, 64, None),
                          q.apr_last_error())[1]


def test_prefill_layer_argument_errors(q):
    import ctypes

    lib = q.library()

    def args(**kw):
        base = dict(qtype=2, leg=0, Wqkv=A, Wo=2 * A, Wg=3 * A, Wu=4 * A, Wd=5 * A, hidden=256, inter=512,
                    num_heads=2, num_kv_heads=1, head_dim=256, T=8, pos0=0, attn_norm=6 * A, ffn_norm=7 * A,
                    eps=1e-6, X=8 * A, K_cache=9 * A, V_cache=10 * A, chunk=0, stream=None)
        base.update(kw)
        return q.capi._LayerArgs(*[base[f] for f, _ in q.capi._LayerArgs._fields_])

    assert lib.apr_prefill_layer(None) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(qtype=3))) == q.APR_E_QTYPE
    assert lib.apr_prefill_layer(ctypes.byref(args(head_dim=128))) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(num_heads=3, num_kv_heads=2))) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(hidden=100))) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(eps=-1.0))) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(chunk=-1))) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(Wo=None))) == q.APR_E_INVAL
    assert lib.apr_prefill_layer(ctypes.byref(args(X=8 * A + 4))) == q.APR_E_ALIGN
    # X overlapping the K cache, and a cache overlapping a weight
    assert lib.apr_prefill_layer(ctypes.byref(args(K_cache=8 * A + 4096))) == q.APR_E_ALIAS
    assert lib.apr_prefill_layer(ctypes.byref(args(V_cache=A + 4096))) == q.APR_E_ALIAS
    assert lib.apr_prefill_layer(ctypes.byref(args(T=0))) == q.APR_OK


def test_read_stream_argument_errors(q):
    import torch

    lib = q.library()
    assert lib.apr_read_stream(A, 24, None) == q.APR_E_INVAL
    assert lib.apr_read_stream(A, -16, None) == q.APR_E_INVAL
    assert lib.apr_read_stream(None, 32, None) == q.APR_E_INVAL
    assert lib.apr_read_stream(A + 8, 32, None) == q.APR_E_ALIGN
    assert lib.apr_read_stream(A, 0, None) == q.APR_OK
    if not torch.cuda.is_available():
        assert lib.apr_read_stream(A, 32, None) == q.APR_E_DEVICE
