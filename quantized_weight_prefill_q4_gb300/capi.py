"""ctypes binding of libapr_qgemm (include/apr_qgemm.h), same names.

Argument marshalling only: tensors become device pointers, sizes are checked
against the tensors so that no call can address past an allocation, and a
nonzero status raises :class:`AprError`. Every step of the computation runs
in the CUDA library; there is no fallback, and importing this module fails if
the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libapr_qgemm.so")

APR_F16 = 1
APR_Q4_0 = 2
APR_Q8_0 = 8
APR_Q4_K = 12
APR_Q5_K = 13
APR_Q6_K = 14
APR_IQ4_XS = 23
APR_LEG_F16 = 0
APR_LEG_EXACT_F32 = 1
APR_PATH_AUTO = 0
APR_PATH_GEMV = 1
APR_PATH_GEMM = 2
APR_OK = 0
APR_E_INVAL = -1
APR_E_QTYPE = -2
APR_E_ALIGN = -3
APR_E_ALIAS = -4
APR_E_DEVICE = -5
APR_E_LAUNCH = -6
APR_E_TIMEOUT = -7
APR_E_NOMEM = -8
APR_GEMV_MAX_T = 16
APR_AUTO_GEMV_MAX_T = 4
APR_NOALLOC_MAX_TK = 8 * 1024 * 1024
APR_FFN_CHUNK_ROWS = 2048

BLOCK_BYTES = {APR_F16: 64, APR_Q4_0: 18, APR_Q8_0: 34, APR_Q4_K: 18, APR_Q5_K: 22, APR_IQ4_XS: 17}  # per 32 weights
SUPERBLOCK_BYTES = {APR_Q6_K: 210}  # bytes per 256 weights, for the formats without whole bytes per 32


def row_bytes(qtype, k):
    """Bytes of one weight row of k elements (0 for an unknown qtype)."""
    if qtype in SUPERBLOCK_BYTES:
        return k // 256 * SUPERBLOCK_BYTES[qtype]
    return k // 32 * BLOCK_BYTES.get(qtype, 0)

# Every symbol include/apr_qgemm.h declares.
EXPORTS = (
    "apr_gemv_max_T",
    "apr_qgemm",
    "apr_qgemm_gate_up_swiglu",
    "apr_qgemv",
    "apr_qgemm_ex",
    "apr_convert_f32_to_f16",
    "apr_qgemm_f16_in",
    "apr_qgemm_noalloc",
    "apr_ffn_sublayer",
    "apr_qgemm_rmsnorm",
    "apr_prefill_attention",
    "apr_prefill_layer",
    "apr_dequant",
    "apr_stream_status",
    "apr_read_stream",
    "apr_test_bounded_wait",
    "apr_last_error",
)


class AprError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"apr status {status}: {message}")
        self.status = status


class _Args(ctypes.Structure):
    _fields_ = [
        ("qtype", ctypes.c_int),
        ("leg", ctypes.c_int),
        ("path", ctypes.c_int),
        ("W", ctypes.c_void_p),
        ("Wu", ctypes.c_void_p),
        ("n", ctypes.c_int),
        ("k", ctypes.c_int),
        ("T", ctypes.c_int),
        ("X", ctypes.c_void_p),
        ("residual", ctypes.c_void_p),
        ("Y", ctypes.c_void_p),
        ("stream", ctypes.c_void_p),
        ("ldy", ctypes.c_int),
    ]


class _FfnArgs(ctypes.Structure):
    _fields_ = [
        ("qtype", ctypes.c_int),
        ("leg", ctypes.c_int),
        ("Wg", ctypes.c_void_p),
        ("Wu", ctypes.c_void_p),
        ("Wd", ctypes.c_void_p),
        ("hidden", ctypes.c_int),
        ("inter", ctypes.c_int),
        ("T", ctypes.c_int),
        ("norm_weight", ctypes.c_void_p),
        ("eps", ctypes.c_float),
        ("X", ctypes.c_void_p),
        ("stream", ctypes.c_void_p),
    ]


class _LayerArgs(ctypes.Structure):
    _fields_ = [
        ("qtype", ctypes.c_int),
        ("leg", ctypes.c_int),
        ("Wqkv", ctypes.c_void_p),
        ("Wo", ctypes.c_void_p),
        ("Wg", ctypes.c_void_p),
        ("Wu", ctypes.c_void_p),
        ("Wd", ctypes.c_void_p),
        ("hidden", ctypes.c_int),
        ("inter", ctypes.c_int),
        ("num_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("T", ctypes.c_int),
        ("pos0", ctypes.c_int),
        ("attn_norm", ctypes.c_void_p),
        ("ffn_norm", ctypes.c_void_p),
        ("eps", ctypes.c_float),
        ("X", ctypes.c_void_p),
        ("K_cache", ctypes.c_void_p),
        ("V_cache", ctypes.c_void_p),
        ("chunk", ctypes.c_int),
        ("stream", ctypes.c_void_p),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built: run quantized_weight_prefill_q4_gb300.build.build_library() (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci = ctypes.c_void_p, ctypes.c_int
    sig = {
        "apr_gemv_max_T": ([], ci),
        "apr_qgemm": ([ci, vp, ci, ci, vp, ci, vp, vp, vp], ci),
        "apr_qgemm_gate_up_swiglu": ([ci, vp, vp, ci, ci, vp, ci, vp, vp], ci),
        "apr_qgemv": ([ci, vp, ci, ci, vp, ci, vp, vp, vp], ci),
        "apr_qgemm_ex": ([ctypes.POINTER(_Args)], ci),
        "apr_convert_f32_to_f16": ([vp, ctypes.c_longlong, vp, vp], ci),
        "apr_qgemm_f16_in": ([ci, vp, vp, ci, ci, vp, ci, vp, vp, vp], ci),
        "apr_qgemm_noalloc": ([ci, vp, ci, ci, vp, ci, vp, vp, vp], ci),
        "apr_ffn_sublayer": ([ctypes.POINTER(_FfnArgs)], ci),
        "apr_qgemm_rmsnorm": ([ctypes.POINTER(_Args), vp, ctypes.c_float], ci),
        "apr_prefill_attention": ([vp, vp, vp, vp, ci, ci, ci, ci, ci, vp], ci),
        "apr_prefill_layer": ([ctypes.POINTER(_LayerArgs)], ci),
        "apr_dequant": ([ci, vp, ci, ci, vp, vp], ci),
        "apr_stream_status": ([vp], ci),
        "apr_test_bounded_wait": ([ctypes.c_uint, vp], ci),
        "apr_read_stream": ([vp, ctypes.c_longlong, vp], ci),
        "apr_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _check(status: int) -> int:
    if status != APR_OK:
        raise AprError(status, _lib.apr_last_error().decode(errors="replace"))
    return status


def _ptr(x, name: str, *, dtype=None, min_bytes: int = 0):
    """Device pointer of a CUDA tensor (checked), an int (trusted), or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch

    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a CUDA tensor or a device pointer, got {type(x).__name__}")
    if not x.is_cuda:
        raise ValueError(f"{name}: tensor is on {x.device}, the library takes device memory")
    if not x.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {x.dtype}")
    nbytes = x.numel() * x.element_size()
    if nbytes < min_bytes:
        raise ValueError(f"{name}: holds {nbytes} bytes, the call addresses {min_bytes}")
    return x.data_ptr()


def _rows_ptr(x, name: str, rows: int, cols: int, ld: int):
    """Device pointer of f32 rows `ld` apart (a 2-D view with strides (ld, 1),
    or any contiguous tensor), checked to hold (rows - 1) * ld + cols floats."""
    if x is None or isinstance(x, int):
        return x
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32:
        raise ValueError(f"{name}: expected a float32 CUDA tensor")
    if not x.is_contiguous() and not (x.dim() == 2 and x.stride() == (ld, 1)):
        raise ValueError(f"{name}: expected a contiguous tensor or a 2-D view with strides ({ld}, 1)")
    need = ((rows - 1) * ld + cols) * 4 if rows > 0 else 0
    have = x.untyped_storage().nbytes() - x.storage_offset() * 4
    if have < need:
        raise ValueError(f"{name}: holds {have} bytes from its start, the call addresses {need}")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _sizes(qtype, n, k, T):
    n_, k_, T_ = max(n, 0), max(k, 0), max(T, 0)
    return n_ * row_bytes(qtype, k_), T_ * k_ * 4, T_ * n_ * 4


def _dtypes():
    import torch

    return torch.uint8, torch.float32


def apr_gemv_max_T() -> int:
    return _lib.apr_gemv_max_T()


def apr_last_error() -> str:
    return _lib.apr_last_error().decode(errors="replace")


def apr_qgemm(qtype, W, n, k, X, T, Y, residual=None, stream=None) -> int:
    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    return _check(_lib.apr_qgemm(qtype, _ptr(W, "W", dtype=u8, min_bytes=wb), n, k,
                                 _ptr(X, "X", dtype=f32, min_bytes=xb), T,
                                 _ptr(Y, "Y", dtype=f32, min_bytes=yb),
                                 _ptr(residual, "residual", dtype=f32, min_bytes=yb), _stream(stream)))


def apr_qgemm_gate_up_swiglu(qtype, Wg, Wu, n, k, X, T, Y, stream=None) -> int:
    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    return _check(_lib.apr_qgemm_gate_up_swiglu(qtype, _ptr(Wg, "Wg", dtype=u8, min_bytes=wb),
                                                _ptr(Wu, "Wu", dtype=u8, min_bytes=wb), n, k,
                                                _ptr(X, "X", dtype=f32, min_bytes=xb), T,
                                                _ptr(Y, "Y", dtype=f32, min_bytes=yb), _stream(stream)))


def apr_qgemv(qtype, W, n, k, X, T, Y, residual=None, stream=None) -> int:
    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    return _check(_lib.apr_qgemv(qtype, _ptr(W, "W", dtype=u8, min_bytes=wb), n, k,
                                 _ptr(X, "X", dtype=f32, min_bytes=xb), T,
                                 _ptr(Y, "Y", dtype=f32, min_bytes=yb),
                                 _ptr(residual, "residual", dtype=f32, min_bytes=yb), _stream(stream)))


def apr_qgemm_ex(qtype, W, n, k, X, T, Y, *, residual=None, Wu=None, leg=APR_LEG_F16, path=APR_PATH_AUTO,
                 stream=None, ldy=0) -> int:
    """Full form; ldy > 0 writes row t of Y at Y + t * ldy (and reads the
    residual's rows the same way): Y and residual may then be 2-D views with
    strides (ldy, 1)."""
    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    if ldy:
        rp = _rows_ptr(residual, "residual", T, n, ldy)
        yp = _rows_ptr(Y, "Y", T, n, ldy)
    else:
        rp = _ptr(residual, "residual", dtype=f32, min_bytes=yb)
        yp = _ptr(Y, "Y", dtype=f32, min_bytes=yb)
    a = _Args(qtype, leg, path, _ptr(W, "W", dtype=u8, min_bytes=wb), _ptr(Wu, "Wu", dtype=u8, min_bytes=wb),
              n, k, T, _ptr(X, "X", dtype=f32, min_bytes=xb), rp, yp, _stream(stream), ldy)
    return _check(_lib.apr_qgemm_ex(ctypes.byref(a)))


def apr_convert_f32_to_f16(X, count, X16, stream=None) -> int:
    import torch

    return _check(_lib.apr_convert_f32_to_f16(_ptr(X, "X", dtype=torch.float32, min_bytes=4 * max(count, 0)), count,
                                              _ptr(X16, "X16", dtype=torch.float16, min_bytes=2 * max(count, 0)),
                                              _stream(stream)))


def apr_qgemm_f16_in(qtype, W, n, k, X16, T, Y, residual=None, Wu=None, stream=None) -> int:
    import torch

    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    return _check(_lib.apr_qgemm_f16_in(qtype, _ptr(W, "W", dtype=u8, min_bytes=wb),
                                        _ptr(Wu, "Wu", dtype=u8, min_bytes=wb), n, k,
                                        _ptr(X16, "X16", dtype=torch.float16, min_bytes=xb // 2), T,
                                        _ptr(Y, "Y", dtype=f32, min_bytes=yb),
                                        _ptr(residual, "residual", dtype=f32, min_bytes=yb), _stream(stream)))


def apr_qgemm_noalloc(qtype, W, n, k, X, T, Y, residual=None, stream=None) -> int:
    """apr_qgemm's tensor-core GEMM without device allocation (fixed scratch)."""
    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    return _check(_lib.apr_qgemm_noalloc(qtype, _ptr(W, "W", dtype=u8, min_bytes=wb), n, k,
                                         _ptr(X, "X", dtype=f32, min_bytes=xb), T,
                                         _ptr(Y, "Y", dtype=f32, min_bytes=yb),
                                         _ptr(residual, "residual", dtype=f32, min_bytes=yb), _stream(stream)))


def apr_qgemm_rmsnorm(qtype, W, n, k, X, T, Y, norm_weight, eps, *, residual=None, Wu=None, leg=APR_LEG_F16,
                      path=APR_PATH_AUTO, stream=None, ldy=0) -> int:
    """apr_qgemm_ex on RMSNorm(X) (norm_weight, eps): Y = h . W^T (+ residual),
    or the gate/up SwiGLU of h with Wu."""
    u8, f32 = _dtypes()
    wb, xb, yb = _sizes(qtype, n, k, T)
    if ldy:
        rp = _rows_ptr(residual, "residual", T, n, ldy)
        yp = _rows_ptr(Y, "Y", T, n, ldy)
    else:
        rp = _ptr(residual, "residual", dtype=f32, min_bytes=yb)
        yp = _ptr(Y, "Y", dtype=f32, min_bytes=yb)
    a = _Args(qtype, leg, path, _ptr(W, "W", dtype=u8, min_bytes=wb), _ptr(Wu, "Wu", dtype=u8, min_bytes=wb),
              n, k, T, _ptr(X, "X", dtype=f32, min_bytes=xb), rp, yp, _stream(stream), ldy)
    return _check(_lib.apr_qgemm_rmsnorm(ctypes.byref(a), _ptr(norm_weight, "norm_weight", dtype=f32,
                                                               min_bytes=max(k, 0) * 4), float(eps)))


def apr_ffn_sublayer(qtype, Wg, Wu, Wd, hidden, inter, T, norm_weight, eps, X, leg=APR_LEG_F16, stream=None) -> int:
    """X[T][hidden] += down(silu(h . Wg^T) * (h . Wu^T)), h = RMSNorm(X) with
    norm_weight and eps; X is updated in place."""
    u8, f32 = _dtypes()
    h_, i_, t_ = max(hidden, 0), max(inter, 0), max(T, 0)
    wgu = i_ * row_bytes(qtype, h_)
    wd = h_ * row_bytes(qtype, i_)
    a = _FfnArgs(qtype, leg, _ptr(Wg, "Wg", dtype=u8, min_bytes=wgu), _ptr(Wu, "Wu", dtype=u8, min_bytes=wgu),
                 _ptr(Wd, "Wd", dtype=u8, min_bytes=wd), hidden, inter, T,
                 _ptr(norm_weight, "norm_weight", dtype=f32, min_bytes=h_ * 4), float(eps),
                 _ptr(X, "X", dtype=f32, min_bytes=t_ * h_ * 4), _stream(stream))
    return _check(_lib.apr_ffn_sublayer(ctypes.byref(a)))


def apr_prefill_attention(Q, K_cache, V_cache, out, T, pos0, num_heads, num_kv_heads, head_dim=256,
                          stream=None) -> int:
    """Causal attention of the T query rows at positions pos0 .. pos0 + T - 1
    over the cache rows 0 .. pos0 + T - 1: Q and out [T][num_heads * head_dim],
    the caches [>= pos0 + T][num_kv_heads * head_dim], all float32."""
    _, f32 = _dtypes()
    t_, p_ = max(T, 0), max(pos0, 0)
    qb = t_ * max(num_heads, 0) * max(head_dim, 0) * 4
    cb = (t_ + p_) * max(num_kv_heads, 0) * max(head_dim, 0) * 4 if t_ else 0
    return _check(_lib.apr_prefill_attention(
        _ptr(Q, "Q", dtype=f32, min_bytes=qb), _ptr(K_cache, "K_cache", dtype=f32, min_bytes=cb),
        _ptr(V_cache, "V_cache", dtype=f32, min_bytes=cb), _ptr(out, "out", dtype=f32, min_bytes=qb), T, pos0,
        num_heads, num_kv_heads, head_dim, _stream(stream)))


def apr_dequant(qtype, W, n, k, out, stream=None) -> int:
    u8, f32 = _dtypes()
    wb, _, _ = _sizes(qtype, n, k, 0)
    ob = max(n, 0) * max(k, 0) * 4
    return _check(_lib.apr_dequant(qtype, _ptr(W, "W", dtype=u8, min_bytes=wb), n, k,
                                   _ptr(out, "out", dtype=f32, min_bytes=ob), _stream(stream)))


def apr_stream_status(stream=None) -> int:
    return _check(_lib.apr_stream_status(_stream(stream)))


def apr_test_bounded_wait(limit_us, stream=None) -> int:
    """Enqueues the failure-detection test kernel (a bounded wait that runs
    out after limit_us microseconds); apr_stream_status then reports the
    timeout."""
    return _check(_lib.apr_test_bounded_wait(int(limit_us), _stream(stream)))


def apr_prefill_layer(qtype, Wqkv, Wo, Wg, Wu, Wd, hidden, inter, num_heads, num_kv_heads, T, pos0, attn_norm,
                      ffn_norm, eps, X, K_cache, V_cache, *, leg=APR_LEG_F16, chunk=0, head_dim=256,
                      stream=None) -> int:
    """One prefill layer over X[T][hidden] in place (attention sublayer with k
    and v written into the cache rows pos0 .., then the FFN sublayer), in
    chunks of `chunk` rows."""
    u8, f32 = _dtypes()
    h_, i_, t_ = max(hidden, 0), max(inter, 0), max(T, 0)
    qd, kvd = max(num_heads, 0) * max(head_dim, 0), max(num_kv_heads, 0) * max(head_dim, 0)
    crow = max(pos0, 0) + t_
    hrow = row_bytes(qtype, h_)
    a = _LayerArgs(qtype, leg, _ptr(Wqkv, "Wqkv", dtype=u8, min_bytes=(qd + 2 * kvd) * hrow),
                   _ptr(Wo, "Wo", dtype=u8, min_bytes=h_ * row_bytes(qtype, qd)),
                   _ptr(Wg, "Wg", dtype=u8, min_bytes=i_ * hrow),
                   _ptr(Wu, "Wu", dtype=u8, min_bytes=i_ * hrow),
                   _ptr(Wd, "Wd", dtype=u8, min_bytes=h_ * row_bytes(qtype, i_)), hidden, inter, num_heads,
                   num_kv_heads, head_dim, T, pos0, _ptr(attn_norm, "attn_norm", dtype=f32, min_bytes=h_ * 4),
                   _ptr(ffn_norm, "ffn_norm", dtype=f32, min_bytes=h_ * 4), float(eps),
                   _ptr(X, "X", dtype=f32, min_bytes=t_ * h_ * 4),
                   _ptr(K_cache, "K_cache", dtype=f32, min_bytes=crow * kvd * 4),
                   _ptr(V_cache, "V_cache", dtype=f32, min_bytes=crow * kvd * 4), chunk, _stream(stream))
    return _check(_lib.apr_prefill_layer(ctypes.byref(a)))


def apr_read_stream(src, nbytes, stream=None) -> int:
    """Streams nbytes of the device tensor src as the T = 1 GEMV streams its
    weight, computing nothing (a measurement reference)."""
    return _check(_lib.apr_read_stream(_ptr(src, "src", min_bytes=int(nbytes)), int(nbytes), _stream(stream)))
