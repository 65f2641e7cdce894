"""GGUF Q4_0 / Q8_0 prefill projections for GB300 (sm_103a).

``Y = X . dequant(W)^T (+ R)``, ``silu(X . Wg^T) * (X . Wu^T)`` and the small-T
GEMV, computed by the hand-written CUDA kernels of ``libapr_qgemm.so``
(C ABI: ``include/apr_qgemm.h``). The names below come from the binding
module :mod:`quantized_weight_prefill_q4_gb300.capi`, loaded on first use so
that :mod:`quantized_weight_prefill_q4_gb300.build` can run before the library
exists; using any of them without the built library raises ``ImportError``.
"""


import importlib


def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    capi = importlib.import_module(__name__ + ".capi")
    try:
        return getattr(capi, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
