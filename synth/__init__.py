"""Seeded synthetic inputs for the Q4_0 / Q8_0 prefill GEMM.

This package is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It only *makes* inputs: seeded normal draws and the GGUF block
encoders that turn an f32 weight into Q4_0 / Q8_0 / F16 bytes. It holds none of the
arithmetic the prefill path computes (block decoding, the products, the
epilogues): that lives, twice and independently, in ``oracle/`` and in the
CUDA library.
"""

from .gen import (  # noqa: F401
    F16,
    Q4_0,
    Q8_0,
    Q4_K,
    Q5_K,
    Q6_K,
    IQ4_XS,
    BLOCK_ELEMS,
    block_bytes,
    quantize,
    quantize_q4_0,
    quantize_q8_0,
    quantize_f16,
    quantize_q4_k,
    quantize_q5_k,
    quantize_q6_k,
    quantize_iq4_xs,
    row_bytes,
    weight_f32,
    activations,
    make_case,
    attention_case,
    WORKLOADS,
    SCALE_CLASSES,
    random_blocks,
)
