"""CPU oracle (float64) for the Q4_0 / Q8_0 / F16 / Q4_K / Q5_K / Q6_K / IQ4_XS prefill projections.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline legs use it. It shares no code with the CUDA
library and never imports it.
"""

from .qref import (  # noqa: F401
    F16,
    Q4_0,
    Q8_0,
    Q4_K,
    Q5_K,
    Q6_K,
    IQ4_XS,
    IQ4_NL_VALUES,
    iq4_xs_scales,
    q4_k_scales_mins,
    fp16_bits_to_f64,
    block_scales_and_codes,
    dequant_f64,
    dequant_f32,
    qgemm_f64,
    qgemm,
    silu_f64,
    gate_up_swiglu_f64,
    gate_up_swiglu,
    qgemm_f16_inputs_f64,
    gate_up_swiglu_f16_inputs_f64,
    rmsnorm_f64,
    ffn_sublayer_f64,
    normed_qgemm_f64,
    prefill_attention_f64,
    prefill_attention_f16_inputs_f64,
    prefill_layer_f64,
)
