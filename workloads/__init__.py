"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This package draws random numbers and rounds them to bfloat16. It holds none
of the denoise step's arithmetic (no attention, softmax, credit or selection),
so that the oracle and the kernels can both consume identical input bits
without sharing any code of the method itself.
"""

from .gen import (  # noqa: F401
    MOE_CONFIGS,
    SERVE_MIXES,
    STEP_CONFIGS,
    bf16_bits_to_f32,
    bf16_bits_to_f64,
    f32_to_bf16_bits,
    make_e2e_inputs,
    make_moe_inputs,
    make_serve_inputs,
    make_serve_trace,
    make_step_inputs,
    step_config,
)
