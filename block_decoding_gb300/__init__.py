"""GB300-native block-decoding denoise step for masked-diffusion LLMs.

The kernels (sm_103a CUDA) live in ``libdllm.so`` behind the C ABI of
``include/dllm.h``; this package is its thin Python binding. Importing it
without the built library raises: there is no CPU fallback.
"""

from ._binding import (  # noqa: F401
    LIB,
    LIB_PATH,
    DllmError,
    Params,
    StepArgs,
    block_attn,
    block_attn_workspace,
    commit,
    denoise_step,
    denoise_step_workspace,
    device_status,
    head_confidence,
    head_workspace,
    launch_count,
    params_struct,
    status_string,
    step_args,
    workspace,
    gemm_bf16,
    model_desc,
    model_forward,
    decode_step,
    decode_step_workspace,
    moe_ffn,
)
from .decoder import BlockDecoder  # noqa: F401
