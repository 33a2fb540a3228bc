"""CPU oracle for the block-decoding denoise step (TEST INFRASTRUCTURE ONLY).

A plain, slow, float64 NumPy statement of what one denoising iteration of
block-cached masked-diffusion decoding computes, written from the dInfer
article ("dInfer: ...", sections on vicinity KV refresh and on hierarchical,
credit and iteration-smoothing decoding) and the Sangam abstract (cached dLLM
inference, block-sized decodes, recurring prefills).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
leg (and its ``--impl reference`` arm) may import this package. The product
path never does: it shares no code, header, table or helper with the CUDA
library, and neither side imports the other. Inputs come from ``workloads``.

Pinned functions (see ``tests/test_oracle_*.py``): ``block_attention``,
``lm_head_logits``, ``vocab_softmax_stats``, ``expected_embedding``,
``commit``, ``denoise_step``, the e2e model pieces in ``oracle.model``, the
step-level scheduler in ``oracle.sched`` and the MoE FFN in ``oracle.moe``.
"""

from .attention import block_attention  # noqa: F401
from .head import (  # noqa: F401
    expected_embedding,
    head_confidence,
    lm_head_logits,
    vocab_softmax_stats,
)
from .commit import commit, hierarchical_select, masked_spans  # noqa: F401
from .step import ambiguity, denoise_step, step_inputs_f64  # noqa: F401
