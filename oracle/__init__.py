"""CPU oracle for exact attention (fp64).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product path. Nothing here calls or
imports the CUDA library, and the CUDA library shares no code with it.
"""
from .attention import (  # noqa: F401
    attention_backward,
    attention_backward_rows,
    attention_forward,
    attention_forward_rows,
    batched_backward,
    batched_forward,
    blocked_attention_forward,
    gather_pages,
    merge_states,
    online_softmax_state,
    paged_decode_forward,
    probabilities,
    safe_softmax,
    softmax_grad,
    varlen_backward,
    varlen_forward,
    visible,
)
