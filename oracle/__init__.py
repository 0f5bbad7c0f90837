"""CPU oracle (fp64) for the packed paged-attention step.

Test infrastructure only: imported by tests, the smoke check and the benchmark's
CPU-baseline leg, never by the product path.
"""
from .paged_step import (  # noqa: F401
    BLOCK_SIZE,
    attention_dense_mask,
    attention_reference,
    bf16_to_f64,
    block_diagonal_causal_mask,
    gather_request,
    packed_key_layout,
    physical_slot,
    reference_cache_write,
    request_histories,
    softmax_weights,
    step_reference,
)
