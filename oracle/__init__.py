"""Float64 CPU oracle for paged attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
legs use this package.  The library never imports it.
"""
from .paged_attention import (  # noqa: F401
    add_sink_ref,
    admissible_mask,
    attention_logits,
    cascade_ref,
    gather_ref,
    lse_log2_to_ln,
    merge_attn_states_ref,
    merge_many_ref,
    paged_attention_ref,
    reshape_and_cache_ref,
    use_cascade_attention_ref,
    varlen_attention_ref,
)
