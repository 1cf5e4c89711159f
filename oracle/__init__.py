"""fp64 CPU oracle for blockwise ring attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import this package.  The
product path (``ring_attn_gb300``) never imports it, and the oracle never
imports the product path; the two share no code.

Every function here is plain numpy in float64 and cites the passage of the
pages it follows.  Nothing is blocked, fused or reordered beyond what the
definition states: row blocks of queries exist only to bound memory.
"""
from .attention import (  # noqa: F401
    LAYOUTS,
    attention_bwd,
    attention_fwd,
    attention_rows,
    block_attention,
    key_grads,
    llama3_rank_attention,
    lse_merge,
    online_softmax_attention,
    permute,
    ring_attention_sharded,
    segment_ids,
    token_of_position,
    unpermute,
    varlen_token_of_position,
)
