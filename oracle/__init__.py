"""fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import this package. The GPU path never does.
"""
from .attention import (  # noqa: F401
    attention_probs,
    attn_bwd_ref,
    attn_bwd_unit,
    attn_fwd_ref,
    attn_fwd_rows,
    attn_fwd_unit,
    expand_block_mask,
)
from .bruteforce import bwd_bruteforce, fwd_bruteforce  # noqa: F401
from .philox import dropout_keep, dropout_threshold, philox4x32_10  # noqa: F401
