"""Float64 CPU oracle for gated GQA attention (head_dim 256).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline / reference leg may import it; the library never does.  It shares no
code with the CUDA path.  Every function is pinned by a test that does not retype
its formula (brute force in 40-digit arithmetic, closed forms, invariants, and a
library routine), and by planted-mistake tests that show those pins catch a
dropped term, a wrong index or sign, or a transposed operand.
"""
from .attention import (  # noqa: F401
    HEAD_DIM, SCALE, sigmoid, kv_head_of, prefill_visible, verify_visible,
    attend_rows, prefill, decode, lse_merge, head_chunk_plan, decode_head_chunked,
    tree_visible_keys, decode_tree, chain_masks, kv_append, kv_keep, masked_rows, sdpa_masked,
)
