"""Oracle for the paged decode path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct CPU statement of what the paged KV cache and its
decode attention compute: a pure-Python block manager, a NumPy model of the two
paged caches, and fp64 gather-then-dense softmax attention.  It shares no code
with the CUDA path (no kernels, headers, helpers or constants) and imports
nothing from it.  Only the test suite, the smoke check and the bench's CPU
baseline may import it; the product path never does.

Sources (web pages on PagedAttention):
  * "PagedAttention: Virtual Memory Guide for LLM Inference" -- block translation
    and address formula ("The Mathematics of Block Translation"), demand paging and
    copy-on-write ("Key Architectural Mechanics"), block pool and sequence manager
    ("Reference Implementation: Block Table & Paged Cache Manager").
  * "Solving the LLM Memory Wall: A Deep Dive into PagedAttention" -- cache layout
    [num_blocks, block_size, heads, dim] ("The Architecture at a Glance"), the
    attention equation ("1. The Mathematical Foundation"), gather/flatten/trim then
    SDPA ("Implementation: Simulating PagedAttention in PyTorch").
  * "PagedAttention, simply explained" -- the 100-block worked allocation trace
    ("How PagedAttention solves it").

Every function here has at least one pin in tests/test_oracle_*.py that checks it
against something other than itself (printed traces, closed forms, a different
library's attention, brute force, invariants).
"""

from .block_manager import (  # noqa: F401
    OracleBlockManager,
    OutOfBlocks,
    UnknownSequence,
    SequenceExists,
    DOUBLE_FREE,
)
from .cache import OracleKVCache, decode_storage, split_layout  # noqa: F401
from .attention import (  # noqa: F401
    attention_fp64,
    paged_decode,
    paged_prefill,
    prefill_weight_bound,
    partial_state,
    lse_merge,
    round_to_storage,
)
from .replay import replay  # noqa: F401
