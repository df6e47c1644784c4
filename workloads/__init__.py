"""Seeded synthetic inputs for the paged decode path.

This package is the one piece shared by the CUDA-path tests, ``bench.py`` and the
oracle.  It draws random numbers and lays out shapes and operation lists; it holds
none of the paged-attention method's arithmetic (no slot, block-table or
attention computation).  Each side replays a :class:`Workload` with its own code.
"""

from .gen import (  # noqa: F401
    DTYPES,
    Workload,
    beam_search,
    build,
    chunked_prefill,
    custom,
    decode_steps,
    mcts_tree,
    prefill_batch,
    prefix_ids,
    random_storage,
    shared_prefix,
    CONFIG_IDS,
    storage_numpy_dtype,
)
