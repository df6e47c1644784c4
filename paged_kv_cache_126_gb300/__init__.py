"""Paged KV-cache decode attention for NVIDIA GB300 (sm_103a).

The C-ABI library ``libpa.so`` (include/pa.h) holds the host block manager and
the CUDA kernels; this package is its thin Python binding plus a small engine
that sequences one decode step.  Importing it loads ``libpa.so`` and fails if the
library has not been built (``python paged_kv_cache_126_gb300/build.py``).
"""

from ._binding import (  # noqa: F401
    EXPORTED,
    BlockManager,
    PAError,
    PaDecodeParams,
    PaTensor,
    PA_DEV_BAD_BLOCK,
    PA_DEV_BAD_COPY,
    PA_DEV_BAD_LEN,
    PA_DEV_BAD_SLOT,
    PA_DEV_TIMEOUT,
    PA_ERR_OUT_OF_BLOCKS,
    PA_ERR_SCRATCH_LIMIT,
    PA_ERR_HOST_MEMORY,
    PA_ERR_CAPACITY,
    PA_ERR_SEQ_EXISTS,
    PA_ERR_UNKNOWN_SEQ,
    PA_ERR_UNSUPPORTED,
    PA_WARN_DOUBLE_FREE,
    pa_cache_append,
    pa_cache_append_split,
    pa_copy_blocks,
    pa_decode,
    pa_decode_ex,
    pa_decode_split,
    pa_decode_static,
    pa_prefill,
    pa_step_decode,
    pa_get_device_status,
    pa_selftest_wait_timeout,
    pa_launch_count,
    pa_shutdown,
    strerror as pa_strerror,
    tensor_desc,
)
from .engine import PagedKVEngine, run_workload_ops, to_device_rows  # noqa: F401
from . import _binding as _b

LIB_PATH = _b._LIB_PATH
LIB = _b.LIB
