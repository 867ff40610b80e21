"""GB300-native (sm_103a) paged KV-cache decode.

The work happens in ``libpagedkv.so`` (hand-written CUDA kernels behind the C ABI
declared in ``include/pagedkv.h``); this package holds its sources (``csrc/``),
its build (``build.py``), the thin ctypes binding (``_lib.py``) and the seeded
synthetic workloads (``workloads.py``).
"""
from ._lib import (  # noqa: F401
    DEVERR_BLOCK_ID, DEVERR_CONTEXT, DEVERR_PREFIX, DEVERR_SLOT, DEVERR_TIMEOUT, EXPORTED, PA_BF16, PA_ERR_CUDA,
    PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE_TOO_SMALL, PA_F16, PA_INT8_BF16, PA_INT8_F16, PA_OK,
    CacheDesc, PagedKVError, cache_bytes, cache_element_offset, cache_scale_offset, copy_blocks, decode,
    decode_partition_size, decode_shared_prefix, decode_shared_prefix_partition_size,
    decode_shared_prefix_workspace_bytes, decode_window, decode_window_span, decode_workspace_bytes, load, prefill,
    read_device_errors, reshape_and_cache, status_string, swap_blocks,
)
