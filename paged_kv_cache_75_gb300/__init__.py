"""Paged KV-cache attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libpa_kv.so`` (C ABI in ``include/pa_kv.h``): it
turns torch tensors into pointers, sizes and the current CUDA stream and
raises on a non-OK status.  Every step of the path runs in the library's
CUDA kernels; there is no fallback.  The library is loaded on first use and
a missing library is an error.
"""
from ._binding import (  # noqa: F401
    PA_F16, PA_BF16, PA_FP8_E4M3, PaError, KVCache, BlockPool, library, library_path,
    pa_status_str, pa_version, pa_kv_cache_write, pa_copy_blocks, pa_decode_workspace_size,
    pa_decode, pa_decode_append, pa_decode_cascade, pa_decode_cascade_workspace_size, pa_decode_partition_size, pa_decode_static_ws, pa_decode_test_wait_timeout, pa_prefill_varlen, pa_prefill_varlen_packed, pa_slot_mapping, pa_swap_blocks, pa_varlen_mixed, pa_varlen_mixed_workspace_size, torch_dtype_code,
)
