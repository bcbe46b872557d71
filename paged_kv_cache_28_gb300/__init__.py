"""Paged-KV decode attention for NVIDIA GB300 (sm_103a).

The compute lives in libpa.so (hand-written CUDA, C ABI in include/pa.h); this
package is its ctypes binding plus the seeded workload generator used by the
tests and the benchmark.  The binding is loaded on first use; calling an entry
point without the built library or without a CUDA device raises.
"""
from ._lib import (PA_DEVERR_BLOCK_ID, PA_DEVERR_FP8_CONFLICT, PA_DEVERR_SEQ_LEN,
                   PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT, PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_INT4, PAError,
                   make_shape, pa_decode, pa_decode_splitkv, pa_default_num_splits,
                   pa_merge_lse, pa_read_error_flag, pa_reshape_and_cache, pa_shape,
                   pa_splitkv_workspace_bytes, status_string)

__all__ = [
    "PA_DEVERR_BLOCK_ID", "PA_DEVERR_FP8_CONFLICT", "PA_DEVERR_SEQ_LEN", "PA_DEVERR_SLOT",
    "PA_DEVERR_TIMEOUT", "PA_KV_BF16", "PA_KV_FP8_E4M3", "PA_KV_INT4", "PAError", "make_shape", "pa_decode",
    "pa_decode_splitkv", "pa_default_num_splits", "pa_merge_lse", "pa_read_error_flag",
    "pa_reshape_and_cache", "pa_shape", "pa_splitkv_workspace_bytes", "status_string",
]
