"""paged_kv_cache_213_gb300 -- paged decode attention for GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind a C ABI
(``include/pagedkv.h``, built into ``_build/libpagedkv.so``).  The Python
functions here only marshal torch tensors to that ABI; there is no CPU
fallback.  The library is loaded on first use, which raises if it was not
built.
"""
from .binding import (  # noqa: F401
    PKV_ERRBIT_BLOCK_ID,
    PKV_ERRBIT_CONTEXT,
    PKV_ERRBIT_SLOT,
    PKV_ERRBIT_TIMEOUT,
    PKV_ERRBIT_WORKSPACE,
    PKV_ERRBIT_APPEND,
    PKV_TABLES_READY,
    PKV_APPEND_NEWEST,
    PKV_WORKSPACE_COUNTER_BYTES,
    PagedKVError,
    decode_plan,
    decode_plan_fp8,
    default_scale,
    get_error,
    library,
    library_path,
    multi_plan,
    paged_decode_attention,
    paged_decode_attention_fp8,
    paged_decode_attention_multi,
    paged_decode_attention_prefix_shared,
    paged_decode_attention_prefix_shared_fp8,
    paged_kv_append,
    paged_kv_append_fp8,
    paged_decode_step,
    paged_decode_step_fp8,
    paged_decode_workspace_clear,
    paged_copy_in,
    prefix_shared_plan,
    prefix_shared_plan_fp8,
    status_string,
    step_launches,
)
