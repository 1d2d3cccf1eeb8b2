"""paged_gqa_gb300 -- paged grouped-query attention for GB300 (sm_103a).

A thin ctypes binding over ``libpaged_gqa.so`` (C ABI in ``include/paged_gqa.h``).
The functions here only marshal torch tensors into ``pg_tensor`` descriptors and
pass the current CUDA stream; every step of the computation runs in the library's
CUDA kernels. There is no CPU or PyTorch fallback: if the library cannot be built
or loaded, the calls raise.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    PagedGQAError,
    lib_path,
    load,
    paged_gqa_attn,
    paged_gqa_attn_ex,
    paged_gqa_attn_quant_q,
    paged_gqa_sparse_attn,
    paged_gqa_cache_write,
    paged_gqa_check_device_errors,
    paged_gqa_last_error,
    paged_gqa_last_plan,
    paged_gqa_set_kernel_events,
    paged_gqa_set_path,
    paged_gqa_set_stall_test,
    paged_gqa_version,
    paged_gqa_workspace_size,
    exported_symbols,
)
