"""GB300-native paged-KV attention step: KV append + paged attention.

The kernels live in ``libpagedkv.so`` (hand-written CUDA for sm_103a behind the
C ABI of ``include/pagedkv.h``); this package is its thin Python binding plus
the seeded workload generator.  Build with ``paged_kv_cache_195_gb300.build``.
"""
from ._binding import (  # noqa: F401
    Dims, PagedKVError, Workspace, load_library, make_dims, paged_attention,
    paged_kv_append, pkv_append, pkv_attention, pkv_attention_noalloc, pkv_copy_blocks,
    pkv_attention_workspace_size, pkv_append_fp8, pkv_attention_fp8kv,
    CascadeWorkspace, pkv_attention_cascade, pkv_append_attention,
    pkv_get_device_error, pkv_last_error, pkv_workspace_init,
)
