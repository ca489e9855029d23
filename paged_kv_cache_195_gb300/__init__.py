"""GB300-native paged-KV attention step: KV append + paged attention.

The kernels live in ``libpagedkv.so`` (hand-written CUDA for sm_103a behind the
C ABI of ``include/pagedkv.h``); this package is its thin Python binding plus
the seeded workload generator.  Build with ``paged_kv_cache_195_gb300.build``.

One layer of an engine step is ``pkv_append`` then ``pkv_attention`` (or the
two as one call, ``pkv_append_attention``); ``pkv_append_fp8`` /
``pkv_attention_fp8kv`` (and ``pkv_append_attention_fp8``) do the same over
e4m3 pools, ``pkv_attention_cascade``
reads prompts shared by groups of requests once per group, and
``pkv_copy_blocks`` copies or swaps whole blocks.  ``get_options`` /
``set_options`` / ``options`` read and change the launch and routing options.
"""
from ._binding import (  # noqa: F401
    Dims, PagedKVError, Workspace, load_library, make_dims, paged_attention,
    paged_kv_append, pkv_append, pkv_attention, pkv_attention_noalloc, pkv_copy_blocks,
    pkv_attention_workspace_size, pkv_append_fp8, pkv_attention_fp8kv,
    CascadeWorkspace, pkv_attention_cascade, pkv_append_attention, pkv_append_attention_fp8,
    pkv_get_device_error, pkv_last_error, pkv_workspace_init,
    Options, get_options, set_options, options,
)
