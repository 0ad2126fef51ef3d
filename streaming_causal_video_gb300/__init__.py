"""GB300 (sm_103a) streaming causal-video chunk attention: thin Python binding of libsdv2.so.

The functions below have the names of the C ABI in include/sdv2.h and only marshal arguments:
torch tensors become device pointers, Python sequences become host int64 arrays, and a
non-zero status becomes an SDV2Error.  Every step of the path runs in the library's kernels;
there is no fallback -- if the library is missing or cannot be loaded, the calls raise.
"""
from ._binding import (  # noqa: F401
    NoiseCtl,
    SDV2Error,
    StreamConfig,
    cache_bytes,
    cache_reset,
    check_device_error,
    chunk_attention,
    chunk_attention_noalloc,
    debug_drop_kv_tile,
    debug_kv_schedule,
    debug_set_kv_splits,
    last_kv_splits,
    exported_symbols,
    lib,
    lib_path,
    meta_bytes,
    motion_l2,
    noalloc_check_device_error,
    noise_from_motion,
    qkv_rope_append,
    rope_append_kv,
    rope_refresh_rerotate,
    set_wait_timeout_ns,
    sink_update,
    visible_tokens,
    workspace_bytes,
    workspace_init,
)
from .layer import LayerCache, StreamSession  # noqa: F401
