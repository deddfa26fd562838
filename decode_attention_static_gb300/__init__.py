"""GB300-native decode attention over a static KV cache.

The compute lives in libdecode_attn.so (CUDA, sm_103a), declared in
include/decode_attn.h; this package is its thin Python binding. Importing it
does not load the library; the first call does, and raises LibraryNotBuilt
if it is missing.
"""
from ._binding import (  # noqa: F401
    DA_BF16,
    DA_DEVERR_KV_LEN,
    DA_DEVERR_POSITION,
    DA_DEVERR_TIMEOUT,
    DA_DEVERR_WORKSPACE,
    DA_F16,
    DecodeAttnError,
    LibraryNotBuilt,
    alloc_workspace,
    decode_attn_fwd,
    decode_attn_fwd_static_scratch,
    STATIC_SCRATCH_BYTES,
    decode_attn_workspace_size,
    decode_step_fwd,
    decode_step_layers_fwd,
    decode_step_rope_fwd,
    exported_symbols,
    kernel_for,
    kvcache_append,
    library_path,
    load_library,
    plan_splits,
    prefix_ready,
    set_prefix_ready,
    set_timing_events,
    shard_heads,
    splits_for,
    status_string,
    test_skip_slot,
    workspace_init,
)


def build_library(force: bool = False):
    """Compile the CUDA library in place (nvcc, sm_103a)."""
    from .build import build_library as _build

    return _build(force=force)
