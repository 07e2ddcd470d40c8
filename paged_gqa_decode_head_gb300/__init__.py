"""Paged GQA decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpgqa.so`` built from ``csrc/``;
``binding`` marshals arguments to it through ctypes. Importing this package
does not load the library: the first call of a binding function does, and it
raises if the library is missing (there is no CPU fallback).
"""
from .binding import (  # noqa: F401
    PgqaError,
    attn_host_direct,
    attn_host_direct_partition_count,
    attn_host_direct_workspace_size,
    attn_host_tiled_run,
    attn_partition_merge,
    attn_tile_finalize,
    attn_tile_init,
    attn_tile_update,
    decode_attn_int8_workspace_size,
    decode_attn_multi_workspace_size,
    decode_attn_paged,
    decode_attn_paged_int8,
    decode_attn_paged_multi,
    decode_attn_paged_static,
    decode_step_paged,
    decode_step_paged_int8,
    decode_step_paged_multi,
    decode_attn_partition_count,
    decode_attn_workspace_size,
    device_error_flags,
    library_path,
    load_library,
    qk_norm_rope_append,
    qk_norm_rope_append_int8,
    qk_norm_rope_append_multi,
)
