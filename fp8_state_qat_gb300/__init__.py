"""GB300 (sm_103a) chunked gated-delta-rule forward with dynamic FP8 E4M3 state/W QDQ.

The computation lives in the CUDA library ``libgdnqat.so`` (C ABI: include/gdnqat.h);
this package is its ctypes binding plus the seeded synthetic-input generators.
"""
from .gdnqat import (  # noqa: F401
    EXPORTED,
    GDN_FLAG_KDA,
    GDN_FLAG_STATE_INT8,
    GDN_FLAG_STATE_QDQ,
    GDN_FLAG_W_QDQ,
    ChunkArgs,
    GdnError,
    chunk_bwd_workspace_bytes,
    chunk_workspace_bytes,
    fp8_tile_qdq,
    gdn_check_device_status,
    gdn_chunk_bwd,
    gdn_chunk_fwd,
    gdn_decode_step,
    gdn_prefill_decode_fwd,
    int8_block_qdq,
    kda_chunk_bwd,
    kda_chunk_fwd,
    kda_prefill_decode_fwd,
    lib_path,
    load,
    prefill_decode_workspace_bytes,
    status_string,
    workspace_bytes,
)
