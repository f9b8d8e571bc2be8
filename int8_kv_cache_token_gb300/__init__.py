"""INT8 KV-cache paged attention for GB300 (sm_103a).

The compute lives in libi8kv.so (hand-written CUDA, C ABI in include/i8kv.h);
this package holds its sources (csrc/), the in-tree build (build.py) and the
thin ctypes binding (binding.py)."""
from .binding import (  # noqa: F401
    BLOCK_SIZE,
    OUT_BF16,
    OUT_F32,
    PARTITION,
    ROUTE_BF16,
    ROUTE_INT8,
    I8KVError,
    alloc_bf16_cache,
    alloc_int8_cache,
    bf16_kv_prefix_attn,
    bf16_kv_write,
    bf16_paged_decode_attn,
    bf16_prefix_attn,
    debug_prefix_i32,
    debug_qk_i32,
    decode_workspace,
    decode_workspace_bytes,
    device_error,
    int8_paged_decode_attn,
    int8_decode_step,
    int8_paged_decode_attn_noalloc,
    int8_prefix_attn,
    kv_quant_write,
    kv_rope_quant_write,
    last_error,
    lib,
    library_path,
    prefill_chunk,
    prefix_workspace,
    prefix_workspace_bytes,
    version,
)
