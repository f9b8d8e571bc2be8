"""Thin Python binding of libi8kv.so (the C ABI in include/i8kv.h).

Argument marshalling only: every function checks dtypes/shapes/devices of the
torch tensors it is given, passes their device pointers and the current CUDA
stream to the C entry point of the same name, and raises I8KVError on a non-OK
status.  All arithmetic happens in the CUDA kernels.  There is no fallback: if
the library is not built, or a call fails, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE = range(6)
OUT_F32, OUT_BF16 = 0, 1
BLOCK_SIZE = 16
PARTITION = 256


class I8KVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"i8kv status {status}: {msg}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

_SIGS = {
    "i8kv_last_error": [ctypes.c_char_p, _Z],
    "i8kv_device_error": [ctypes.POINTER(ctypes.c_int)],
    "i8kv_version": [],
    "i8kv_kv_quant_write": [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P],
    "i8kv_kv_rope_quant_write": [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _P,
                                 _P, _F, _P, _P, _P, _P],
    "i8kv_decode_workspace_bytes": [_I, _I, _I, _I, _I, _I, _I],
    "i8kv_int8_paged_decode_attn": [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z,
                                    _P],
    "i8kv_int8_paged_decode_attn_u8p": [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P,
                                        _Z, _P],
    "i8kv_int8_decode_step": [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P],
    "i8kv_int8_paged_decode_attn_noalloc": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                            _P],
    "i8kv_prefix_workspace_bytes": [_I, _I, _I, _I],
    "i8kv_int8_prefix_attn": [_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _Z, _P],
    "i8kv_bf16_prefix_attn": [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _Z, _P],
    "i8kv_prefill_chunk": [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _Z,
                           _P, _P],
    "i8kv_debug_prefix_i32": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _Z,
                              _P],
    "i8kv_debug_qk_i32": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P],
    "i8kv_bf16_kv_write": [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P],
    "i8kv_bf16_kv_prefix_attn": [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _Z, _P],
    "i8kv_bf16_paged_decode_attn": [_P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P],
}


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libi8kv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise I8KVError(ERR_CUDA, f"{path} is missing: build it with int8_kv_cache_token_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _I
        L.i8kv_decode_workspace_bytes.restype = _Z
        L.i8kv_prefix_workspace_bytes.restype = _Z
        _lib = L
    return _lib


def last_error() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().i8kv_last_error(buf, 512)
    return buf.value.decode(errors="replace")


def _check(status: int):
    if status != OK:
        raise I8KVError(status, last_error())


def version() -> int:
    return int(lib().i8kv_version())


def device_error() -> int:
    """Synchronize, read and clear the device error word (0 = no failure)."""
    code = ctypes.c_int(0)
    st = lib().i8kv_device_error(ctypes.byref(code))
    if st not in (OK, ERR_DEVICE):
        _check(st)
    return int(code.value)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise I8KVError(ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise I8KVError(ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise I8KVError(ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _out(t: torch.Tensor):
    """An attention output: fp32, or bf16 (the fp32 result rounded to nearest even).
    Returns (pointer, out_dtype code)."""
    if t.dtype == torch.float32:
        return _ptr(t, None, "out"), OUT_F32
    if t.dtype == torch.bfloat16:
        return _ptr(t, None, "out"), OUT_BF16
    raise I8KVError(ERR_INVALID_ARG, f"out must be float32 or bfloat16, got {t.dtype}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _bf16(t, name):
    """bf16 tensors travel as raw 16-bit payloads (torch.bfloat16 or int16/uint16 bit patterns)."""
    if t is None:
        return None
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise I8KVError(ERR_INVALID_ARG, f"{name} must be bfloat16 (or its 16-bit pattern), got {t.dtype}")
    return _ptr(t, None, name)


# ----------------------------------------------------------------------------- cache helpers
def alloc_int8_cache(num_blocks: int, Hkv: int, D: int, device="cuda"):
    """Zeroed INT8 cache tensors in the library's layouts."""
    return dict(
        k_cache=torch.zeros((num_blocks, Hkv, D // 16, BLOCK_SIZE, 16), dtype=torch.int8, device=device),
        v_cache=torch.zeros((num_blocks, Hkv, D, BLOCK_SIZE), dtype=torch.int8, device=device),
        k_scale=torch.zeros((num_blocks, BLOCK_SIZE, Hkv), dtype=torch.float32, device=device),
        v_scale=torch.zeros((num_blocks, BLOCK_SIZE, Hkv), dtype=torch.float32, device=device),
    )


def alloc_bf16_cache(num_blocks: int, Hkv: int, D: int, device="cuda"):
    return dict(
        k_cache=torch.zeros((num_blocks, Hkv, D // 8, BLOCK_SIZE, 8), dtype=torch.bfloat16, device=device),
        v_cache=torch.zeros((num_blocks, Hkv, D, BLOCK_SIZE), dtype=torch.bfloat16, device=device),
    )


def _cache_geom(k_cache: torch.Tensor, elems_per_chunk: int):
    if k_cache.dim() != 5 or k_cache.shape[3] != BLOCK_SIZE or k_cache.shape[4] != elems_per_chunk:
        raise I8KVError(ERR_INVALID_ARG, f"k_cache shape {tuple(k_cache.shape)} is not [NB, Hkv, D/x, 16, x]")
    NB, Hkv, nchunk = k_cache.shape[:3]
    return NB, Hkv, nchunk * elems_per_chunk


# ----------------------------------------------------------------------------- producer
def kv_quant_write(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, q=None, q_i8=None, q_scale=None,
                   stream=None):
    """Quantize k, v [T, Hkv, D] (bf16) into the paged INT8 cache at slot_mapping [T];
    with q [T, Hq, D] also write q_i8 [T, Hq, D] and q_scale [T, Hq]."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    T = k.shape[0]
    Hq = 0 if q is None else q.shape[1]
    _check(lib().i8kv_kv_quant_write(
        _bf16(k, "k"), _bf16(v, "v"), _ptr(slot_mapping, torch.int32, "slot_mapping"), T, Hkv, D, BLOCK_SIZE, NB,
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _bf16(q, "q"), Hq, _ptr(q_i8, torch.int8, "q_i8"), _ptr(q_scale, torch.float32, "q_scale"),
        _stream(stream)))


def kv_rope_quant_write(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, positions=None, cos_sin=None,
                        rotary_dim: int = 0, q=None, q_i8=None, q_scale=None, q_norm_weight=None,
                        k_norm_weight=None, norm_eps: float = 1e-6, q_out=None, k_out=None, k_smooth=None,
                        stream=None):
    """kv_quant_write with Q/K RMSNorm (optional bf16 weights [D]) and rotate-half
    RoPE on the first rotary_dim dims (positions int32 [T], cos_sin float32
    [max_position, rotary_dim]) applied before the quantization; q_out / k_out
    (bf16, nullable) receive the transformed vectors; k_smooth (float32 [Hkv, D],
    nullable) smooths K's channels (K times 1/s, Q times s) before the quantization."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    T = k.shape[0]
    Hq = 0 if q is None else q.shape[1]
    max_pos = 0
    if cos_sin is not None:
        if cos_sin.dim() != 2 or cos_sin.shape[1] != rotary_dim:
            raise I8KVError(ERR_INVALID_ARG, "cos_sin must be [max_position, rotary_dim]")
        max_pos = cos_sin.shape[0]
    _check(lib().i8kv_kv_rope_quant_write(
        _bf16(k, "k"), _bf16(v, "v"), _ptr(slot_mapping, torch.int32, "slot_mapping"), T, Hkv, D, BLOCK_SIZE, NB,
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _bf16(q, "q"), Hq, _ptr(q_i8, torch.int8, "q_i8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(positions, torch.int32, "positions"), _ptr(cos_sin, torch.float32, "cos_sin"), max_pos, rotary_dim,
        _bf16(q_norm_weight, "q_norm_weight"), _bf16(k_norm_weight, "k_norm_weight"), float(norm_eps),
        _bf16(q_out, "q_out"), _bf16(k_out, "k_out"), _ptr(k_smooth, torch.float32, "k_smooth"), _stream(stream)))


def bf16_kv_write(k, v, slot_mapping, k_cache, v_cache, stream=None):
    NB, Hkv, D = _cache_geom(k_cache, 8)
    _check(lib().i8kv_bf16_kv_write(
        _bf16(k, "k"), _bf16(v, "v"), _ptr(slot_mapping, torch.int32, "slot_mapping"), k.shape[0], Hkv, D,
        BLOCK_SIZE, NB, _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"), _stream(stream)))


# ----------------------------------------------------------------------------- decode
def decode_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, max_blocks: int) -> int:
    return int(lib().i8kv_decode_workspace_bytes(B, Hq, Hkv, D, max_blocks, BLOCK_SIZE, PARTITION))


def decode_workspace(B: int, Hq: int, Hkv: int, D: int, max_blocks: int, device="cuda") -> torch.Tensor:
    """A zero-filled decode workspace (reusable by later calls on the same stream)."""
    n = decode_workspace_bytes(B, Hq, Hkv, D, max_blocks)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def int8_paged_decode_attn(out, q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                           workspace, softmax_scale: float = 0.0, partition: int = PARTITION, stream=None,
                           u8_probs: bool = False):
    """out [B, Hq, D] (float32, or bfloat16 = the fp32 result rounded to nearest even) <- INT8
    paged decode attention of q_i8 [B, Hq, D] over the cache.

    u8_probs: UINT8 probability codes (0..255, sW = A / 255, s8 x u8 MMA) instead of 0..127."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    B, Hq, _ = q_i8.shape
    fn = lib().i8kv_int8_paged_decode_attn_u8p if u8_probs else lib().i8kv_int8_paged_decode_attn
    _check(fn(
        *_out(out), _ptr(q_i8, torch.int8, "q_i8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(block_tables, torch.int32, "block_tables"), _ptr(seq_lens, torch.int32, "seq_lens"),
        B, Hq, Hkv, D, BLOCK_SIZE, block_tables.shape[1], NB, float(softmax_scale), partition,
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)))


def int8_decode_step(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, workspace,
                     softmax_scale: float = 0.0, partition: int = PARTITION, stream=None):
    """One decode step in one launch: quantize and write each sequence's newest
    token (k_new, v_new bf16 [B, Hkv, D], at position seq_lens[b] - 1) into the
    cache, quantize q (bf16 [B, Hq, D]) and attend; out [B, Hq, D] fp32."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    B, Hq, _ = q.shape
    _check(lib().i8kv_int8_decode_step(
        *_out(out), _bf16(q, "q"), _bf16(k_new, "k_new"), _bf16(v_new, "v_new"),
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(block_tables, torch.int32, "block_tables"), _ptr(seq_lens, torch.int32, "seq_lens"),
        B, Hq, Hkv, D, BLOCK_SIZE, block_tables.shape[1], NB, float(softmax_scale), partition,
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)))


def int8_paged_decode_attn_noalloc(out, q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                                   softmax_scale: float = 0.0, partition: int = PARTITION, stream=None):
    """int8_paged_decode_attn for callers that cannot allocate: the merge scratch is
    the library's fixed device array (see include/i8kv.h for the size limit and
    why concurrent calls must not overlap)."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    B, Hq, _ = q_i8.shape
    _check(lib().i8kv_int8_paged_decode_attn_noalloc(
        _ptr(out, torch.float32, "out"), _ptr(q_i8, torch.int8, "q_i8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(block_tables, torch.int32, "block_tables"), _ptr(seq_lens, torch.int32, "seq_lens"),
        B, Hq, Hkv, D, BLOCK_SIZE, block_tables.shape[1], NB, float(softmax_scale), partition, _stream(stream)))


def bf16_paged_decode_attn(out, q, k_cache, v_cache, block_tables, seq_lens, workspace, softmax_scale: float = 0.0,
                           partition: int = PARTITION, stream=None):
    NB, Hkv, D = _cache_geom(k_cache, 8)
    B, Hq, _ = q.shape
    _check(lib().i8kv_bf16_paged_decode_attn(
        *_out(out), _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"),
        _ptr(block_tables, torch.int32, "block_tables"), _ptr(seq_lens, torch.int32, "seq_lens"),
        B, Hq, Hkv, D, BLOCK_SIZE, block_tables.shape[1], NB, float(softmax_scale), partition,
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)))


def bf16_kv_prefix_attn(out, q, k_cache, v_cache, block_table, history_len: int, workspace=None,
                        softmax_scale: float = 0.0, stream=None):
    """out [C, Hq, D] (float32 or bfloat16) <- the prefix chunk over the bf16 paged cache: bf16 q
    [C, Hq, D] (positions history_len ..) over every cached key 0 .. history_len + j (the chunk's
    own K/V already written by bf16_kv_write)."""
    NB, Hkv, D = _cache_geom(k_cache, 8)
    C, Hq, _ = q.shape
    if workspace is None:
        workspace = prefix_workspace(int(history_len), C, Hkv, D, device=out.device)
    _check(lib().i8kv_bf16_kv_prefix_attn(
        *_out(out), _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"),
        _ptr(block_table, torch.int32, "block_table"), int(history_len), C, Hq, Hkv, D, BLOCK_SIZE, NB,
        float(softmax_scale), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def debug_qk_i32(acc, q_i8, k_cache, block_tables, seq_lens, stream=None):
    """acc [B, Hq, max_len] int32 <- raw INT8 QK accumulators."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    B, Hq, _ = q_i8.shape
    _check(lib().i8kv_debug_qk_i32(
        _ptr(acc, torch.int32, "acc"), _ptr(q_i8, torch.int8, "q_i8"), _ptr(k_cache, torch.int8, "k_cache"),
        _ptr(block_tables, torch.int32, "block_tables"), _ptr(seq_lens, torch.int32, "seq_lens"),
        B, Hq, Hkv, D, BLOCK_SIZE, block_tables.shape[1], NB, acc.shape[2], _stream(stream)))


# ----------------------------------------------------------------------------- prefix
def prefix_workspace_bytes(history_len: int, chunk_len: int, Hkv: int, D: int) -> int:
    return int(lib().i8kv_prefix_workspace_bytes(history_len, chunk_len, Hkv, D))


def prefix_workspace(history_len: int, chunk_len: int, Hkv: int, D: int, device="cuda") -> torch.Tensor:
    """A prefix workspace (the f16 operand tiles; reusable by later calls on the same stream)."""
    n = prefix_workspace_bytes(history_len, chunk_len, Hkv, D)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def int8_prefix_attn(out, q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, history_len: int,
                     workspace=None, softmax_scale: float = 0.0, stream=None):
    """out [C, Hq, D] fp32 <- INT8 prefix-chunk attention of q_i8 [C, Hq, D] over history + chunk.

    workspace: a prefix_workspace(...) tensor; when None one is allocated for this call."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    C, Hq, _ = q_i8.shape
    if workspace is None:
        workspace = prefix_workspace(int(history_len), C, Hkv, D, device=out.device)
    _check(lib().i8kv_int8_prefix_attn(
        *_out(out), _ptr(q_i8, torch.int8, "q_i8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(block_table, torch.int32, "block_table"), int(history_len), C, Hq, Hkv, D, BLOCK_SIZE, NB,
        float(softmax_scale), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def debug_prefix_i32(q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, history_len: int,
                     workspace=None, softmax_scale: float = 0.0, stream=None):
    """The prefix kernel's raw integer contractions on int8_prefix_attn's arguments.
    Returns (s_acc int32 [C, Hq, H + C], wq uint8 [C, Hq, NG * 32], pv_acc int32
    [C, Hq, NG, D], out float32 [C, Hq, D]) with NG = ceil((H + C) / 32)."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    C, Hq, _ = q_i8.shape
    H = int(history_len)
    ng = (H + C + 31) // 32
    dev = q_i8.device
    s_acc = torch.empty((C, Hq, H + C), dtype=torch.int32, device=dev)
    wq = torch.empty((C, Hq, ng * 32), dtype=torch.uint8, device=dev)
    pv = torch.empty((C, Hq, ng, D), dtype=torch.int32, device=dev)
    out = torch.empty((C, Hq, D), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = prefix_workspace(H, C, Hkv, D, device=dev)
    _check(lib().i8kv_debug_prefix_i32(
        _ptr(s_acc), _ptr(wq), _ptr(pv), _ptr(out), _ptr(q_i8, torch.int8, "q_i8"),
        _ptr(q_scale, torch.float32, "q_scale"), _ptr(k_cache, torch.int8, "k_cache"),
        _ptr(v_cache, torch.int8, "v_cache"), _ptr(k_scale, torch.float32, "k_scale"),
        _ptr(v_scale, torch.float32, "v_scale"), _ptr(block_table, torch.int32, "block_table"), H, C, Hq, Hkv, D,
        BLOCK_SIZE, NB, float(softmax_scale), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))
    return s_acc, wq, pv, out


ROUTE_BF16, ROUTE_INT8 = 0, 1


def bf16_prefix_attn(out, q, k_chunk, v_chunk, history_len: int = 0, k_cache=None, v_cache=None, k_scale=None,
                     v_scale=None, block_table=None, workspace=None, softmax_scale: float = 0.0, stream=None):
    """out [C, Hq, D] fp32 <- high-precision chunk attention: bf16 q [C, Hq, D] over the INT8
    history (read back as code x scale) and the chunk's own bf16 k_chunk / v_chunk [C, Hkv, D]."""
    C, Hq, D = q.shape
    Hkv = k_chunk.shape[1]
    NB = 0
    if history_len > 0:
        NB, Hkv_c, D_c = _cache_geom(k_cache, 16)
        if (Hkv_c, D_c) != (Hkv, D):
            raise I8KVError(ERR_INVALID_ARG, "cache geometry does not match k_chunk")
    if workspace is None:
        workspace = prefix_workspace(int(history_len), C, Hkv, D, device=out.device)
    _check(lib().i8kv_bf16_prefix_attn(
        *_out(out), _bf16(q, "q"), _bf16(k_chunk, "k_chunk"), _bf16(v_chunk, "v_chunk"),
        _ptr(k_cache, torch.int8, "k_cache"), _ptr(v_cache, torch.int8, "v_cache"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(block_table, torch.int32, "block_table"), int(history_len), C, Hq, Hkv, D, BLOCK_SIZE, NB,
        float(softmax_scale), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def prefill_chunk(out, q, k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, block_table, history_len: int,
                  int8_min_history: int = 4096, q_i8=None, q_scale=None, workspace=None, softmax_scale: float = 0.0,
                  stream=None) -> int:
    """One routed prefill chunk: the producer writes the chunk's K/V to the INT8 cache, then the
    chunk runs on INT8 attention when history_len >= int8_min_history, else on the high-precision
    path.  Returns the route taken (ROUTE_BF16 or ROUTE_INT8)."""
    NB, Hkv, D = _cache_geom(k_cache, 16)
    C, Hq, _ = q.shape
    if workspace is None:
        workspace = prefix_workspace(int(history_len), C, Hkv, D, device=out.device)
    route = ctypes.c_int(-1)
    _check(lib().i8kv_prefill_chunk(
        *_out(out), _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"),
        _ptr(slot_mapping, torch.int32, "slot_mapping"), _ptr(k_cache, torch.int8, "k_cache"),
        _ptr(v_cache, torch.int8, "v_cache"), _ptr(k_scale, torch.float32, "k_scale"),
        _ptr(v_scale, torch.float32, "v_scale"), _ptr(block_table, torch.int32, "block_table"), int(history_len), C,
        Hq, Hkv, D, BLOCK_SIZE, NB, int(int8_min_history), float(softmax_scale), _ptr(q_i8, torch.int8, "q_i8"),
        _ptr(q_scale, torch.float32, "q_scale"), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        ctypes.byref(route), _stream(stream)))
    return int(route.value)
