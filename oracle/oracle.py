"""CPU oracle for INT8 KV-cache paged attention: ctypes wrapper and numpy references.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg import this module.  The CUDA library never
does, and this module imports nothing from it.

The arithmetic lives in ``i8kv_oracle.c`` (plain loops, cited there against the
pages).  This file builds that C file with gcc, marshals numpy arrays, and adds
two plain numpy definitions used to pin the C code from the outside:

* ``attention_fp64`` -- unquantized softmax attention in fp64 (the textbook
  definition; library matmul and exp as steps).
* ``group_form`` -- the closed form that the pages' partition / online-softmax
  schemes all reduce to ([PV] "gfx936 DCU上实现INT8 PV MMAC" §1-§2): since
  ``Wq = round(W / (max W / 127))`` does not change when every W of a group is
  scaled by the same positive factor, for any constant c

      O = sum_j (A_j/127) sum_{t in j} round(127 w_t / A_j) Vq_t  /  sum_t e^(s_t - c)
      with w_t = e^(s_t - c) sV_t and A_j = max_{t in j} w_t.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "i8kv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 32          # tokens per probability group ([PV] §1: one INT8 MMA K-step)
PARTITION = 256     # decode partition ([PV] §2.2)
KEY_TILE = 64       # prefix key tile; any multiple of GROUP gives the same result


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/liboracle.so (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # I8KV_ORACLE_LIB points the wrapper at another build of i8kv_oracle.c
            # (the mutation tests plant known mistakes in a copy and load it here).
            path = os.environ.get("I8KV_ORACLE_LIB")
            if not path:
                path = build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_quantize_vector.argtypes = [P, I, P, P]
            lib.orc_quantize_vector.restype = None
            lib.orc_kv_quant_write.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, I, P, P]
            lib.orc_kv_rope_quant_write.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, I, P, P, P, P, I, I, P, P,
                                                    ctypes.c_float, P, P, P]
            lib.orc_qk_i32.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I]
            lib.orc_decode_attn.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float,
                                            I, I, I, I, I, I, P, P, P, P, I]
            lib.orc_prefix_attn.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, I,
                                            P, I, I, I]
            lib.orc_bf16_kv_write.argtypes = [P, P, P, I, I, I, I, P, P]
            lib.orc_bf16_prefix_attn.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, I,
                                                 I]
            lib.orc_bf16_decode_attn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_double, I]
            lib.orc_bf16_kv_prefix_attn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, I, I]
            for name in ("orc_kv_quant_write", "orc_kv_rope_quant_write", "orc_qk_i32", "orc_decode_attn", "orc_prefix_attn",
                         "orc_bf16_kv_write", "orc_bf16_decode_attn", "orc_bf16_prefix_attn",
                         "orc_bf16_kv_prefix_attn", "orc_max_threads"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a: np.ndarray) -> np.ndarray:
    """bf16 payload as raw uint16 bits (accepts uint16 already)."""
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 arrays are passed as uint16 bit patterns"
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (status {rc})")


def max_threads() -> int:
    return int(_load().orc_max_threads())


# --------------------------------------------------------------------------- producer
def quantize_vector(x_bf16: np.ndarray):
    """[KV] §2.1: returns (q int8 [n], scale float32)."""
    x = _u16(x_bf16).ravel()
    q = np.empty(x.size, np.int8)
    s = np.empty(1, np.float32)
    _load().orc_quantize_vector(_p(x), x.size, _p(q), _p(s))
    return q, s[0]


def kv_quant_write(k, v, slot_mapping, num_blocks, block_size, q=None, k_cache=None, v_cache=None,
                   k_scale=None, v_scale=None):
    """[KV] §2.2-§2.3 producer.  k, v: uint16 [T, Hkv, D]; q: uint16 [T, Hq, D] or None.

    Returns dict with k_cache [NB,Hkv,D/16,bs,16] i8, v_cache [NB,Hkv,D,bs] i8,
    k_scale/v_scale [NB,bs,Hkv] f32 and, with q, q_i8 [T,Hq,D] / q_scale [T,Hq].
    Existing caches may be passed in to be updated in place."""
    k, v = _u16(k), _u16(v)
    T, Hkv, D = k.shape
    bs = block_size
    if k_cache is None:
        k_cache = np.zeros((num_blocks, Hkv, D // 16, bs, 16), np.int8)
        v_cache = np.zeros((num_blocks, Hkv, D, bs), np.int8)
        k_scale = np.zeros((num_blocks, bs, Hkv), np.float32)
        v_scale = np.zeros((num_blocks, bs, Hkv), np.float32)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    out = dict(k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale)
    Hq = 0
    q_i8 = q_scale = None
    if q is not None:
        q = _u16(q)
        Hq = q.shape[1]
        q_i8 = np.empty(q.shape, np.int8)
        q_scale = np.empty(q.shape[:2], np.float32)
        out.update(q_i8=q_i8, q_scale=q_scale)
    rc = _load().orc_kv_quant_write(_p(k), _p(v), _p(slots), T, Hkv, D, bs, _p(k_cache), _p(v_cache),
                                    _p(k_scale), _p(v_scale), _p(q), Hq, _p(q_i8), _p(q_scale))
    _check(rc, "kv_quant_write")
    return out


BAD_POSITION = 2   # orc_kv_rope_quant_write: some token's position was outside the table


def kv_rope_quant_write(k, v, slot_mapping, num_blocks, block_size, positions=None, cos_sin=None, rotary_dim=0,
                        q=None, q_norm_weight=None, k_norm_weight=None, eps=1e-6, quantize_q=True,
                        q_out=False, k_out=False, k_smooth=None):
    """Fused producer: optional Q/K RMSNorm, RoPE (rotate-half on the first
    ``rotary_dim`` dims, table ``cos_sin`` float32 [max_position, rotary_dim]),
    then the [KV] §2.1 quantization and the paged scatter of kv_quant_write.

    Returns the kv_quant_write dict plus ``q_out`` / ``k_out`` (bf16 bits of the
    transformed Q / K) when asked, and ``status`` (0, or BAD_POSITION when some
    token was skipped because its position lay outside the table).  k_smooth
    (float32 [Hkv, D], optional): per-channel K smoothing factors -- K is
    multiplied by RN(1/s), Q by s of its KV head, before the quantization."""
    k, v = _u16(k), _u16(v)
    T, Hkv, D = k.shape
    bs = block_size
    out = dict(k_cache=np.zeros((num_blocks, Hkv, D // 16, bs, 16), np.int8),
               v_cache=np.zeros((num_blocks, Hkv, D, bs), np.int8),
               k_scale=np.zeros((num_blocks, bs, Hkv), np.float32),
               v_scale=np.zeros((num_blocks, bs, Hkv), np.float32))
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
    cs = None if cos_sin is None else np.ascontiguousarray(cos_sin, dtype=np.float32)
    max_pos = 0 if cs is None else cs.shape[0]
    if cs is not None:
        assert cs.shape[1] == rotary_dim, "cos_sin rows must hold rotary_dim values"
    Hq = 0
    q_i8 = q_scale = qo = None
    if q is not None:
        q = _u16(q)
        Hq = q.shape[1]
        if quantize_q:
            q_i8 = np.zeros(q.shape, np.int8)
            q_scale = np.zeros(q.shape[:2], np.float32)
            out.update(q_i8=q_i8, q_scale=q_scale)
        if q_out:
            qo = np.zeros(q.shape, np.uint16)
            out["q_out"] = qo
    ko = None
    if k_out:
        ko = np.zeros(k.shape, np.uint16)
        out["k_out"] = ko
    qw = None if q_norm_weight is None else _u16(q_norm_weight)
    kw = None if k_norm_weight is None else _u16(k_norm_weight)
    ks = None if k_smooth is None else np.ascontiguousarray(k_smooth, np.float32)
    rc = _load().orc_kv_rope_quant_write(_p(k), _p(v), _p(slots), T, Hkv, D, bs, _p(out["k_cache"]),
                                         _p(out["v_cache"]), _p(out["k_scale"]), _p(out["v_scale"]), _p(q), Hq,
                                         _p(q_i8), _p(q_scale), _p(pos), _p(cs), max_pos, rotary_dim, _p(qw),
                                         _p(kw), float(eps), _p(qo), _p(ko), _p(ks))
    if rc not in (0, BAD_POSITION):
        _check(rc, "kv_rope_quant_write")
    out["status"] = rc
    return out


# --------------------------------------------------------------------------- QK
def qk_i32(q_i8, k_cache, block_tables, seq_lens, Hkv, block_size, max_len=None):
    """INT32 QK accumulators [B, Hq, max_len]."""
    q_i8 = np.ascontiguousarray(q_i8, np.int8)
    B, Hq, D = q_i8.shape
    bt = np.ascontiguousarray(block_tables, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    if max_len is None:
        max_len = int(sl.max()) if sl.size else 0
    acc = np.zeros((B, Hq, max_len), np.int32)
    rc = _load().orc_qk_i32(_p(acc), _p(q_i8), _p(k_cache), _p(bt), _p(sl), B, Hq, Hkv, D, block_size,
                            bt.shape[1], max_len)
    _check(rc, "qk_i32")
    return acc


# --------------------------------------------------------------------------- decode
def decode_attn(q_i8, q_scale, cache, block_tables, seq_lens, block_size, softmax_scale=None,
                partition=PARTITION, group=GROUP, fp32_decisions=True, nthreads=0, trace=None, pmax=127):
    """Literal decode ([PV] §2.2): 256-token partitions, LSE merge.  Returns out [B,Hq,D] fp64.

    pmax: the probability code range, 127 (signed INT8, the pages' kernels) or
    255 (UINT8 probabilities, [PV] §6).
    trace=(b, h) additionally returns per-token arrays W, Wq, sW, c (see the C file)."""
    lib = _load()
    q_i8 = np.ascontiguousarray(q_i8, np.int8)
    B, Hq, D = q_i8.shape
    Hkv = cache["k_cache"].shape[1]
    qs = np.ascontiguousarray(q_scale, np.float32)
    bt = np.ascontiguousarray(block_tables, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    out = np.empty((B, Hq, D), np.float64)
    tb, th = (-1, -1) if trace is None else trace
    tr = None
    if trace is not None:
        L = int(sl[tb])
        tr = dict(W=np.zeros(L), Wq=np.zeros(L, np.int16), sW=np.zeros(L), c=np.zeros(L))
    rc = lib.orc_decode_attn(_p(out), _p(q_i8), _p(qs), _p(cache["k_cache"]), _p(cache["v_cache"]),
                             _p(cache["k_scale"]), _p(cache["v_scale"]), _p(bt), _p(sl), B, Hq, Hkv, D,
                             block_size, bt.shape[1], softmax_scale, partition, group, int(fp32_decisions),
                             nthreads, tb, th, _p(tr["W"]) if tr else None, _p(tr["Wq"]) if tr else None,
                             _p(tr["sW"]) if tr else None, _p(tr["c"]) if tr else None, int(pmax))
    _check(rc, "decode_attn")
    return (out, tr) if trace is not None else out


# --------------------------------------------------------------------------- prefix
def prefix_attn(q_i8, q_scale, cache, block_table, history_len, block_size, softmax_scale=None, rows=None,
                key_tile=KEY_TILE, group=GROUP, fp32_decisions=True, nthreads=0):
    """Literal prefix chunk ([PV] §2.1): one online softmax over history + causal chunk.

    q_i8 [C,Hq,D]; rows selects chunk rows.  Returns out [len(rows) or C, Hq, D] fp64."""
    lib = _load()
    q_i8 = np.ascontiguousarray(q_i8, np.int8)
    C, Hq, D = q_i8.shape
    Hkv = cache["k_cache"].shape[1]
    qs = np.ascontiguousarray(q_scale, np.float32)
    bt = np.ascontiguousarray(block_table, np.int32).ravel()
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    nrows = C if r is None else r.size
    out = np.empty((nrows, Hq, D), np.float64)
    rc = lib.orc_prefix_attn(_p(out), _p(q_i8), _p(qs), _p(cache["k_cache"]), _p(cache["v_cache"]),
                             _p(cache["k_scale"]), _p(cache["v_scale"]), _p(bt), history_len, C, Hq, Hkv, D,
                             block_size, softmax_scale, key_tile, group, _p(r), nrows, int(fp32_decisions),
                             nthreads)
    _check(rc, "prefix_attn")
    return out


def bf16_prefix_attn(q, k_chunk, v_chunk, cache, block_table, history_len, block_size, softmax_scale=None,
                     rows=None, nthreads=0):
    """High-precision chunk attention ([KV] §3.1, §4 routing): chunk rows of q
    (uint16 bf16 [C,Hq,D]) over the INT8 history read back as code * scale and
    the chunk's own bf16 k_chunk / v_chunk [C,Hkv,D], causal.  fp64 out
    [len(rows) or C, Hq, D].  cache / block_table may be None when
    history_len == 0."""
    q, kc, vc = _u16(q), _u16(k_chunk), _u16(v_chunk)
    C, Hq, D = q.shape
    Hkv = kc.shape[1]
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    nrows = C if r is None else r.size
    out = np.empty((nrows, Hq, D), np.float64)
    c = cache or {}
    bt = None if block_table is None else np.ascontiguousarray(block_table, np.int32).ravel()
    rc = _load().orc_bf16_prefix_attn(_p(out), _p(q), _p(kc), _p(vc), _p(c.get("k_cache")), _p(c.get("v_cache")),
                                      _p(c.get("k_scale")), _p(c.get("v_scale")), _p(bt), history_len, C, Hq, Hkv,
                                      D, block_size, float(softmax_scale), _p(r), nrows, nthreads)
    _check(rc, "bf16_prefix_attn")
    return out


# --------------------------------------------------------------------------- BF16-KV comparison
def bf16_kv_write(k, v, slot_mapping, num_blocks, block_size, k_cache=None, v_cache=None):
    """BF16 paged cache: K [NB,Hkv,D/8,bs,8], V [NB,Hkv,D,bs], uint16 bit patterns."""
    k, v = _u16(k), _u16(v)
    T, Hkv, D = k.shape
    if k_cache is None:
        k_cache = np.zeros((num_blocks, Hkv, D // 8, block_size, 8), np.uint16)
        v_cache = np.zeros((num_blocks, Hkv, D, block_size), np.uint16)
    slots = np.ascontiguousarray(slot_mapping, np.int32)
    rc = _load().orc_bf16_kv_write(_p(k), _p(v), _p(slots), T, Hkv, D, block_size, _p(k_cache), _p(v_cache))
    _check(rc, "bf16_kv_write")
    return dict(k_cache=k_cache, v_cache=v_cache)


def bf16_decode_attn(q, cache, block_tables, seq_lens, block_size, softmax_scale=None, nthreads=0):
    """fp64 softmax attention over the bf16 paged cache.  q: uint16 [B,Hq,D]."""
    q = _u16(q)
    B, Hq, D = q.shape
    Hkv = cache["k_cache"].shape[1]
    bt = np.ascontiguousarray(block_tables, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    out = np.empty((B, Hq, D), np.float64)
    rc = _load().orc_bf16_decode_attn(_p(out), _p(q), _p(cache["k_cache"]), _p(cache["v_cache"]), _p(bt),
                                      _p(sl), B, Hq, Hkv, D, block_size, bt.shape[1], float(softmax_scale),
                                      nthreads)
    _check(rc, "bf16_decode_attn")
    return out


def bf16_kv_prefix_attn(q, cache, block_table, history_len, block_size, softmax_scale=None, rows=None,
                        nthreads=0):
    """BF16-KV comparison of the prefix chunk: chunk rows of q (uint16 bf16
    [C,Hq,D]) over keys 0 .. history_len + j of the bf16 paged cache (history
    and chunk alike), causal, plain softmax in fp64.  Out [len(rows) or C, Hq, D]."""
    q = _u16(q)
    C, Hq, D = q.shape
    Hkv = cache["k_cache"].shape[1]
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    nrows = C if r is None else r.size
    out = np.empty((nrows, Hq, D), np.float64)
    bt = np.ascontiguousarray(block_table, np.int32).ravel()
    rc = _load().orc_bf16_kv_prefix_attn(_p(out), _p(q), _p(cache["k_cache"]), _p(cache["v_cache"]), _p(bt),
                                         history_len, C, Hq, Hkv, D, block_size, float(softmax_scale), _p(r), nrows,
                                         nthreads)
    _check(rc, "bf16_kv_prefix_attn")
    return out


# --------------------------------------------------------------------------- numpy definitions
def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention_fp64(q, k, v, kv_lens, softmax_scale=None):
    """Plain softmax attention in fp64.

    q [Nq,Hq,D], k/v [L,Hkv,D] (float64), kv_lens [Nq]: query row r sees keys
    0 .. kv_lens[r]-1.  Query head h reads KV head h // (Hq // Hkv)."""
    Nq, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    out = np.zeros((Nq, Hq, D))
    for r in range(Nq):
        n = int(kv_lens[r])
        if n == 0:
            continue
        for h in range(Hq):
            s = k[:n, h // G, :] @ q[r, h] * softmax_scale
            p = np.exp(s - s.max())
            out[r, h] = (p / p.sum()) @ v[:n, h // G, :]
    return out


def group_form(scores: np.ndarray, sV: np.ndarray, Vq: np.ndarray, group: int = GROUP, pmax: int = 127) -> np.ndarray:
    """Closed group form for one query row in fp64 (see module docstring; pmax
    replaces 127 for the UINT8 probability codes).

    scores [L] fp64, sV [L], Vq [L, D] int -> O [D]."""
    c = scores.max()
    e = np.exp(scores - c)
    w = e * sV
    num = np.zeros(Vq.shape[1])
    for j0 in range(0, scores.size, group):
        wj = w[j0:j0 + group]
        A = wj.max()
        if A == 0:
            continue
        wq = np.rint(wj / (A / pmax))
        num += (A / pmax) * (wq @ Vq[j0:j0 + group].astype(np.float64))
    return num / e.sum()
