"""The C-ABI library builds, loads and exports every entry point include/i8kv.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from int8_kv_cache_token_gb300 import build
    return ctypes.CDLL(build.build())


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "i8kv.h"), encoding="utf-8").read()
    return sorted(set(re.findall(r"^(?:i8kv_status|size_t|int)\s+(i8kv_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/i8kv.h but not exported"


def test_version(lib):
    assert lib.i8kv_version() == 100


def _last_error(lib):
    buf = ctypes.create_string_buffer(256)
    lib.i8kv_last_error(buf, 256)
    return buf.value.decode()


def test_argument_checks_without_gpu(lib):
    P = ctypes.c_void_p
    # unsupported block size
    f = lib.i8kv_kv_quant_write
    f.restype = ctypes.c_int
    assert f(P(16), P(16), P(16), 4, 4, 256, 8, 10, P(16), P(16), P(16), P(16), None, 0, None, None, None) == 2
    assert "block_size" in _last_error(lib)
    # unsupported head_dim
    assert f(P(16), P(16), P(16), 4, 4, 64, 16, 10, P(16), P(16), P(16), P(16), None, 0, None, None, None) == 2
    # null pointers with T > 0
    assert f(None, P(16), P(16), 4, 4, 256, 16, 10, P(16), P(16), P(16), P(16), None, 0, None, None, None) == 1
    # misaligned cache pointer
    assert f(P(16), P(16), P(16), 4, 4, 256, 16, 10, P(17), P(16), P(16), P(16), None, 0, None, None, None) == 1
    assert "aligned" in _last_error(lib)
    # T == 0 is a no-op
    assert f(None, None, None, 0, 4, 256, 16, 10, None, None, None, None, None, 0, None, None, None) == 0
    # decode: Hq not a multiple of Hkv, G > 8, partition != 256
    d = lib.i8kv_int8_paged_decode_attn
    d.restype = ctypes.c_int
    d.argtypes = [P, ctypes.c_int] + [P] * 8 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int, P,
                                                                   ctypes.c_size_t, P]
    args = [P(16)] * 8
    assert d(P(16), 0, *args, 1, 10, 4, 256, 16, 8, 10, 0.0, 256, P(16), 1 << 20, None) == 1
    assert d(P(16), 0, *args, 1, 72, 4, 256, 16, 8, 10, 0.0, 256, P(16), 1 << 20, None) == 2
    assert d(P(16), 0, *args, 1, 24, 4, 256, 16, 8, 10, 0.0, 512, P(16), 1 << 20, None) == 2
    assert "partition" in _last_error(lib)
    # the output type: fp32 (0) or bf16 (1), 16-byte aligned
    assert d(P(16), 2, *args, 1, 24, 4, 256, 16, 8, 10, 0.0, 256, P(16), 1 << 20, None) == 1
    assert "out_dtype" in _last_error(lib)
    assert d(P(8), 1, *args, 1, 24, 4, 256, 16, 8, 10, 0.0, 256, P(16), 1 << 20, None) == 1
    assert "out must be 16-byte aligned" in _last_error(lib)
    # decode step: the new token's K/V are required and 16-byte aligned
    st = lib.i8kv_int8_decode_step
    st.restype = ctypes.c_int
    st.argtypes = [P, ctypes.c_int] + [P] * 9 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int, P,
                                                                    ctypes.c_size_t, P]
    base = [P(16), 0] + [P(16)] * 9
    assert st(P(16), 0, P(16), None, P(16), *([P(16)] * 6), 1, 24, 4, 256, 16, 8, 10, 0.0, 256, P(16), 1 << 20,
              None) == 1
    assert "k_new" in _last_error(lib)
    assert st(P(16), 0, P(16), P(24), P(16), *([P(16)] * 6), 1, 24, 4, 256, 16, 8, 10, 0.0, 256, P(16), 1 << 20,
              None) == 1
    assert "aligned" in _last_error(lib)
    assert st(*base, 1, 24, 4, 64, 16, 8, 10, 0.0, 256, P(16), 1 << 20, None) == 2
    # prefix: chunk_len == 0 is a no-op; negative history rejected
    pf = lib.i8kv_int8_prefix_attn
    pf.restype = ctypes.c_int
    pf.argtypes = [P, ctypes.c_int] + [P] * 7 + [ctypes.c_int] * 7 + [ctypes.c_float, P, ctypes.c_size_t, P]
    pa = [P(16), 0] + [P(16)] * 7
    assert pf(*pa, 100, 0, 24, 4, 256, 16, 10, 0.0, None, 0, None) == 0
    assert pf(*pa, -1, 5, 24, 4, 256, 16, 10, 0.0, P(16), 1 << 30, None) == 1
    assert pf(P(16), 5, *([P(16)] * 7), 100, 5, 24, 4, 256, 16, 10, 0.0, P(16), 1 << 30, None) == 1
    assert "out_dtype" in _last_error(lib)
    # the workspace: size from i8kv_prefix_workspace_bytes, checked before any launch
    wb = lib.i8kv_prefix_workspace_bytes
    wb.restype = ctypes.c_size_t
    wb.argtypes = [ctypes.c_int] * 4
    need = wb(100, 5, 4, 256)
    tiles = 4 * ((100 + 5 + 31) // 32) * (2 * 32 * 256 * 2 + 256)
    part_slot = 128 * (256 + 4) * 4  # the split parts' (o, m, l) rows, 2 per SM
    assert need > tiles and (need - tiles) % (2 * part_slot) == 0
    assert wb(100, 5, 4, 64) == 0
    assert pf(*pa, 100, 5, 24, 4, 256, 16, 10, 0.0, None, need, None) == 3
    assert pf(*pa, 100, 5, 24, 4, 256, 16, 10, 0.0, P(16), need - 1, None) == 3
    assert "workspace" in _last_error(lib)
    assert pf(*pa, 100, 5, 24, 4, 256, 16, 10, 0.0, P(24), need, None) == 1


def test_rope_producer_argument_checks_without_gpu(lib):
    P = ctypes.c_void_p
    f = lib.i8kv_kv_rope_quant_write
    f.restype = ctypes.c_int
    f.argtypes = ([P, P, P] + [ctypes.c_int] * 5 + [P] * 5 + [ctypes.c_int] + [P] * 4 + [ctypes.c_int] * 2 +
                  [P, P, ctypes.c_float, P, P, P, P])

    def call(rd=128, pos=P(16), cs=P(16), max_pos=64, qw=None, kw=None, eps=1e-6, q=None, q_i8=None, q_scale=None,
             q_out=None, k_out=None, T=4, Hq=8, smooth=None):
        return f(P(16), P(16), P(16), T, 4, 128, 16, 10, P(16), P(16), P(16), P(16), q, Hq, q_i8, q_scale, pos, cs,
                 max_pos, rd, qw, kw, eps, q_out, k_out, smooth, None)

    assert call(rd=48) == 2 and "multiple of 32" in _last_error(lib)
    assert call(rd=256) == 1 and "rotary_dim" in _last_error(lib)
    assert call(pos=None) == 1 and "positions" in _last_error(lib)
    assert call(cs=P(24)) == 1 and "cos_sin" in _last_error(lib)
    assert call(max_pos=0) == 1
    assert call(kw=P(16), eps=0.0) == 1 and "norm_eps" in _last_error(lib)
    assert call(kw=P(18)) == 1 and "aligned" in _last_error(lib)
    assert call(q=P(16), q_i8=P(16)) == 1 and "q_scale" in _last_error(lib)
    assert call(q=P(16)) == 1 and "q_out" in _last_error(lib)
    assert call(q_out=P(16)) == 1 and "without q" in _last_error(lib)
    assert call(k_out=P(8)) == 1 and "aligned" in _last_error(lib)
    assert call(smooth=P(20)) == 1 and "k_smooth" in _last_error(lib)
    assert call(smooth=P(16), q=P(16), q_i8=P(16), q_scale=P(16), Hq=6) == 1 and "multiple" in _last_error(lib)
    # rotary_dim 0 needs no table; T == 0 is a no-op after the shape checks
    assert call(rd=0, pos=None, cs=None, max_pos=0, T=0) == 0


def test_prefill_route_decision_without_gpu(lib):
    # i8kv_prefill_chunk reports its route before any launch: INT8 once the
    # history reaches int8_min_history, the high-precision path below it; a
    # zero-length chunk then returns without touching the device.
    P = ctypes.c_void_p
    f = lib.i8kv_prefill_chunk
    f.restype = ctypes.c_int
    f.argtypes = ([P, ctypes.c_int] + [P] * 9 + [ctypes.c_int] * 8 +
                  [ctypes.c_float, P, P, P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int), P])

    def route(history, threshold):
        r = ctypes.c_int(-1)
        st = f(P(16), 0, *([P(16)] * 9), history, 0, 24, 4, 256, 16, 10, threshold, 0.0, None, None, None, 0,
               ctypes.byref(r), None)
        assert st == 0
        return r.value

    BF16, INT8 = 0, 1  # I8KV_ROUTE_BF16, I8KV_ROUTE_INT8
    assert route(0, 4096) == BF16 and route(4095, 4096) == BF16
    assert route(4096, 4096) == INT8 and route(20000, 4096) == INT8
    assert route(0, 0) == INT8  # threshold 0: every chunk INT8
    # bad shapes are rejected before the route is used
    r = ctypes.c_int(-1)
    assert f(P(16), 0, *([P(16)] * 9), 10, 4, 24, 5, 256, 16, 10, 0, 0.0, None, None, None, 0, ctypes.byref(r),
             None) != 0
