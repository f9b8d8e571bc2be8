"""GPU parity of the high-precision chunk path (first prefill chunk, and chunks
below the routing threshold) and of the routed prefill entry.

The kernel rounds the dequantized history K/V and the probabilities p~ to bf16
for the tensor-core MMAs, so it is compared with the oracle's fp64 attention
within a bound derived from those roundings: p~ and a history V value each move
by at most 2^-9 of themselves, so an output moves by at most 2^-8 max|V|; a
history K rounding moves a score by about 2^-9 |q.k| / sqrt(D), allowed for by
a further 1e-3.  The mean error must also stay below 1e-3 (random roundings
average out; a systematic slip would not)."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host, gpu_quantize_rows

pytestmark = pytest.mark.gpu


def _check_close(got, ref, v_max, what):
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * v_max + 1e-3
    assert np.isfinite(got).all(), what
    assert err.max() <= bound and err.mean() <= 1e-3, \
        f"{what}: max-abs {err.max():.3e} (bound {bound:.3e}), mean-abs {err.mean():.3e}"
    return err.max()


def _run_bf16(w: wl.PrefixWorkload, rows=None):
    k, v = w.kv()
    q = w.q()
    H, C = w.history, w.chunk
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    if H:
        i8.kv_quant_write(dev(k[:H]), dev(v[:H]), dev(w.slots(0, H)), **cache)
    out = torch.full((C, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    i8.bf16_prefix_attn(out, dev(q), dev(k[H:]), dev(v[H:]), H, cache["k_cache"], cache["v_cache"],
                        cache["k_scale"], cache["v_scale"], dev(w.block_table))
    got = host(out)
    assert i8.device_error() == 0
    oc = orc.kv_quant_write(k[:H], v[:H], w.slots(0, H), w.num_blocks, w.block_size) if H else None
    ref = orc.bf16_prefix_attn(q, k[H:], v[H:], oc, w.block_table, H, w.block_size, rows=rows)
    if rows is not None:
        got = got[rows]
    return _check_close(got, ref, np.abs(wl.bf16_values(v)).max(), w.name)


@pytest.mark.parametrize("H,C", [(0, 1), (0, 37), (0, 300), (100, 37), (256, 70), (1000, 200)])
@pytest.mark.parametrize("Hq,Hkv,D", [(24, 4, 256), (32, 8, 128), (8, 1, 256)])
def test_bf16_prefix_small(H, C, Hq, Hkv, D):
    _run_bf16(wl.PrefixWorkload("b", Hq, Hkv, D, H, C, seed=H + C + D))


def test_bf16_first_chunk_full_size_sampled_rows():
    # the pages' first chunk: no history, 4096 new tokens, 24 / 4 heads, head_dim 256
    w = wl.PrefixWorkload("first4k", 24, 4, 256, 0, 4096, seed=5)
    rows = np.array([0, 1, 31, 32, 127, 128, 1000, 2047, 2048, 4000, 4095], np.int32)
    _run_bf16(w, rows=rows)


def test_bf16_prefix_single_key_returns_value():
    # independent of the oracle: the first query of a first chunk sees one key,
    # so its output is that key's V row (bf16 p~ = 1 exactly)
    w = wl.PrefixWorkload("one", 8, 2, 128, 0, 3, seed=1)
    k, v = w.kv()
    out = torch.empty((3, 8, 128), dtype=torch.float32, device="cuda")
    i8.bf16_prefix_attn(out, dev(w.q()), dev(k), dev(v))
    got = host(out)[0]
    expect = np.repeat(wl.bf16_values(v[0]), 4, axis=0)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("H,thr", [(0, 4096), (512, 4096), (4096, 4096), (512, 0)])
def test_prefill_chunk_routes(H, thr):
    # The routed entry writes the chunk to the INT8 cache (bit-exact with the
    # oracle producer) and returns exactly what the chosen path returns.
    C, Hq, Hkv, D = 130, 8, 2, 128
    w = wl.PrefixWorkload("route", Hq, Hkv, D, H, C, seed=H + 7)
    k, v = w.kv()
    q = w.q()
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    if H:
        i8.kv_quant_write(dev(k[:H]), dev(v[:H]), dev(w.slots(0, H)), **cache)
    out = torch.empty((C, Hq, D), dtype=torch.float32, device="cuda")
    q_i8 = torch.empty((C, Hq, D), dtype=torch.int8, device="cuda")
    q_s = torch.empty((C, Hq), dtype=torch.float32, device="cuda")
    bt = dev(w.block_table)
    route = i8.prefill_chunk(out, dev(q), dev(k[H:]), dev(v[H:]), dev(w.slots(H)), cache["k_cache"],
                             cache["v_cache"], cache["k_scale"], cache["v_scale"], bt, H, int8_min_history=thr,
                             q_i8=q_i8, q_scale=q_s)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    assert route == (i8.ROUTE_INT8 if H >= thr else i8.ROUTE_BF16)
    oc = orc.kv_quant_write(k, v, w.slots(), w.num_blocks, w.block_size)
    for key in ("k_cache", "v_cache", "k_scale", "v_scale"):
        g, r = host(cache[key]), oc[key]
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        assert np.array_equal(g, r), key
    direct = torch.empty_like(out)
    if route == i8.ROUTE_INT8:
        qi, qs = gpu_quantize_rows(q, Hkv, cache)
        i8.int8_prefix_attn(direct, qi, qs, cache["k_cache"], cache["v_cache"], cache["k_scale"], cache["v_scale"],
                            bt, H)
        ref = orc.prefix_attn(host(qi), host(qs), oc, w.block_table, H, w.block_size)
    else:
        i8.bf16_prefix_attn(direct, dev(q), dev(k[H:]), dev(v[H:]), H, cache["k_cache"], cache["v_cache"],
                            cache["k_scale"], cache["v_scale"], bt)
        ref = orc.bf16_prefix_attn(q, k[H:], v[H:], oc, w.block_table, H, w.block_size)
    assert torch.equal(out, direct)
    if route == i8.ROUTE_INT8:
        assert np.abs(host(out) - ref).max() <= 2e-3  # the INT8 path's own tolerance
    else:
        _check_close(host(out), ref, np.abs(wl.bf16_values(v)).max(), "routed bf16")


def test_bf16_prefix_split_tail_blocks():
    # 176 row blocks (700 tokens, 32 / 8 heads, head_dim 128): the tail is split
    _run_bf16(wl.PrefixWorkload("bsplit", 32, 8, 128, 300, 700, seed=11))
