"""GPU parity of the high-precision chunk path (first prefill chunk, and chunks
below the routing threshold) and of the routed prefill entry.

Per-element bound, from the arithmetic the kernel documents.  It reads a
history key or value back from the INT8 cache as bf16(code x scale) (the fp32
product rounded to nearest-even bf16), while the oracle uses code x scale
exactly; so the reference for the kernel's own rounding is A_r, fp64 softmax
attention over exactly those bf16 values, computed here in numpy.  The kernel
then rounds each p~ = exp(s - m) to bf16 for the P x V product (relative error
<= 2^-9) while l sums the unrounded fp32 p~, which moves output element (j, d)
by at most 2^-9 sum_t p_t |v_td|; the bound allows 2^-8 of it.  fp32 scores,
ex2 and accumulation add at most 3e-4.  So, element by element,

    |out - oracle| <= |oracle - A_r| + 2^-8 sum_t p_t |v_td| + 3e-4

with p the softmax weights of A_r.  The history term |oracle - A_r| is computed,
not bounded: it is the documented bf16 read-back of the INT8 history."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host, gpu_quantize_rows
from tests.helpers import gather_int8

pytestmark = pytest.mark.gpu


def _bf16_round(x32: np.ndarray) -> np.ndarray:
    return wl.bf16_values(wl.bf16_bits(x32)).astype(np.float64)


def _kernel_reference(w, q, k, v, oc, rows):
    """A_r [rows, Hq, D] and the bound's P-rounding term 2^-8 sum_t p_t |v_td|."""
    H, C, Hq, Hkv, D = w.history, w.chunk, w.Hq, w.Hkv, w.D
    G = Hq // Hkv
    T = H + C
    Kv = np.empty((T, Hkv, D))
    Vv = np.empty((T, Hkv, D))
    if H:
        Kt, Vt, sK, sV = gather_int8(oc, w.block_table, H, Hkv, D)
        # fp32 product code x scale, then RNE to bf16 (the kernel's read-back)
        Kv[:H] = _bf16_round(Kt.astype(np.float32) * sK[:, :, None].astype(np.float32))
        Vv[:H] = _bf16_round(Vt.astype(np.float32) * sV[:, :, None].astype(np.float32))
    Kv[H:] = wl.bf16_values(k[H:])
    Vv[H:] = wl.bf16_values(v[H:])
    qv = wl.bf16_values(q).astype(np.float64)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    rows = np.arange(C) if rows is None else np.asarray(rows)
    ref = np.empty((rows.size, Hq, D))
    pterm = np.empty((rows.size, Hq, D))
    for i, j in enumerate(rows):
        n = H + j + 1
        for h in range(Hq):
            s = Kv[:n, h // G, :] @ qv[j, h] * scale
            p = np.exp(s - s.max())
            p /= p.sum()
            ref[i, h] = p @ Vv[:n, h // G, :]
            pterm[i, h] = 2.0 ** -8 * (p @ np.abs(Vv[:n, h // G, :]))
    return ref, pterm


def _check_close(got, oracle_out, a_r, pterm, what):
    err = np.abs(got - oracle_out)
    bound = np.abs(oracle_out - a_r) + pterm + 3e-4
    assert np.isfinite(got).all(), what
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements past the bound, worst at "
                           f"{np.unravel_index(np.argmax(err - bound), err.shape)}: "
                           f"err {err.max():.3e}, bound there {bound.flat[np.argmax(err - bound)]:.3e}")
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
    a_r, pterm = _kernel_reference(w, q, k, v, oc, rows)
    return _check_close(got, ref, a_r, pterm, w.name), (got, ref, a_r, pterm)


@pytest.mark.parametrize("H,C", [(0, 1), (0, 37), (0, 300), (100, 37), (256, 70), (1000, 200)])
@pytest.mark.parametrize("Hq,Hkv,D", [(24, 4, 256), (32, 8, 128), (8, 1, 256)])
def test_bf16_prefix_small(H, C, Hq, Hkv, D):
    _run_bf16(wl.PrefixWorkload("b", Hq, Hkv, D, H, C, seed=H + C + D))


def test_bf16_first_chunk_full_size_sampled_rows():
    # the pages' first chunk: no history, 4096 new tokens, 24 / 4 heads, head_dim 256
    w = wl.PrefixWorkload("first4k", 24, 4, 256, 0, 4096, seed=5)
    rows = np.array([0, 1, 31, 32, 127, 128, 1000, 2047, 2048, 4000, 4095], np.int32)
    _run_bf16(w, rows=rows)


def test_bf16_prefix_bound_catches_a_one_row_slip():
    # The bound is tight enough to fail on a 1e-2 error confined to one row
    # (planted here in the GPU output, after the kernel ran).
    w = wl.PrefixWorkload("plant", 24, 4, 256, 256, 70, seed=3)
    _, (got, ref, a_r, pterm) = _run_bf16(w)
    slipped = got.copy()
    slipped[40, 7, :] += 1e-2
    with pytest.raises(AssertionError):
        _check_close(slipped, ref, a_r, pterm, "planted")
    slipped = got.copy()
    slipped[3, 0, 100] -= 1e-2
    with pytest.raises(AssertionError):
        _check_close(slipped, ref, a_r, pterm, "planted element")


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
        a_r, pterm = _kernel_reference(w, q, k, v, oc, None)
        _check_close(host(out), ref, a_r, pterm, "routed bf16")


def test_bf16_prefix_split_tail_blocks():
    # 176 row blocks (700 tokens, 32 / 8 heads, head_dim 128): the tail is split
    _run_bf16(wl.PrefixWorkload("bsplit", 32, 8, 128, 300, 700, seed=11))
