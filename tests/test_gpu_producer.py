"""GPU parity of the KV producer (kv_quant_write): cache bytes, scales and the
quantized query must be bit-identical to the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host
from tests.helpers import read_golden

pytestmark = pytest.mark.gpu


def _assert_same(gpu: dict, ref: dict, keys):
    for k in keys:
        g = host(gpu[k])
        r = ref[k]
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        bad = np.flatnonzero(g.ravel() != r.ravel())
        assert bad.size == 0, f"{k}: {bad.size} mismatches, first at flat index {bad[:5]}"


def _run(k, v, slots, num_blocks, q=None):
    T, Hkv, D = k.shape
    gc = i8.alloc_int8_cache(num_blocks, Hkv, D)
    extra = {}
    if q is not None:
        extra = dict(q=dev(q), q_i8=torch.empty(q.shape, dtype=torch.int8, device="cuda"),
                     q_scale=torch.empty(q.shape[:2], dtype=torch.float32, device="cuda"))
    i8.kv_quant_write(dev(k), dev(v), dev(slots), **gc, **extra)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    gc.update({kk: extra[kk] for kk in ("q_i8", "q_scale")} if q is not None else {})
    ref = orc.kv_quant_write(k, v, slots, num_blocks, wl.BLOCK_SIZE, q=q)
    return gc, ref


def test_producer_gqa_workload_bit_exact():
    # 8192 new tokens, 8 KV heads, head_dim 128, 2% outliers x10, block-aligned slots
    # (the transposed V path) plus the 32-head query.
    p = wl.producer_tokens()
    gc, ref = _run(p["k"], p["v"], p["slots"], p["num_blocks"], q=p["q"])
    _assert_same(gc, ref, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])


@pytest.mark.parametrize("D,Hkv,Hq,T", [(256, 4, 24, 37), (128, 8, 32, 19), (256, 1, 8, 1), (128, 2, 4, 48)])
def test_producer_scattered_slots_bit_exact(D, Hkv, Hq, T):
    # random slots (byte-scatter V path), a skipped token (slot -1), ragged tile
    rng = np.random.default_rng(T)
    NB = (T + 15) // 16 + 3
    slots = rng.permutation(NB * 16)[:T].astype(np.int32)
    slots[T // 2] = -1
    k = wl.randn_bf16(rng, (T, Hkv, D))
    v = wl.randn_bf16(rng, (T, Hkv, D))
    q = wl.randn_bf16(rng, (T, Hq, D))
    gc, ref = _run(k, v, slots, NB, q=q)
    _assert_same(gc, ref, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])


@pytest.mark.parametrize("D,Hkv,Hq,T", [(128, 3, 7, 200), (256, 6, 18, 333), (128, 5, 10, 1000), (256, 8, 64, 520),
                                       (128, 1, 2, 5000)])
def test_producer_uneven_head_groups_bit_exact(D, Hkv, Hq, T):
    # The producer's work units hold up to 1024 / D heads of one tensor: head
    # counts that do not fill them (3, 5, 6 KV heads; 7 query heads, not a
    # multiple of the KV heads) give units of different sizes, warps without a
    # task in some units, and -- with thousands of tokens -- several tiles per
    # CTA.  One sequence's block-aligned slots (the transposed V path), the tail
    # ragged.
    rng = np.random.default_rng(T + Hkv)
    tables, NB = wl.paged_tables([T], perm_seed=T)
    slots = wl.slot_mapping(tables[0], np.arange(T))
    k = wl.randn_bf16(rng, (T, Hkv, D))
    v = wl.randn_bf16(rng, (T, Hkv, D))
    q = wl.randn_bf16(rng, (T, Hq, D))
    gc, ref = _run(k, v, slots, NB, q=q)
    _assert_same(gc, ref, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])


def test_producer_mixed_aligned_and_partial_tiles():
    # positions 5 .. 5+70 of one sequence: no tile starts on a block boundary
    D, Hkv = 256, 4
    tables, NB = wl.paged_tables([80])
    slots = wl.slot_mapping(tables[0], np.arange(5, 75))
    rng = np.random.default_rng(1)
    k = wl.randn_bf16(rng, (70, Hkv, D))
    v = wl.randn_bf16(rng, (70, Hkv, D))
    gc, ref = _run(k, v, slots, NB)
    _assert_same(gc, ref, ["k_cache", "v_cache", "k_scale", "v_scale"])


def test_producer_golden_cases_on_gpu():
    # The worked cases of the quantization rule, checked against their stated codes
    # directly (not through the oracle): ties to even, exact scales, zero vectors.
    rows = read_golden("quant_rne.txt")
    D, Hkv = 128, 1
    T = len(rows)
    k = np.zeros((T, Hkv, D), np.float32)
    for t, (vals, _, _) in enumerate(rows):
        k[t, 0, : len(vals)] = [float(x) for x in vals]
    kb = wl.bf16_bits(k)
    gc = i8.alloc_int8_cache(1, Hkv, D)
    i8.kv_quant_write(dev(kb), dev(kb), dev(np.arange(T, dtype=np.int32)), **gc)
    K5 = host(gc["k_cache"])
    ks = host(gc["k_scale"])
    vs = host(gc["v_scale"])
    V4 = host(gc["v_cache"])
    for t, (vals, scale, codes) in enumerate(rows):
        n = len(vals)
        got = K5[0, 0, :, t, :].ravel()[:n]
        assert got.tolist() == [int(c) for c in codes]
        assert not K5[0, 0, :, t, :].ravel()[n:].any()
        assert ks[0, t, 0] == np.float32(scale[0]) and vs[0, t, 0] == np.float32(scale[0])
        assert V4[0, 0, :n, t].tolist() == [int(c) for c in codes]


def test_producer_rejects_bad_arguments():
    gc = i8.alloc_int8_cache(2, 4, 256)
    k = torch.zeros((3, 4, 256), dtype=torch.bfloat16, device="cuda")
    st = i8.lib().i8kv_kv_quant_write(k.data_ptr(), k.data_ptr(), None, 3, 4, 256, 8, 2, None, None, None, None,
                                      None, 0, None, None, None)
    assert st == 2 and "block_size" in i8.last_error()
    with pytest.raises(i8.I8KVError):
        i8.kv_quant_write(k, k, torch.zeros(3, dtype=torch.int64, device="cuda"), **gc)
    # slots beyond the pool are skipped and recorded, not written
    i8.kv_quant_write(k, k, torch.tensor([0, 1, 999], dtype=torch.int32, device="cuda"), **gc)
    assert i8.device_error() == 2
    assert i8.device_error() == 0
