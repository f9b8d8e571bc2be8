"""Pins for the oracle's high-precision chunk attention (the first-chunk path of
"gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §3.1 and the low-history
side of its routing): it must equal textbook softmax attention computed with
numpy's matmul and exp on the same keys -- the chunk's bf16 K/V, preceded by
the INT8 history read back through numpy reshapes of the documented cache
layouts -- and reduce to the value row when a query sees a single key."""
import numpy as np
import pytest

import workloads as wl
from oracle import oracle as orc
from tests.helpers import gather_int8

BS = wl.BLOCK_SIZE


def _chunk(C, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    return (wl.randn_bf16(rng, (C, Hq, D)), wl.randn_bf16(rng, (C, Hkv, D)), wl.randn_bf16(rng, (C, Hkv, D)))


@pytest.mark.parametrize("C,Hq,Hkv,D", [(37, 4, 2, 128), (20, 6, 2, 256)])
def test_first_chunk_is_causal_softmax_attention(C, Hq, Hkv, D):
    q, k, v = _chunk(C, Hq, Hkv, D, C)
    got = orc.bf16_prefix_attn(q, k, v, None, None, 0, BS)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    ref = orc.attention_fp64(orc.bf16_to_f64(q), orc.bf16_to_f64(k), orc.bf16_to_f64(v), np.arange(1, C + 1),
                             softmax_scale=scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_history_is_read_back_from_the_int8_cache():
    H, C, Hq, Hkv, D = 45, 19, 4, 2, 128
    rng = np.random.default_rng(3)
    kh, vh = wl.randn_bf16(rng, (H, Hkv, D)), wl.randn_bf16(rng, (H, Hkv, D))
    tables, NB = wl.paged_tables([H + C], perm_seed=7)
    cache = orc.kv_quant_write(kh, vh, wl.slot_mapping(tables[0], np.arange(H)), NB, BS)
    q, k, v = _chunk(C, Hq, Hkv, D, 4)
    rows = np.array([0, 5, C - 1], np.int32)
    got = orc.bf16_prefix_attn(q, k, v, cache, tables[0], H, BS, rows=rows)
    Kq, Vq, sK, sV = gather_int8(cache, tables[0], H, Hkv, D)
    K = np.concatenate([Kq * sK[..., None].astype(np.float64), orc.bf16_to_f64(k)])
    V = np.concatenate([Vq * sV[..., None].astype(np.float64), orc.bf16_to_f64(v)])
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    ref = orc.attention_fp64(orc.bf16_to_f64(q)[rows], K, V, H + rows + 1, softmax_scale=scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_single_visible_key_returns_its_value():
    q, k, v = _chunk(1, 4, 2, 128, 9)
    got = orc.bf16_prefix_attn(q, k, v, None, None, 0, BS)
    expect = np.repeat(orc.bf16_to_f64(v), 2, axis=1)  # q-heads 0,1 -> kv 0; 2,3 -> kv 1
    assert np.array_equal(got, expect)


def test_bf16_kv_prefix_is_causal_attention_over_the_bf16_cache():
    # The BF16-KV comparison of the prefix chunk: every key (history and chunk)
    # comes from the bf16 paged cache; read back here through numpy reshapes of
    # its documented layout ([NB, Hkv, D/8, 16, 8] and [NB, Hkv, D, 16]).
    H, C, Hq, Hkv, D = 70, 21, 6, 2, 128
    rng = np.random.default_rng(8)
    k, v = wl.randn_bf16(rng, (H + C, Hkv, D)), wl.randn_bf16(rng, (H + C, Hkv, D))
    q = wl.randn_bf16(rng, (C, Hq, D))
    tables, NB = wl.paged_tables([H + C], perm_seed=9)
    cache = orc.bf16_kv_write(k, v, wl.slot_mapping(tables[0], np.arange(H + C)), NB, BS)
    rows = np.array([0, 1, 10, C - 1], np.int32)
    got = orc.bf16_kv_prefix_attn(q, cache, tables[0], H, BS, rows=rows)
    pos = np.arange(H + C)
    blk, off = tables[0][pos // BS], pos % BS
    K = cache["k_cache"].reshape(NB, Hkv, D // 8, BS, 8)[blk, :, :, off, :].reshape(H + C, Hkv, D)
    V = cache["v_cache"].reshape(NB, Hkv, D, BS)[blk, :, :, off]
    assert np.array_equal(K, k) and np.array_equal(V, v)  # the layout round trip
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    ref = orc.attention_fp64(orc.bf16_to_f64(q)[rows], orc.bf16_to_f64(K), orc.bf16_to_f64(V), H + rows + 1,
                             softmax_scale=scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # the last visible key matters: dropping it changes the row
    short = orc.attention_fp64(orc.bf16_to_f64(q)[rows], orc.bf16_to_f64(K), orc.bf16_to_f64(V), H + rows,
                               softmax_scale=scale)
    assert np.abs(got - short).max() > 1e-3
