"""GPU parity of the BF16-KV comparison of the prefix chunk (the pages' BF16
control when they compare BF16 and INT8 attention on prefill chunks by
history, "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §4.2).

Every key comes from the bf16 paged cache, so the oracle's fp64 attention on
those bf16 values is the reference.  The kernel rounds each p~ = exp(s - m) to
bf16 for the P x V product (relative error <= 2^-9) while l sums the fp32 p~,
so output element (j, d) moves by at most 2^-9 sum_t p_t |v_td|; the bound
allows 2^-8 of it, plus 3e-4 for fp32 scores, ex2 and accumulation:

    |out - oracle| <= 2^-8 sum_t p_t |v_td| + 3e-4   (element by element)."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def _pterm(w, q, k, v, rows):
    G = w.Hq // w.Hkv
    K, V = (wl.bf16_values(x).astype(np.float64) for x in (k, v))
    qv = wl.bf16_values(q).astype(np.float64)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(w.D)))
    out = np.empty((len(rows), w.Hq, w.D))
    for i, j in enumerate(rows):
        n = w.history + j + 1
        for h in range(w.Hq):
            s = K[:n, h // G] @ qv[j, h] * scale
            p = np.exp(s - s.max())
            out[i, h] = 2.0 ** -8 * ((p / p.sum()) @ np.abs(V[:n, h // G]))
    return out


def _run(w: wl.PrefixWorkload, rows=None, plant=False):
    k, v = w.kv()
    q = w.q()
    cache = i8.alloc_bf16_cache(w.num_blocks, w.Hkv, w.D)
    i8.bf16_kv_write(dev(k), dev(v), dev(w.slots()), **cache)
    out = torch.full((w.chunk, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    i8.bf16_kv_prefix_attn(out, dev(q), cache["k_cache"], cache["v_cache"], dev(w.block_table), w.history)
    got = host(out)
    assert i8.device_error() == 0
    oc = orc.bf16_kv_write(k, v, w.slots(), w.num_blocks, w.block_size)
    assert np.array_equal(host(cache["k_cache"]), oc["k_cache"]) and np.array_equal(host(cache["v_cache"]),
                                                                                      oc["v_cache"])
    rows = np.arange(w.chunk) if rows is None else np.asarray(rows, np.int32)
    ref = orc.bf16_kv_prefix_attn(q, oc, w.block_table, w.history, w.block_size, rows=rows)
    got = got[rows]
    bound = _pterm(w, q, k, v, rows) + 3e-4
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"{w.name}: {int((err > bound).sum())} elements past the bound, max-abs {err.max():.3e}"
    if plant:  # the bound catches a 1e-2 slip confined to one row
        got[len(rows) // 2, 1, :] += 1e-2
        assert (np.abs(got - ref) > bound).any()
    return err.max()


@pytest.mark.parametrize("H,C", [(0, 1), (0, 45), (100, 37), (256, 70), (1000, 200)])
@pytest.mark.parametrize("Hq,Hkv,D", [(24, 4, 256), (32, 8, 128), (8, 1, 256)])
def test_bf16_kv_prefix_small(H, C, Hq, Hkv, D):
    _run(wl.PrefixWorkload("bkv", Hq, Hkv, D, H, C, seed=H + C + D + 1), plant=(H == 256))


def test_bf16_kv_prefix_split_tail_blocks():
    # 176 row blocks (700 tokens, 32 / 8 heads, head_dim 128): the last wave is split and merged
    _run(wl.PrefixWorkload("bkvsplit", 32, 8, 128, 300, 700, seed=12))


def test_bf16_kv_prefix_pages_chunk_sampled():
    # the pages' chunk shape: 2048 queries after 16384 cached tokens, 24 / 4 heads, head_dim 256
    w = wl.prefix_chunk()
    _run(w, rows=np.array([0, 1, 100, 1023, 2047], np.int32))
