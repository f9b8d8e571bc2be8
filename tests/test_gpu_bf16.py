"""GPU parity of the BF16-KV comparison path: the bf16 paged cache write is a
byte-exact scatter, and the decode matches fp64 softmax attention over the same
bf16 cache (the oracle) within 2e-3."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _caches(w):
    gc = i8.alloc_bf16_cache(w.num_blocks, w.Hkv, w.D)
    oc = None
    for b in range(w.B):
        k, v = w.kv(b)
        i8.bf16_kv_write(dev(k), dev(v), dev(w.slots(b)), **gc)
        oc = orc.bf16_kv_write(k, v, w.slots(b), w.num_blocks, w.block_size, **({} if oc is None else oc))
    return gc, oc


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([1], 24, 4, 256), ([300, 17], 24, 4, 256), ([129, 0, 1000], 32, 8, 128),
                                            ([4096], 24, 4, 256)])
def test_bf16_write_and_decode(lens, Hq, Hkv, D):
    w = wl.DecodeWorkload("bf16", Hq, Hkv, D, lens, seed=sum(lens) + 5)
    gc, oc = _caches(w)
    assert np.array_equal(host(gc["k_cache"]), oc["k_cache"])
    assert np.array_equal(host(gc["v_cache"]), oc["v_cache"])
    q = w.q()
    out = torch.full((w.B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = i8.decode_workspace(w.B, Hq, Hkv, D, w.block_tables.shape[1])
    i8.bf16_paged_decode_attn(out, dev(q), gc["k_cache"], gc["v_cache"], dev(w.block_tables), dev(w.seq_lens), ws)
    got = host(out)
    assert i8.device_error() == 0
    ref = orc.bf16_decode_attn(q, oc, w.block_tables, w.seq_lens, w.block_size)
    err = np.abs(got - ref).max()
    assert err <= TOL, f"max-abs {err:.3e}"
    for b, L in enumerate(lens):
        if L == 0:
            assert not got[b].any()


def test_bf16_decode_long_outlier_history():
    w = wl.decode_outlier(16384)
    gc, oc = _caches(w)
    q = w.q()
    out = torch.empty((1, 24, 256), dtype=torch.float32, device="cuda")
    ws = i8.decode_workspace(1, 24, 4, 256, w.block_tables.shape[1])
    i8.bf16_paged_decode_attn(out, dev(q), gc["k_cache"], gc["v_cache"], dev(w.block_tables), dev(w.seq_lens), ws)
    ref = orc.bf16_decode_attn(q, oc, w.block_tables, w.seq_lens, w.block_size)
    assert np.abs(host(out) - ref).max() <= TOL
