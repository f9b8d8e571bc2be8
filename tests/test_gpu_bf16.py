"""GPU parity of the BF16-KV comparison path: the bf16 paged cache write is a
byte-exact scatter, and the decode matches fp64 softmax attention over the same
bf16 cache (the oracle).

Tolerance, from the arithmetic: the kernel rounds each softmax weight
p~ = exp(s - m) to bf16 (8 significant bits, relative error <= 2^-8) before the
bf16 P x V product, while l sums the unrounded fp32 weights.  So output element
(h, j) is off by at most 2^-8 * sum_t (p_t / l) |v_tj| (the softmax-weighted
mean of |v|), plus fp32 rounding of the scores, exp and accumulation (bounded
here by 2e-4).  The bound is computed per element from the inputs in fp64."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def _caches(w):
    gc = i8.alloc_bf16_cache(w.num_blocks, w.Hkv, w.D)
    oc = None
    for b in range(w.B):
        k, v = w.kv(b)
        i8.bf16_kv_write(dev(k), dev(v), dev(w.slots(b)), **gc)
        oc = orc.bf16_kv_write(k, v, w.slots(b), w.num_blocks, w.block_size, **({} if oc is None else oc))
    return gc, oc


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _tol(w, q):
    """[B, Hq, D] per-element bound 2^-8 * sum_t (p_t / l) |v_tj| + 2e-4."""
    G = w.Hq // w.Hkv
    tol = np.full((w.B, w.Hq, w.D), 2e-4)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        if L == 0:
            continue
        k, v = (_f32(x) for x in w.kv(b))
        for h in range(w.Hq):
            s = k[:, h // G, :] @ _f32(q[b, h]) / np.sqrt(w.D)
            p = np.exp(s - s.max())
            tol[b, h] += 2.0 ** -8 * (p / p.sum()) @ np.abs(v[:, h // G, :])
    return tol


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
    err = np.abs(got - ref)
    tol = _tol(w, q)
    assert (err <= tol).all(), f"max-abs {err.max():.3e}, worst err/bound {(err / tol).max():.2f}"
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
    assert (np.abs(host(out) - ref) <= _tol(w, q)).all()
