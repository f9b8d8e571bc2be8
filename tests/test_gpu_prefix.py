"""GPU parity of the INT8 prefix-prefill chunk (one online softmax over cached
history + the causal chunk), against the oracle's literal online softmax."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host, gpu_quantize_rows

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _prefix_parity(w: wl.PrefixWorkload, rows=None, k=None, v=None):
    if k is None:
        k, v = w.kv()
    q = w.q()
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    i8.kv_quant_write(dev(k), dev(v), dev(w.slots()), **cache)
    q_i8, q_s = gpu_quantize_rows(q, w.Hkv, cache)
    out = torch.full((w.chunk, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    i8.int8_prefix_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"], cache["v_scale"],
                        dev(w.block_table), w.history)
    out = host(out)
    assert i8.device_error() == 0
    oc = orc.kv_quant_write(k, v, w.slots(), w.num_blocks, w.block_size)
    for key in ("k_cache", "v_cache"):
        assert np.array_equal(host(cache[key]), oc[key])
    ref = orc.prefix_attn(host(q_i8), host(q_s), oc, w.block_table, w.history, w.block_size, rows=rows)
    got = out if rows is None else out[rows]
    err = np.abs(got - ref).max()
    assert err <= TOL, f"{w.name}: max-abs {err:.3e}"
    return out, err


@pytest.mark.parametrize("H,C", [(0, 5), (0, 64), (64, 1), (100, 37), (256, 70), (1000, 200)])
@pytest.mark.parametrize("Hq,Hkv,D", [(24, 4, 256), (32, 8, 128), (4, 4, 128), (8, 1, 256)])
def test_prefix_small(H, C, Hq, Hkv, D):
    _prefix_parity(wl.PrefixWorkload("p", Hq, Hkv, D, H, C, seed=H + C + D))


def test_prefix_equal_scores_causal_mean_on_gpu():
    # Independent of the oracle: Q = 0 and integer V with sV = 1 -> row j returns the
    # mean of V over positions 0 .. H + j.
    H, C, Hq, Hkv, D = 300, 77, 6, 1, 256
    w = wl.PrefixWorkload("cm", Hq, Hkv, D, H, C, seed=2)
    rng = np.random.default_rng(3)
    k, _ = w.kv()
    vv = rng.integers(-127, 128, size=(H + C, Hkv, D)).astype(np.float32)
    vv[np.arange(H + C), 0, rng.integers(0, D, H + C)] = -127.0
    v = wl.bf16_bits(vv)
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    i8.kv_quant_write(dev(k), dev(v), dev(w.slots()), **cache)
    q_i8 = torch.zeros((C, Hq, D), dtype=torch.int8, device="cuda")
    q_s = torch.zeros((C, Hq), dtype=torch.float32, device="cuda")
    out = torch.empty((C, Hq, D), dtype=torch.float32, device="cuda")
    i8.int8_prefix_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"], cache["v_scale"],
                        dev(w.block_table), H)
    out = host(out)
    csum = np.cumsum(vv[:, 0].astype(np.float64), axis=0)
    for j in (0, 1, 31, 32, 76):
        ref = csum[H + j] / (H + j + 1)
        assert np.abs(out[j] - ref[None, :]).max() < 1e-3 * 127


def split_row_blocks(C, G, Hkv, nsm, max_split=6):
    """The launcher's work split, restated from its documented rule: 128-row blocks
    (rows = (chunk token, q-head of the group) pairs, token-major) of each KV
    head, ordered heaviest first, one CTA each; when the blocks outnumber the
    SMs and leave a partial last wave, each block of that wave is split into k
    parts over its key groups (k <= 6, tail * k <= 2 * SMs, minimizing
    ceil(tail * k / SMs) / k).  Returns the split blocks as (KV head, first row)."""
    R = C * G
    nrb = (R + 127) // 128
    RB = nrb * Hkv
    tail = RB % nsm if RB > nsm else 0
    k, best = 1, 1.0
    for kk in range(2, max_split + 1):
        if tail == 0 or tail * kk > 2 * nsm:
            break
        cost = ((tail * kk + nsm - 1) // nsm) / kk
        if cost < best - 1e-9:
            best, k = cost, kk
    full = RB - tail if k > 1 else RB
    return [(blk % Hkv, (nrb - 1 - blk // Hkv) * 128) for blk in range(full, RB)]


def test_prefix_chunk_pages_shape_sampled():
    # 2048 chunk queries after 16384 cached tokens, 24 q / 4 kv heads, head_dim
    # 256, as the benchmark launches it.  Checked rows: every 16th chunk token
    # (128 tokens across the chunk, all heads) plus every token of one row block
    # of two blocks of the split last wave (the lightest blocks, whose key
    # groups are split over several CTAs and merged by log-sum-exp).
    w = wl.prefix_chunk()
    G = w.Hq // w.Hkv
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    split = split_row_blocks(w.chunk, G, w.Hkv, nsm)
    assert split, "the pages' chunk leaves a split last wave on this GPU"
    rows = np.arange(0, w.chunk, 16)
    for _, r0 in (split[0], split[-1]):  # the heaviest and the lightest split block
        rows = np.union1d(rows, np.arange(r0 // G, min(w.chunk, (r0 + 128 + G - 1) // G)))
    rows = np.union1d(rows, [w.chunk - 1]).astype(np.int32)
    assert rows.size >= 128
    _prefix_parity(w, rows=rows)


@pytest.mark.parametrize("H", [100, 1000])
def test_prefix_split_tail_blocks(H):
    # 700 chunk tokens x 32 q-heads over 8 KV heads = 176 row blocks of 128 rows,
    # more than the SMs: the last wave's blocks are split over their key groups
    # and merged by log-sum-exp; the whole chunk is checked against the oracle.
    _prefix_parity(wl.PrefixWorkload("split", 32, 8, 128, H, 700, seed=H + 7))
