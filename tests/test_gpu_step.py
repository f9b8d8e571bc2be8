"""GPU parity of the one-launch decode step (i8kv_int8_decode_step).

The step must equal the two-call sequence it replaces bit for bit:
kv_quant_write of every sequence's newest token (position seq_lens[b] - 1)
with its query, then int8_paged_decode_attn.  Both start from the same cache
holding positions 0 .. L-2; afterwards the caches, the scales and the outputs
must be identical, and the output is also checked against the oracle.  The
cases put the new token at every kind of position: alone, first of a block,
last of a block, first of a 32-token group and of a 128-token unit, inside a
batch with an empty sequence, and at the end of a long outlier history."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host
from tests.helpers import oracle_decode_cache, oracle_query

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _history_cache(w):
    """Cache with positions 0 .. L_b - 2 of every sequence."""
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        if L > 1:
            k, v = w.kv(b)
            i8.kv_quant_write(dev(k[:L - 1]), dev(v[:L - 1]), dev(w.slots(b, 0, L - 1)), **cache)
    return cache


def _new_tokens(w):
    k_new = np.zeros((w.B, w.Hkv, w.D), np.uint16)
    v_new = np.zeros((w.B, w.Hkv, w.D), np.uint16)
    slots = np.full((w.B,), -1, np.int32)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        if L > 0:
            k, v = w.kv(b)
            k_new[b], v_new[b] = k[L - 1], v[L - 1]
            slots[b] = w.slots(b, L - 1, L)[0]
    return k_new, v_new, slots


def _run_both(w):
    k_new, v_new, slots = _new_tokens(w)
    q = dev(w.q())
    bt, sl = dev(w.block_tables), dev(w.seq_lens)
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
    # two calls
    c1 = _history_cache(w)
    q_i8 = torch.empty((w.B, w.Hq, w.D), dtype=torch.int8, device="cuda")
    q_s = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    i8.kv_quant_write(dev(k_new), dev(v_new), dev(slots), **c1, q=q, q_i8=q_i8, q_scale=q_s)
    out1 = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    i8.int8_paged_decode_attn(out1, q_i8, q_s, c1["k_cache"], c1["v_cache"], c1["k_scale"], c1["v_scale"], bt, sl, ws)
    # one launch
    c2 = _history_cache(w)
    out2 = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    i8.int8_decode_step(out2, q, dev(k_new), dev(v_new), c2["k_cache"], c2["v_cache"], c2["k_scale"], c2["v_scale"],
                        bt, sl, ws)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    return c1, c2, host(out1), host(out2)


@pytest.mark.parametrize("lens,Hq,Hkv,D", [
    ([1], 24, 4, 256),            # the new token is the whole history
    ([17], 24, 4, 256),           # first token of a block
    ([32], 24, 4, 256),           # last token of a 32-token group
    ([33], 24, 4, 256),           # first token of a group
    ([129], 24, 4, 256),          # first token of a 128-token unit
    ([300, 17, 0, 1000], 32, 8, 128),
    ([4096], 24, 4, 256),
    ([2049, 511, 16], 8, 8, 256),
])
def test_step_equals_two_calls(lens, Hq, Hkv, D):
    w = wl.DecodeWorkload("step", Hq, Hkv, D, lens, seed=sum(lens) + 11)
    c1, c2, out1, out2 = _run_both(w)
    for name in ("k_cache", "v_cache", "k_scale", "v_scale"):
        assert torch.equal(c1[name], c2[name]), name
    assert np.array_equal(out1, out2, equal_nan=False)
    for b, L in enumerate(lens):
        if L == 0:
            assert not out2[b].any()


def test_step_matches_oracle_long_outlier_history():
    w = wl.decode_outlier(16384)
    c1, c2, out1, out2 = _run_both(w)
    assert torch.equal(c1["k_cache"], c2["k_cache"]) and torch.equal(c1["v_scale"], c2["v_scale"])
    assert np.array_equal(out1, out2)
    oc = oracle_decode_cache(w, [0])
    oq, oqs = oracle_query(w, [0])
    ref = orc.decode_attn(oq, oqs, oc, w.block_tables, w.seq_lens, w.block_size)
    assert np.abs(out2 - ref).max() <= TOL


def test_back_to_back_steps_see_the_previous_token():
    """Two steps enqueued back to back on many short sequences: every (sequence,
    KV head) pair lies in one attention CTA, so no merge CTA has partials.  The
    second step's history holds the first step's token, written by the first
    attention kernel; the merge grid between them must still end after that
    kernel, or the second step could read the cache before the write.  The
    result must equal the producer writing both tokens, then one decode."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(3, 33, size=48)]  # one 32-token group per pair
    w = wl.DecodeWorkload("steps2", 24, 4, 256, lens, seed=17)
    L = w.seq_lens.astype(np.int64)
    bt = dev(w.block_tables)
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])

    def token(pos_of):  # the bf16 K/V and slot of position pos_of(b) of every sequence
        k_t = np.zeros((w.B, w.Hkv, w.D), np.uint16)
        v_t = np.zeros((w.B, w.Hkv, w.D), np.uint16)
        sl = np.full((w.B,), -1, np.int32)
        for b in range(w.B):
            k, v = w.kv(b)
            pos = pos_of(b)
            k_t[b], v_t[b] = k[pos], v[pos]
            sl[b] = w.slots(b, pos, pos + 1)[0]
        return k_t, v_t, sl

    first = token(lambda b: int(L[b]) - 2)
    second = token(lambda b: int(L[b]) - 1)
    q1 = dev(np.asarray(wl.randn_bf16(np.random.default_rng(6), (w.B, w.Hq, w.D))))
    q2 = dev(w.q())
    # reference: the producer writes positions 0 .. L-1, then one decode
    c1 = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    for b in range(w.B):
        k, v = w.kv(b)
        i8.kv_quant_write(dev(k[:int(L[b])]), dev(v[:int(L[b])]), dev(w.slots(b, 0, int(L[b]))), **c1)
    q_i8 = torch.empty((w.B, w.Hq, w.D), dtype=torch.int8, device="cuda")
    q_s = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    dummy = torch.zeros((w.B, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
    i8.kv_quant_write(dummy, dummy, torch.full((w.B,), -1, dtype=torch.int32, device="cuda"), **c1, q=q2,
                      q_i8=q_i8, q_scale=q_s)
    out1 = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    i8.int8_paged_decode_attn(out1, q_i8, q_s, c1["k_cache"], c1["v_cache"], c1["k_scale"], c1["v_scale"], bt,
                              dev(w.seq_lens), ws)
    # two steps from the cache of positions 0 .. L-3, no synchronization between them
    c2 = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    for b in range(w.B):
        if L[b] > 2:
            k, v = w.kv(b)
            i8.kv_quant_write(dev(k[:int(L[b]) - 2]), dev(v[:int(L[b]) - 2]), dev(w.slots(b, 0, int(L[b]) - 2)), **c2)
    torch.cuda.synchronize()
    out_a = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    out_b = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    sl_a, sl_b = dev((w.seq_lens - 1).astype(np.int32)), dev(w.seq_lens)
    for _ in range(3):  # repeated, so that a race would have several chances to show
        c2w = {n: t.clone() for n, t in c2.items()}
        i8.int8_decode_step(out_a, q1, dev(first[0]), dev(first[1]), c2w["k_cache"], c2w["v_cache"],
                            c2w["k_scale"], c2w["v_scale"], bt, sl_a, ws)
        i8.int8_decode_step(out_b, q2, dev(second[0]), dev(second[1]), c2w["k_cache"], c2w["v_cache"],
                            c2w["k_scale"], c2w["v_scale"], bt, sl_b, ws)
        torch.cuda.synchronize()
        assert i8.device_error() == 0
        for name in ("k_cache", "v_cache", "k_scale", "v_scale"):
            assert torch.equal(c1[name], c2w[name]), name
        assert np.array_equal(host(out1), host(out_b))


@pytest.mark.parametrize("lens", [[3000], [129, 5, 2000]])
def test_step_wide_block_table(lens):
    """Block tables wider than the lengths need (columns past them are -1): the
    guessed first unit misses and the new token's block comes from the table;
    still bit-identical to the two calls."""
    w = wl.DecodeWorkload("stepwide", 24, 4, 256, lens, seed=sum(lens) + 3)
    w.block_tables = np.pad(w.block_tables, ((0, 0), (0, 100)), constant_values=-1)
    c1, c2, out1, out2 = _run_both(w)
    for name in ("k_cache", "v_cache", "k_scale", "v_scale"):
        assert torch.equal(c1[name], c2[name]), name
    assert np.array_equal(out1, out2)
