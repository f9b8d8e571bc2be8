"""GPU parity of INT8 paged decode attention and of the debug int32 QK path.

Parity bar: int32 QK accumulators bit-exact; decode outputs within max-abs 2e-3
of the oracle (fp32 decisions, as the pages compute) on the same seeded inputs,
with caches written by the CUDA producer (itself bit-exact, see
test_gpu_producer.py).  Full-size workloads are sampled on the oracle side."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host, gpu_decode_cache, gpu_quantize_rows, gpu_decode
from tests.helpers import oracle_decode_cache, oracle_query, gather_int8

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _decode_parity(w: wl.DecodeWorkload, oracle_seqs=None, workspace=None):
    cache = gpu_decode_cache(w)
    q_i8, q_scale = gpu_quantize_rows(w.q(), w.Hkv, cache)
    out = host(gpu_decode(w, cache, q_i8, q_scale, workspace))
    assert i8.device_error() == 0
    seqs = list(range(w.B)) if oracle_seqs is None else list(oracle_seqs)
    oc = oracle_decode_cache(w, seqs)
    oq, oqs = oracle_query(w, seqs)
    assert np.array_equal(host(q_i8)[seqs], oq) and np.array_equal(host(q_scale)[seqs], oqs)
    ref = orc.decode_attn(oq, oqs, oc, w.block_tables[seqs], w.seq_lens[seqs], w.block_size)
    err = np.abs(out[seqs] - ref).max()
    assert err <= TOL, f"{w.name}: max-abs {err:.3e} > {TOL}"
    return out, err


# --------------------------------------------------------------------------- debug QK
@pytest.mark.parametrize("D,Hq,Hkv,lens", [(256, 24, 4, [300, 1, 64, 17]), (128, 32, 8, [513, 256]),
                                             (256, 8, 8, [40])])
def test_debug_qk_bit_exact(D, Hq, Hkv, lens):
    w = wl.DecodeWorkload("qk", Hq, Hkv, D, lens, seed=5)
    cache = gpu_decode_cache(w)
    q_i8, _ = gpu_quantize_rows(w.q(), Hkv, cache)
    max_len = max(lens) + 7
    acc = torch.full((w.B, Hq, max_len), -12345, dtype=torch.int32, device="cuda")
    i8.debug_qk_i32(acc, q_i8, cache["k_cache"], dev(w.block_tables), dev(w.seq_lens))
    oc = oracle_decode_cache(w)
    ref = orc.qk_i32(host(q_i8), oc["k_cache"], w.block_tables, w.seq_lens, Hkv, w.block_size, max_len=max_len)
    assert np.array_equal(host(acc), ref)
    assert i8.device_error() == 0


def test_debug_qk_extreme_values():
    # every code at +-127: |acc| = 127*127*256 = 4,129,024 per token
    D, Hq, Hkv = 256, 4, 2
    w = wl.DecodeWorkload("x", Hq, Hkv, D, [33], seed=0)
    k = wl.bf16_bits(np.full((33, Hkv, D), -2.0, np.float32))
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    i8.kv_quant_write(dev(k), dev(k), dev(w.slots(0)), **cache)
    q_i8 = torch.full((1, Hq, D), 127, dtype=torch.int8, device="cuda")
    acc = torch.zeros((1, Hq, 33), dtype=torch.int32, device="cuda")
    i8.debug_qk_i32(acc, q_i8, cache["k_cache"], dev(w.block_tables), dev(w.seq_lens))
    assert (host(acc) == -4129024).all()


# --------------------------------------------------------------------------- small decode cases
@pytest.mark.parametrize("lens", [[1], [17], [256], [257], [1000], [0, 300, 1, 4096], [33, 0, 0, 600, 255]])
@pytest.mark.parametrize("D,Hq,Hkv", [(256, 24, 4), (128, 32, 8), (128, 8, 1), (256, 4, 4)])
def test_decode_small(lens, D, Hq, Hkv):
    w = wl.DecodeWorkload("small", Hq, Hkv, D, lens, seed=sum(lens) + D)
    out, _ = _decode_parity(w)
    for b, L in enumerate(lens):
        if L == 0:
            assert not out[b].any()


@pytest.mark.parametrize("D,Hq,Hkv,lens", [
    (256, 8, 1, [8000] + [50] * 39),      # 40 pairs; the long pair spans about 100 CTAs
    (128, 16, 2, [33] * 19 + [6000]),     # 40 pairs, the long sequence last
    (256, 24, 4, [700, 0, 9000, 5] * 3),  # 48 pairs, with empty sequences
])
def test_decode_many_pairs_merge(D, Hq, Hkv, lens):
    """Calls with at least #SM / 4 (sequence, KV head) pairs take the merge with
    one warp per query row; a long pair among short ones gives that warp a long
    run of partials (many batches of its loads)."""
    w = wl.DecodeWorkload("manypairs", Hq, Hkv, D, lens, seed=sum(lens) % 997 + D)
    out, _ = _decode_parity(w)
    for b, L in enumerate(lens):
        if L == 0:
            assert not out[b].any()


@pytest.mark.parametrize("B", [37, 38])
def test_decode_merge_choice_boundary(B):
    """The host takes the one-warp-per-row merge at B * Hkv >= #SM / 4 pairs (38
    on 152 SMs) and the CTA merge below; on either side of it the pairs span
    several attention CTAs (about 600 tokens each)."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(300, 900, size=B)]
    w = wl.DecodeWorkload("mergeedge", 8, 1, 256, lens, seed=B)
    _decode_parity(w)


@pytest.mark.parametrize("D,Hq,Hkv,L,pad", [(256, 24, 4, 5000, 300), (128, 32, 8, 777, 64), (256, 8, 1, 40, 1)])
def test_decode_single_sequence_wide_block_table(D, Hq, Hkv, L, pad):
    """One sequence with a block table wider than its length needs.  Before the
    lengths arrive the kernel guesses each CTA's first unit from the table width
    and loads that unit's block-table row; here the guess misses, and the row is
    read again once the work split is known."""
    w = wl.DecodeWorkload("wide", Hq, Hkv, D, [L], seed=L + D)
    cache = gpu_decode_cache(w)
    q_i8, q_scale = gpu_quantize_rows(w.q(), w.Hkv, cache)
    wide = np.pad(w.block_tables, ((0, 0), (0, pad)), constant_values=-1)
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, wide.shape[1])
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    i8.int8_paged_decode_attn(out, q_i8, q_scale, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                              cache["v_scale"], dev(wide), dev(w.seq_lens), ws)
    got = host(out)
    assert i8.device_error() == 0
    oc = oracle_decode_cache(w, [0])
    oq, oqs = oracle_query(w, [0])
    ref = orc.decode_attn(oq, oqs, oc, w.block_tables, w.seq_lens, w.block_size)
    assert np.abs(got - ref).max() <= TOL


def test_decode_workspace_reuse_and_repeat():
    # The workspace holds only this call's partials (no state carried between
    # calls): repeated calls on one workspace give identical results, each written
    # into a NaN-filled output (no stale rows).
    w = wl.DecodeWorkload("rep", 24, 4, 256, [5000, 3000, 40], seed=9)
    cache = gpu_decode_cache(w)
    q_i8, q_s = gpu_quantize_rows(w.q(), w.Hkv, cache)
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
    outs = []
    for _ in range(3):
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
        gpu_decode(w, cache, q_i8, q_s, ws, out=out)
        outs.append(host(out))
    assert np.isfinite(outs[0]).all()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert i8.device_error() == 0


def test_decode_workspace_reuse_across_batches():
    # One workspace (sized for the largest batch) serves calls whose batches,
    # lengths and head shapes differ: every record a call reads is written
    # earlier in the same call, whatever the previous calls left in the buffer.
    shapes = [(24, 4, 256, [5000, 3000, 40]), (24, 4, 256, [40, 9000]), (24, 4, 256, [1, 1, 1, 20000, 7]),
              (32, 8, 128, [700]), (24, 4, 256, [12000])]
    nbytes = max(i8.decode_workspace_bytes(len(l), hq, hkv, d, (max(l) + 15) // 16) for hq, hkv, d, l in shapes)
    ws = torch.zeros(nbytes + 4096, dtype=torch.uint8, device="cuda")
    for k, (hq, hkv, d, lens) in enumerate(shapes):
        _decode_parity(wl.DecodeWorkload(f"reuse{k}", hq, hkv, d, lens, seed=40 + k), workspace=ws)
    assert i8.device_error() == 0


def test_decode_rejects_small_workspace():
    w = wl.DecodeWorkload("ws", 24, 4, 256, [600], seed=1)
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    q_i8 = torch.zeros((1, 24, 256), dtype=torch.int8, device="cuda")
    q_s = torch.zeros((1, 24), dtype=torch.float32, device="cuda")
    out = torch.empty((1, 24, 256), dtype=torch.float32, device="cuda")
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(i8.I8KVError) as e:
        i8.int8_paged_decode_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                  cache["v_scale"], dev(w.block_tables), dev(w.seq_lens), small)
    assert e.value.status == 3


def test_decode_bad_block_table_entry_is_skipped_and_recorded():
    # an out-of-pool block id is not read; the kernel records error 2 and finishes
    w = wl.DecodeWorkload("bad", 8, 2, 128, [100], seed=3)
    cache = gpu_decode_cache(w)
    q_i8, q_s = gpu_quantize_rows(w.q(), w.Hkv, cache)
    bt = w.block_tables.copy()
    bt[0, 2] = w.num_blocks + 5
    out = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    ws = i8.decode_workspace(1, 8, 2, 128, bt.shape[1])
    i8.int8_paged_decode_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                              cache["v_scale"], dev(bt), dev(w.seq_lens), ws)
    assert i8.device_error() == 2
    assert i8.device_error() == 0


def test_decode_closed_form_on_gpu():
    # Independent of the oracle: scores constant on each aligned 32-token group and
    # integer V with sV = 1 make every group's quantization exact, so the GPU must
    # return sum_t P_t V_t (P = softmax of the dequantized scores) up to fp32 rounding.
    rng = np.random.default_rng(4)
    L, Hq, Hkv, D = 1184, 6, 1, 256
    w = wl.DecodeWorkload("cf", Hq, Hkv, D, [L], seed=2)
    base = rng.standard_normal((L // 32, Hkv, D)).astype(np.float32)
    k = wl.bf16_bits(np.repeat(base, 32, axis=0))
    v = rng.integers(-127, 128, size=(L, Hkv, D)).astype(np.float32)
    v[np.arange(L), 0, rng.integers(0, D, L)] = 127.0
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    i8.kv_quant_write(dev(k), dev(wl.bf16_bits(v)), dev(w.slots(0)), **cache)
    q_i8, q_s = gpu_quantize_rows(w.q(), Hkv, cache)
    out = host(gpu_decode(w, cache, q_i8, q_s))
    Kq = host(cache["k_cache"])
    sK = host(cache["k_scale"])
    Kt, _, sKt, _ = gather_int8(dict(k_cache=Kq, v_cache=host(cache["v_cache"]), k_scale=sK,
                                     v_scale=host(cache["v_scale"])), w.block_tables[0], L, Hkv, D)
    c = float(np.float32(1) / np.sqrt(np.float32(D)))
    qi, qs = host(q_i8), host(q_s)
    for h in range(Hq):
        s = (Kt[:, 0].astype(np.int64) @ qi[0, h].astype(np.int64)) * float(qs[0, h]) * sKt[:, 0] * c
        p = np.exp(s - s.max())
        ref = (p / p.sum()) @ v[:, 0].astype(np.float64)
        assert np.abs(out[0, h] - ref).max() < 1e-3 * max(1.0, np.abs(ref).max() / 127)


# --------------------------------------------------------------------------- the pages' workloads
def test_decode_4k_pages_shape():
    w = wl.decode_4k()
    out, err = _decode_parity(w)
    # and against unquantized fp64 attention (the oracle's own bar is 2e-2)
    kd, vd = (orc.bf16_to_f64(a) for a in w.kv(0))
    ref = orc.attention_fp64(orc.bf16_to_f64(w.q()), kd, vd, [4096])
    assert np.abs(out - ref).max() < 2e-2


@pytest.mark.parametrize("L", [8192, 16384, 32768])
def test_decode_outlier_long_history(L):
    _decode_parity(wl.decode_outlier(L))


def test_decode_batch64_sampled():
    w = wl.decode_batch()
    order = np.argsort(w.seq_lens)
    sample = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 0, 63})
    _decode_parity(w, oracle_seqs=sample)


def test_decode_gqa_b16_sampled():
    w = wl.producer_gqa_decode()
    _decode_parity(w, oracle_seqs=[0, 15])
