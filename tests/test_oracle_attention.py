"""Pins of the oracle's QK, decode and prefix attention (CPU only).

Each check is fixed by something other than the oracle's own formula:
 * exact integer arithmetic (brute-force int32 QK through numpy),
 * fp64 unquantized softmax attention (the textbook definition) on N(0,1) data,
 * closed forms (equal scores with sV = 1 give the mean of V; scores constant
   on each aligned 32-token group reproduce sum P V exactly),
 * invariants (log-sum-exp merging of partitions equals one pass; decode of
   the history L equals the prefix row that sees the same L keys),
 * the error decomposition O - O_hat = sum P eV + sum eW Vq with its bound
   ("gfx936 DCU上实现INT8 PV MMAC" §1).
"""
import numpy as np
import pytest

import workloads as wl
from oracle import oracle as orc
from tests.helpers import oracle_decode_cache, oracle_query, gather_int8, quantize_rows


def _small_decode(L, Hq=6, Hkv=2, D=32, seed=0, B=1):
    return wl.DecodeWorkload("t", Hq, Hkv, D, [L] * B if np.isscalar(L) else L, seed=seed)


# --------------------------------------------------------------------------- QK
def test_qk_i32_bruteforce():
    w = _small_decode([50, 1, 33], Hq=4, Hkv=2, D=64, seed=3)
    cache = oracle_decode_cache(w)
    q_i8, _ = oracle_query(w)
    acc = orc.qk_i32(q_i8, cache["k_cache"], w.block_tables, w.seq_lens, w.Hkv, w.block_size, max_len=56)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        Kt, _, _, _ = gather_int8(cache, w.block_tables[b], L, w.Hkv, w.D)
        for h in range(w.Hq):
            ref = Kt[:, h // 2, :].astype(np.int64) @ q_i8[b, h].astype(np.int64)
            assert np.array_equal(acc[b, h, :L], ref)
            assert not acc[b, h, L:].any()


def test_qk_i32_extreme():
    # all codes at the clamp: acc = 127 * 127 * D = 4,129,024 for D = 256 (< 2^24)
    D, bs = 256, 16
    k = wl.bf16_bits(np.full((1, 1, D), 3.0, np.float32))
    c = orc.kv_quant_write(k, k, np.array([5], np.int32), 1, bs)
    q = np.full((1, 1, D), 127, np.int8)
    acc = orc.qk_i32(q, c["k_cache"], np.array([[0]], np.int32), np.array([6], np.int32), 1, bs, max_len=6)
    assert acc[0, 0, 5] == 127 * 127 * 256 == 4129024
    q = -q
    acc = orc.qk_i32(q, c["k_cache"], np.array([[0]], np.int32), np.array([6], np.int32), 1, bs, max_len=6)
    assert acc[0, 0, 5] == -4129024


# --------------------------------------------------------------------------- decode vs fp64
@pytest.mark.parametrize("L,D,Hq,Hkv", [(1, 16, 2, 1), (7, 16, 4, 2), (33, 32, 6, 2), (64, 32, 3, 3), (300, 64, 6, 2)])
def test_decode_vs_fp64_tiny(L, D, Hq, Hkv):
    w = wl.DecodeWorkload("t", Hq, Hkv, D, [L], seed=L)
    cache = oracle_decode_cache(w)
    q_i8, q_s = oracle_query(w)
    out = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size)
    kd, vd = (orc.bf16_to_f64(a) for a in w.kv(0))
    ref = orc.attention_fp64(orc.bf16_to_f64(w.q()), kd, vd, [L])
    assert np.abs(out - ref).max() < 2e-2


def test_decode_vs_fp64_pages_shape():
    # One layer of the pages' model: 24 q / 4 kv heads, head_dim 256, history 4096.
    w = wl.decode_4k()
    cache = oracle_decode_cache(w)
    q_i8, q_s = oracle_query(w)
    out = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size)
    kd, vd = (orc.bf16_to_f64(a) for a in w.kv(0))
    ref = orc.attention_fp64(orc.bf16_to_f64(w.q()), kd, vd, [4096])
    err = np.abs(out - ref).max()
    assert err < 2e-2
    # the quantized path moves the output by far less than the tolerance: a dropped
    # scale or a wrong head mapping would give errors of order 1e-1 .. 1
    assert err < 5e-3


# --------------------------------------------------------------------------- closed forms
def _integer_v(rng, L, Hkv, D):
    """bf16 V with integer entries in [-127, 127] and one +-127 per (token, head): sV = 1."""
    v = rng.integers(-127, 128, size=(L, Hkv, D)).astype(np.float32)
    idx = rng.integers(0, D, size=(L, Hkv))
    sign = rng.choice([-1.0, 1.0], size=(L, Hkv))
    np.put_along_axis(v, idx[..., None], (127 * sign)[..., None], axis=2)
    return v


@pytest.mark.parametrize("L", [1, 2, 31, 32, 33, 255, 256, 257, 600, 1024])
@pytest.mark.parametrize("fp32", [True, False])
def test_decode_equal_scores_give_mean_of_v(L, fp32):
    # Q = 0 -> sQ = 0 -> every score is 0 -> P = 1/L; sV = 1 -> every W of a group is
    # equal -> Wq = 127 -> O = mean_t V_t.  L = 1 gives O = dequant(V_0) = V_0.
    rng = np.random.default_rng(L)
    Hq, Hkv, D = 4, 2, 32
    w = wl.DecodeWorkload("t", Hq, Hkv, D, [L], seed=1)
    k, _ = w.kv(0)
    v = _integer_v(rng, L, Hkv, D)
    cache = orc.kv_quant_write(k, wl.bf16_bits(v), w.slots(0), w.num_blocks, w.block_size)
    assert np.all(cache["v_scale"].reshape(-1, Hkv)[w.slots(0)] == 1.0)
    q_i8 = np.zeros((1, Hq, D), np.int8)
    q_s = np.zeros((1, Hq), np.float32)
    out = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size, fp32_decisions=fp32)
    mean = v.astype(np.float64).mean(axis=0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], mean[h // 2], rtol=0, atol=1e-4 if fp32 else 1e-10)


@pytest.mark.parametrize("fp32", [True, False])
def test_decode_group_constant_scores_exact(fp32):
    # Scores constant on each aligned 32-token group (identical K vectors inside a group)
    # and sV = 1: each group's W are equal, so the group quantization is exact and
    # O = sum_t P_t V_t with P the softmax of the dequantized scores.  Groups that were
    # not aligned to position 0 would mix two W levels and miss by ~1/127 relative.
    rng = np.random.default_rng(4)
    L, Hq, Hkv, D = 416, 2, 1, 32
    w = wl.DecodeWorkload("t", Hq, Hkv, D, [L], seed=2)
    base = rng.standard_normal((L // 32, Hkv, D)).astype(np.float32) * 3
    k = wl.bf16_bits(np.repeat(base, 32, axis=0))
    v = _integer_v(rng, L, Hkv, D)
    cache = orc.kv_quant_write(k, wl.bf16_bits(v), w.slots(0), w.num_blocks, w.block_size)
    q_i8, q_s = oracle_query(w)
    out = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size, fp32_decisions=fp32)
    Kt, Vt, sK, sV = gather_int8(cache, w.block_tables[0], L, Hkv, D)
    c = float(np.float32(1) / np.sqrt(np.float32(D)))
    for h in range(Hq):
        s = (Kt[:, 0].astype(np.int64) @ q_i8[0, h].astype(np.int64)) * float(q_s[0, h]) * sK[:, 0] * c
        p = np.exp(s - s.max())
        ref = (p / p.sum()) @ Vt[:, 0].astype(np.float64)
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=2e-5 if fp32 else 1e-10)


# --------------------------------------------------------------------------- invariants
@pytest.mark.parametrize("pmax", [127, 255])
def test_partition_merge_invariance(pmax):
    # fp64 decisions: partitioned decode + LSE merge == one pass == the closed group form
    # (signed INT8 probability codes, and the UINT8 codes 0..255)
    w = _small_decode([1000, 777, 64, 5], Hq=6, Hkv=2, D=64, seed=7)
    cache = oracle_decode_cache(w)
    q_i8, q_s = oracle_query(w)
    outs = [orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size, partition=p,
                            fp32_decisions=False, pmax=pmax) for p in (32, 64, 256, 512, 1024)]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-12)
    c = 1.0 / np.sqrt(64.0)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        Kt, Vt, sK, sV = gather_int8(cache, w.block_tables[b], L, w.Hkv, w.D)
        for h in range(w.Hq):
            s = (Kt[:, h // 3].astype(np.int64) @ q_i8[b, h].astype(np.int64)) * float(q_s[b, h]) * sK[:, h // 3] * c
            g = orc.group_form(s, sV[:, h // 3].astype(np.float64), Vt[:, h // 3], pmax=pmax)
            np.testing.assert_allclose(outs[0][b, h], g, rtol=0, atol=1e-12)


@pytest.mark.parametrize("pmax", [127, 255])
def test_decode_error_decomposition_and_bound(pmax):
    # O - O_hat = sum_t P_t eV_t + sum_t c_g(t) eW_t Vq_t   with eV = V - sV Vq,
    # eW = W - sW Wq, P_t = c_g(t) * (partition-normalized P_t), for the oracle's
    # own W/Wq/sW trace; plus the a-priori bound |eV| <= sV/2, |eW| <= sW/2.
    w = _small_decode([700], Hq=4, Hkv=2, D=64, seed=11)
    cache = oracle_decode_cache(w)
    q_i8, q_s = oracle_query(w)
    b, h = 0, 3
    out, tr = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size,
                              fp32_decisions=True, trace=(b, h), pmax=pmax)
    L = 700
    kvh = h // 2
    Kt, Vq, sK, sV = gather_int8(cache, w.block_tables[b], L, w.Hkv, w.D)
    vd = orc.bf16_to_f64(w.kv(b)[1])[:, kvh, :]
    Vq = Vq[:, kvh, :].astype(np.float64)
    sV = sV[:, kvh].astype(np.float64)
    # partition-normalized P from the trace: W = P * sV (fp32), so P ~= W / sV
    Ppart = tr["W"] / sV
    P = tr["c"] * Ppart
    # global probabilities agree with an independent softmax of the dequantized scores
    c = float(np.float32(1) / np.sqrt(np.float32(64)))
    s = (Kt[:, kvh].astype(np.int64) @ q_i8[b, h].astype(np.int64)) * float(q_s[b, h]) * sK[:, kvh] * c
    pe = np.exp(s - s.max())
    np.testing.assert_allclose(P, pe / pe.sum(), rtol=1e-5, atol=1e-9)
    eV = vd - sV[:, None] * Vq
    eW = tr["W"] - tr["sW"] * tr["Wq"]
    O_exact = P @ vd
    lhs = O_exact - out[b, h]
    rhs = P @ eV + (tr["c"] * eW) @ Vq
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
    assert np.all(np.abs(eV) <= sV[:, None] * (0.5 + 1e-5))
    assert np.all(np.abs(eW) <= tr["sW"] * (0.5 + 1e-5))
    bound = P @ (sV[:, None] / 2 * np.ones_like(Vq)) + (tr["c"] * tr["sW"] / 2) @ np.abs(Vq)
    assert np.all(np.abs(lhs) <= bound * (1 + 1e-4))
    # the groups the trace shows are aligned 32-token runs with one scale each
    for j0 in range(0, L, 32):
        assert np.unique(tr["sW"][j0:j0 + 32]).size == 1
        Wg = tr["W"][j0:j0 + 32]
        assert tr["Wq"][j0 + int(np.argmax(Wg))] == pmax
        assert tr["Wq"][j0:j0 + 32].min() >= 0


def test_uint8_codes_halve_the_probability_error():
    # With V exact (integer V, sV = 1 so eV = 0) the only error left is the
    # probability rounding, bounded by sW / 2 per token; sW = A / 255 is half of
    # A / 127, so the UINT8 codes' error must come out clearly smaller.
    L, Hq, Hkv, D = 2000, 4, 1, 64
    w = _small_decode([L], Hq=Hq, Hkv=Hkv, D=D, seed=21)
    rng = np.random.default_rng(22)
    k, _ = w.kv(0)
    v = _integer_v(rng, L, Hkv, D)
    cache = orc.kv_quant_write(k, wl.bf16_bits(v), w.slots(0), w.num_blocks, w.block_size)
    q_i8, q_s = oracle_query(w)
    Kt, Vt, sK, sV = gather_int8(cache, w.block_tables[0], L, Hkv, D)
    c = float(np.float32(1) / np.sqrt(np.float32(D)))
    errs = {}
    for pmax in (127, 255):
        out = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size, fp32_decisions=False,
                              pmax=pmax)
        e = []
        for h in range(Hq):
            s = (Kt[:, 0].astype(np.int64) @ q_i8[0, h].astype(np.int64)) * float(q_s[0, h]) * sK[:, 0] * c
            p = np.exp(s - s.max())
            e.append(np.abs(out[0, h] - (p / p.sum()) @ (Vt[:, 0] * sV[:, 0, None]).astype(np.float64)))
        errs[pmax] = np.mean(e)
    assert errs[255] < 0.7 * errs[127], errs


# --------------------------------------------------------------------------- prefix
def _prefix_case(H, C, Hq=6, Hkv=2, D=32, seed=0):
    w = wl.PrefixWorkload("t", Hq, Hkv, D, H, C, seed=seed)
    k, v = w.kv()
    q = w.q()
    cache = orc.kv_quant_write(k, v, w.slots(), w.num_blocks, w.block_size)
    q_i8, q_s = quantize_rows(q)
    return w, k, v, q, cache, q_i8, q_s


@pytest.mark.parametrize("H,C", [(0, 5), (64, 1), (100, 37), (256, 70)])
def test_prefix_vs_fp64_causal(H, C):
    w, k, v, q, cache, q_i8, q_s = _prefix_case(H, C, seed=H + C)
    out = orc.prefix_attn(q_i8, q_s, cache, w.block_table, H, w.block_size)
    ref = orc.attention_fp64(orc.bf16_to_f64(q), orc.bf16_to_f64(k), orc.bf16_to_f64(v), H + np.arange(C) + 1)
    # Rows that see >= 32 keys average the per-token V quantization error (|eV| <= sV/2,
    # sV ~ 3/127 for N(0,1)) down to well under 2e-2; rows with a handful of keys keep
    # most of one token's error and get 5e-2.  A dropped term or a wrong mask is O(1).
    many = H + np.arange(C) + 1 >= 32
    err = np.abs(out - ref).max(axis=(1, 2))
    assert np.all(err[many] < 2e-2)
    assert np.all(err[~many] < 5e-2)


def test_prefix_equal_scores_causal_mean():
    # Q = 0 and sV = 1: chunk row j must return the mean of V over positions 0 .. H + j
    # (a causal mask that leaked or cut one key would miss).
    H, C, Hq, Hkv, D = 90, 40, 2, 1, 32
    w = wl.PrefixWorkload("t", Hq, Hkv, D, H, C, seed=3)
    k, _ = w.kv()
    v = _integer_v(np.random.default_rng(8), H + C, Hkv, D)
    cache = orc.kv_quant_write(k, wl.bf16_bits(v), w.slots(), w.num_blocks, w.block_size)
    q_i8 = np.zeros((C, Hq, D), np.int8)
    q_s = np.zeros((C, Hq), np.float32)
    out = orc.prefix_attn(q_i8, q_s, cache, w.block_table, H, w.block_size, fp32_decisions=False)
    csum = np.cumsum(v[:, 0].astype(np.float64), axis=0)
    for j in range(C):
        np.testing.assert_allclose(out[j, 0], csum[H + j] / (H + j + 1), rtol=0, atol=1e-10)


def test_prefix_equals_decode_and_tile_invariance():
    # Row j of the chunk sees the same H + j + 1 keys as a decode step with that history;
    # with fp64 decisions the online form (unnormalized p~), the partitioned form and
    # any key tile that is a multiple of 32 agree to rounding.
    H, C = 200, 50
    w, k, v, q, cache, q_i8, q_s = _prefix_case(H, C, Hq=4, Hkv=2, D=32, seed=5)
    out = orc.prefix_attn(q_i8, q_s, cache, w.block_table, H, w.block_size, fp32_decisions=False)
    for tile in (32, 128, 512):
        o2 = orc.prefix_attn(q_i8, q_s, cache, w.block_table, H, w.block_size, key_tile=tile, fp32_decisions=False)
        np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12)
    rows = np.array([0, 7, 31, 49], np.int32)
    bt = np.broadcast_to(w.block_table, (rows.size, w.block_table.size)).copy()
    dec = orc.decode_attn(q_i8[rows], q_s[rows], cache, bt, (H + rows + 1).astype(np.int32), w.block_size,
                          fp32_decisions=False)
    np.testing.assert_allclose(dec, out[rows], rtol=0, atol=1e-12)
    sub = orc.prefix_attn(q_i8, q_s, cache, w.block_table, H, w.block_size, rows=rows, fp32_decisions=False)
    np.testing.assert_allclose(sub, out[rows], rtol=0, atol=0)


def test_empty_sequence_gives_zero_row():
    w = _small_decode([0, 20], Hq=2, Hkv=1, D=16, seed=1)
    cache = orc.kv_quant_write(*w.kv(1), w.slots(1), w.num_blocks, w.block_size)
    q_i8, q_s = oracle_query(w)
    out = orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size)
    assert not out[0].any() and np.abs(out[1]).max() > 0


# --------------------------------------------------------------------------- BF16-KV comparison oracle
def test_bf16_decode_matches_dense_fp64():
    w = _small_decode([129, 40], Hq=6, Hkv=2, D=64, seed=2)
    cache = None
    for b in range(w.B):
        k, v = w.kv(b)
        cache = orc.bf16_kv_write(k, v, w.slots(b), w.num_blocks, w.block_size, **({} if cache is None else cache))
    out = orc.bf16_decode_attn(w.q(), cache, w.block_tables, w.seq_lens, w.block_size)
    for b in range(w.B):
        kd, vd = (orc.bf16_to_f64(a) for a in w.kv(b))
        ref = orc.attention_fp64(orc.bf16_to_f64(w.q()[b:b + 1]), kd, vd, [int(w.seq_lens[b])])
        np.testing.assert_allclose(out[b], ref[0], rtol=0, atol=1e-12)
