"""Pins of the oracle's quantizer and KV producer (CPU only).

What fixes the answer here is the pages' quantization rule ("gfx936 DCU上实现INT8
KV与INT8 MMAC Attention推理优化" §2.1) and its cache layouts (§2.3), checked
through worked cases, closed forms and the dequantization bound rather than a
second copy of the formula."""
import numpy as np
import pytest

import workloads as wl
from oracle import oracle as orc
from tests.helpers import read_golden, gather_int8


def test_golden_worked_cases():
    for vals, scale, codes in read_golden("quant_rne.txt"):
        x = wl.bf16_bits(np.array([float(v) for v in vals], np.float32))
        assert np.array_equal(wl.bf16_values(x), np.array([float(v) for v in vals], np.float32)), "fixture not bf16-exact"
        q, s = orc.quantize_vector(x)
        assert s == np.float32(scale[0])
        assert q.tolist() == [int(c) for c in codes]


@pytest.mark.parametrize("e", [-20, -7, 0, 3, 40])
def test_power_of_two_closed_form(e):
    # x = k * 2^e with integer |k| <= 127 and max |k| = 127: scale = 2^e exactly, codes = k.
    rng = np.random.default_rng(e + 100)
    k = rng.integers(-127, 128, size=256)
    k[rng.integers(0, 256)] = 127 * (1 if e % 2 else -1)
    x = wl.bf16_bits((k * 2.0 ** e).astype(np.float32))
    q, s = orc.quantize_vector(x)
    assert s == np.float32(2.0 ** e)
    assert np.array_equal(q.astype(np.int64), k)


@pytest.mark.parametrize("dist", ["normal", "outlier", "tiny"])
def test_dequant_bound_and_range(dist):
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = rng.standard_normal(256).astype(np.float32)
        if dist == "outlier":
            x[rng.integers(0, 256, 3)] *= 20
        if dist == "tiny":
            x *= np.float32(1e-30)
        xb = wl.bf16_bits(x)
        xv = wl.bf16_values(xb).astype(np.float64)
        q, s = orc.quantize_vector(xb)
        amax = np.abs(xv).max()
        assert abs(float(s) - amax / 127) <= amax / 127 * 2.0 ** -23
        assert np.abs(q.astype(int)).max() == 127          # the absmax element maps to +-127
        assert q.min() >= -127                               # -128 is never produced
        # |x - q s| <= s/2 up to the fp32 rounding of x / s
        err = np.abs(xv - q.astype(np.float64) * float(s))
        assert np.all(err <= float(s) * (0.5 + 1e-5))
        i = np.argmax(np.abs(xv))
        assert np.sign(q[i]) == np.sign(xv[i])


def test_zero_vector():
    q, s = orc.quantize_vector(np.zeros(128, np.uint16))
    assert s == 0.0 and not q.any()
    # -0.0 as well
    q, s = orc.quantize_vector(np.full(128, 0x8000, np.uint16))
    assert s == 0.0 and not q.any()


def test_producer_layout_and_skip():
    T, Hkv, Hq, D, bs, NB = 40, 2, 6, 32, 16, 7
    rng = np.random.default_rng(9)
    k = wl.randn_bf16(rng, (T, Hkv, D))
    v = wl.randn_bf16(rng, (T, Hkv, D))
    q = wl.randn_bf16(rng, (T, Hq, D))
    slots = rng.permutation(NB * bs)[:T].astype(np.int32)
    slots[3] = -1
    c = orc.kv_quant_write(k, v, slots, NB, bs, q=q)
    K5 = c["k_cache"].reshape(NB, Hkv, D // 16, bs, 16)
    V4 = c["v_cache"].reshape(NB, Hkv, D, bs)
    written = np.zeros((NB, bs), bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        blk, off = divmod(int(slots[t]), bs)
        written[blk, off] = True
        for h in range(Hkv):
            qk, sk = orc.quantize_vector(k[t, h])
            qv, sv = orc.quantize_vector(v[t, h])
            assert np.array_equal(K5[blk, h, :, off, :].ravel(), qk)
            assert np.array_equal(V4[blk, h, :, off], qv)
            assert c["k_scale"][blk, off, h] == sk and c["v_scale"][blk, off, h] == sv
    # untouched slots (including the skipped token's) stay zero
    assert not c["k_cache"].reshape(NB, Hkv, D // 16, bs, 16).transpose(0, 3, 1, 2, 4)[~written].any()
    assert not c["k_scale"][~written].any()
    for t in range(T):
        for h in range(Hq):
            qq, sq = orc.quantize_vector(q[t, h])
            assert np.array_equal(c["q_i8"][t, h], qq) and c["q_scale"][t, h] == sq


def test_gather_roundtrip_matches_dequant_bound():
    w = wl.DecodeWorkload("t", 4, 2, 64, [37], seed=1)
    k, v = w.kv(0)
    c = orc.kv_quant_write(k, v, w.slots(0), w.num_blocks, w.block_size)
    Kt, Vt, sK, sV = gather_int8(c, w.block_tables[0], 37, 2, 64)
    kd = orc.bf16_to_f64(k)
    assert np.all(np.abs(kd - Kt * sK[..., None].astype(np.float64)) <= sK[..., None] * (0.5 + 1e-5))
    vd = orc.bf16_to_f64(v)
    assert np.all(np.abs(vd - Vt * sV[..., None].astype(np.float64)) <= sV[..., None] * (0.5 + 1e-5))
