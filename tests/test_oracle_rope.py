"""Pins for the oracle's fused producer (Q/K RMSNorm, RoPE, then INT8 quantization).

The pages put RoPE on Q and K inside the producer, before the absmax and the
quantization ("gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §2.2), and
the served model applies a per-head RMSNorm to Q and K before RoPE (same page,
§5.3).  The checks below tie the oracle to facts that do not depend on its own
code: special rotations that are exact permutations, the identity rotation,
fp64 evaluations of the two formulas within their rounding bounds, closed forms
of RMSNorm on constant vectors, scale invariance, and a hand-summed case that
fixes the order of the sum of squares."""
import numpy as np
import pytest

import workloads as wl
from oracle import oracle as orc

BS = wl.BLOCK_SIZE
U32 = 2.0 ** -24      # fp32 unit roundoff
UBF = 2.0 ** -8       # bf16 unit roundoff (8 significant bits)


def _inputs(T, Hkv, D, Hq=0, seed=0):
    rng = np.random.default_rng(seed)
    k = wl.randn_bf16(rng, (T, Hkv, D))
    v = wl.randn_bf16(rng, (T, Hkv, D))
    q = wl.randn_bf16(rng, (T, Hq, D)) if Hq else None
    NB = (T + BS - 1) // BS + 2
    slots = rng.permutation(NB * BS)[:T].astype(np.int32)
    return k, v, q, slots, NB


def _table(rows, rd, cos, sin):
    t = np.empty((rows, rd), np.float32)
    t[:, : rd // 2] = cos
    t[:, rd // 2:] = sin
    return t


def _same(a, b, keys):
    for key in keys:
        x, y = a[key], b[key]
        if x.dtype == np.float32:
            x, y = x.view(np.uint32), y.view(np.uint32)
        assert np.array_equal(x, y), key


@pytest.mark.parametrize("rd", [0, 32, 128])
def test_identity_rotation_is_the_plain_producer(rd):
    # cos = 1, sin = 0 on every row, no norm: the fused producer must reduce to
    # the plain quantize-and-scatter, byte for byte.
    T, Hkv, D, Hq = 21, 2, 128, 4
    k, v, q, slots, NB = _inputs(T, Hkv, D, Hq)
    slots[3] = -1
    plain = orc.kv_quant_write(k, v, slots, NB, BS, q=q)
    pos = np.arange(T, dtype=np.int32)
    cs = _table(T, rd, 1.0, 0.0) if rd else None
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, positions=pos if rd else None, cos_sin=cs,
                                    rotary_dim=rd, q=q, q_out=True, k_out=True)
    assert fused["status"] == 0
    _same(plain, fused, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])
    # the bf16 copies of an untouched vector are the inputs themselves
    assert np.array_equal(fused["k_out"], k) and np.array_equal(fused["q_out"], q)


@pytest.mark.parametrize("D,rd", [(128, 128), (128, 64), (256, 32), (256, 256)])
def test_quarter_turn_is_a_signed_permutation(D, rd):
    # cos = 0, sin = 1: (a, b) -> (-b, a) on the rotated half-pairs, exactly, and
    # the dims past rd are untouched.  Absmax quantization commutes with a signed
    # permutation, so the cache must equal the plain producer on the permuted input.
    T, Hkv, Hq = 19, 2, 6
    k, v, q, slots, NB = _inputs(T, Hkv, D, Hq, seed=D + rd)
    h = rd // 2

    def turn(x):
        y = x.copy()
        y[..., :h] = x[..., h:rd] ^ np.uint16(0x8000)   # -b: flip the bf16 sign bit
        y[..., h:rd] = x[..., :h]
        return y

    pos = np.full(T, 7, np.int32)
    cs = _table(8, rd, 0.0, 1.0)
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, positions=pos, cos_sin=cs, rotary_dim=rd, q=q,
                                    q_out=True, k_out=True)
    plain = orc.kv_quant_write(turn(k), v, slots, NB, BS, q=turn(q))
    _same(plain, fused, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])
    # -0.0 from negating +0.0 is the same value; compare as values
    assert np.array_equal(wl.bf16_values(fused["k_out"]), wl.bf16_values(turn(k)))
    assert np.array_equal(wl.bf16_values(fused["q_out"]), wl.bf16_values(turn(q)))


def _rope_fp64(x, pos, cs, rd):
    """fp64 rotate-half with the fp32 table values as given."""
    x = wl.bf16_values(x).astype(np.float64)
    y = x.copy()
    h = rd // 2
    c = cs[pos][:, None, :h].astype(np.float64)
    s = cs[pos][:, None, h:].astype(np.float64)
    a, b = x[..., :h], x[..., h:rd]
    y[..., :h] = a * c - b * s
    y[..., h:rd] = b * c + a * s
    mag = np.abs(x).copy()
    mag[..., :h] = np.abs(a * c) + np.abs(b * s)
    mag[..., h:rd] = np.abs(b * c) + np.abs(a * s)
    return y, mag


@pytest.mark.parametrize("rd", [64, 128])
def test_rotation_matches_fp64_within_rounding(rd):
    # Distinct positions per token, a real table: the bf16 copy lies within one
    # bf16 rounding of the fp64 rotation plus the fp32 product/sum roundings, and
    # the cache holds the quantized rotated vector (within half a code).
    T, Hkv, D = 40, 2, 128
    k, v, _, slots, NB = _inputs(T, Hkv, D, seed=rd)
    rng = np.random.default_rng(9)
    pos = rng.integers(0, 4096, size=T).astype(np.int32)
    cs = wl.rope_cos_sin(4096, rd)
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, positions=pos, cos_sin=cs, rotary_dim=rd, k_out=True)
    y, mag = _rope_fp64(k, pos, cs, rd)
    got = wl.bf16_values(fused["k_out"]).astype(np.float64)
    bound = UBF * np.abs(y) + 3 * U32 * mag + 1e-30
    assert np.all(np.abs(got - y) <= bound)
    # dequantized cache rows against the fp64 rotation
    blk, off = slots // BS, slots % BS
    for h in range(Hkv):
        codes = fused["k_cache"][blk, h].reshape(T, D // 16, BS, 16)[np.arange(T), :, off, :].reshape(T, D)
        sc = fused["k_scale"][blk, off, h].astype(np.float64)
        err = np.abs(codes * sc[:, None] - y[:, h, :])
        assert np.all(err <= 0.5 * sc[:, None] * (1 + 1e-5) + 3 * U32 * mag[:, h, :] + 1e-30)


def _rms_fp64(x, w, eps):
    x = wl.bf16_values(x).astype(np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * wl.bf16_values(w).astype(np.float64)


@pytest.mark.parametrize("D,eps", [(128, 1e-6), (256, 1e-6), (128, 0.5)])
def test_rmsnorm_matches_fp64(D, eps):
    # sum of squares (log2 D roundings), mean, +eps, sqrt, reciprocal and two
    # products: about 9 fp32 roundings relative, bounded by 16 here.
    T, Hkv, Hq = 17, 2, 4
    k, v, q, slots, NB = _inputs(T, Hkv, D, Hq, seed=D)
    rng = np.random.default_rng(5)
    qw, kw = wl.norm_weight_bf16(rng, D), wl.norm_weight_bf16(rng, D)
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, q=q, q_norm_weight=qw, k_norm_weight=kw, eps=eps,
                                    q_out=True, k_out=True, quantize_q=False)
    assert "q_i8" not in fused
    for x, w, key in ((k, kw, "k_out"), (q, qw, "q_out")):
        y = _rms_fp64(x, w, eps)
        got = wl.bf16_values(fused[key]).astype(np.float64)
        assert np.all(np.abs(got - y) <= UBF * np.abs(y) + 16 * U32 * np.abs(y) + 1e-30), key


def test_rmsnorm_constant_vector_closed_form():
    # x_i = +-2^j for all i, eps = 0: mean x^2 = 4^j, rms = 2^j, 1/rms exact, so
    # y_i = sign(x) * w_i exactly -- with a random weight this also fixes which
    # weight entry meets which dim.
    D = 128
    rng = np.random.default_rng(2)
    w = wl.norm_weight_bf16(rng, D)
    signs = np.array([1.0, -1.0, 1.0, -1.0], np.float32)
    mags = np.array([2.0 ** -3, 1.0, 2.0 ** 5, 2.0 ** 11], np.float32)
    k = np.repeat((signs * mags)[:, None, None], D, axis=2).astype(np.float32)
    kb = wl.bf16_bits(k)
    slots = np.arange(4, dtype=np.int32)
    fused = orc.kv_rope_quant_write(kb, kb, slots, 1, BS, k_norm_weight=w, eps=0.0, k_out=True)
    expect = signs[:, None] * wl.bf16_values(w)[None, :]
    assert np.array_equal(wl.bf16_values(fused["k_out"][:, 0, :]), expect.astype(np.float32))


def test_rmsnorm_scale_invariance():
    # eps = 0: multiplying a vector by 2^k scales every intermediate exactly, so
    # the normalized output (and its cache bytes) must not change at all.
    D, T, Hkv = 128, 9, 2
    k, v, _, slots, NB = _inputs(T, Hkv, D, seed=11)
    w = wl.norm_weight_bf16(np.random.default_rng(3), D)
    base = orc.kv_rope_quant_write(k, v, slots, NB, BS, k_norm_weight=w, eps=0.0, k_out=True)
    for e in (-20, 7, 40):
        ks = wl.bf16_bits(wl.bf16_values(k) * np.float32(2.0 ** e))
        r = orc.kv_rope_quant_write(ks, v, slots, NB, BS, k_norm_weight=w, eps=0.0, k_out=True)
        _same(base, r, ["k_cache", "k_scale", "v_cache", "v_scale", "k_out"])


def test_sum_of_squares_order_is_the_balanced_tree():
    # x = (2^12, 1, 1, ..., 1), D = 128.  Exact sum of squares 2^24 + 127.  In
    # fp32 a left-to-right sum stays at 2^24 (each +1 is a tie, rounded to even);
    # the balanced tree adds 2^24 + 1 -> 2^24 at the first level and then the
    # exact partial sums 2, 4, ..., 64 of the other subtrees: 2^24 + 126.
    D = 128
    x = np.ones(D, np.float32)
    x[0] = 4096.0
    kb = wl.bf16_bits(x[None, None, :])
    w = wl.bf16_bits(np.ones(D, np.float32))
    got = orc.kv_rope_quant_write(kb, kb, np.zeros(1, np.int32), 1, BS, k_norm_weight=w, eps=0.0)["k_scale"]

    # The bf16 copy is too coarse to see the difference; the fp32 scale
    # amax / 127 = (2^12 / rms) / 127 is not.
    def scale(ss):
        inv = np.float32(1.0) / np.sqrt(np.float32(ss) * np.float32(1.0 / D))
        return np.float32(np.float32(4096.0) * inv) / np.float32(127.0)

    tree, seq = scale(2.0 ** 24 + 126), scale(2.0 ** 24)
    assert tree != seq
    assert got[0, 0, 0] == tree


def test_norm_comes_before_rope():
    # With a non-uniform weight the two orders differ far beyond rounding;
    # the bf16 copy must match fp64 rope(rmsnorm(x)).
    T, Hkv, D, rd = 12, 2, 128, 128
    k, v, _, slots, NB = _inputs(T, Hkv, D, seed=13)
    w = wl.norm_weight_bf16(np.random.default_rng(4), D)
    pos = np.arange(100, 100 + T, dtype=np.int32)
    cs = wl.rope_cos_sin(256, rd)
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, positions=pos, cos_sin=cs, rotary_dim=rd,
                                    k_norm_weight=w, eps=1e-6, k_out=True)
    n = _rms_fp64(k, w, 1e-6)
    h = rd // 2
    c = cs[pos][:, None, :h].astype(np.float64)
    s = cs[pos][:, None, h:].astype(np.float64)
    y = n.copy()
    y[..., :h] = n[..., :h] * c - n[..., h:] * s
    y[..., h:] = n[..., h:] * c + n[..., :h] * s
    got = wl.bf16_values(fused["k_out"]).astype(np.float64)
    scale = np.abs(n).max()
    assert np.all(np.abs(got - y) <= UBF * np.abs(y) + 40 * U32 * scale)


def test_v_is_never_transformed():
    T, Hkv, D = 16, 2, 128
    k, v, _, slots, NB = _inputs(T, Hkv, D, seed=21)
    w = wl.norm_weight_bf16(np.random.default_rng(6), D)
    cs = wl.rope_cos_sin(64, 128)
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, positions=np.arange(T, dtype=np.int32) + 30,
                                    cos_sin=cs, rotary_dim=128, k_norm_weight=w, eps=1e-6)
    plain = orc.kv_quant_write(k, v, slots, NB, BS)
    _same(plain, fused, ["v_cache", "v_scale"])
    assert not np.array_equal(plain["k_cache"], fused["k_cache"])


def test_bad_position_skips_only_that_token():
    T, Hkv, D, Hq = 6, 1, 128, 2
    k, v, q, slots, NB = _inputs(T, Hkv, D, Hq, seed=31)
    cs = wl.rope_cos_sin(10, 128)
    pos = np.array([0, 3, 10, 9, -1, 2], np.int32)
    r = orc.kv_rope_quant_write(k, v, slots, NB, BS, positions=pos, cos_sin=cs, rotary_dim=128, q=q,
                                k_out=True)
    assert r["status"] == orc.BAD_POSITION
    good = np.array([0, 1, 3, 5])
    ok = orc.kv_rope_quant_write(k[good], v[good], slots[good], NB, BS, positions=pos[good], cos_sin=cs,
                                 rotary_dim=128, q=q[good], k_out=True)
    assert ok["status"] == 0
    _same(ok, r, ["k_cache", "v_cache", "k_scale", "v_scale"])
    for key in ("q_i8", "q_scale", "k_out"):
        assert np.array_equal(r[key][good], ok[key])
        assert not r[key][[2, 4]].any()


# --------------------------------------------------------------------------- per-channel K smoothing
def test_unit_smoothing_changes_nothing():
    T, Hkv, D, Hq = 20, 2, 128, 6
    k, v, q, slots, NB = _inputs(T, Hkv, D, Hq, seed=41)
    a = orc.kv_rope_quant_write(k, v, slots, NB, BS, q=q)
    b = orc.kv_rope_quant_write(k, v, slots, NB, BS, q=q, k_smooth=np.ones((Hkv, D), np.float32))
    _same(a, b, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])


@pytest.mark.parametrize("D,Hkv,Hq", [(128, 2, 6), (256, 4, 4)])
def test_power_of_two_smoothing_is_exact_channel_scaling(D, Hkv, Hq):
    # s = 2^e per (KV head, channel): K' = K 2^-e and Q' = Q 2^e exactly, so the
    # caches must equal the plain producer's on bf16 inputs scaled channel-wise
    # in numpy -- which fixes which factor meets which channel, that K takes 1/s
    # and Q takes s, and that query head hq uses KV head hq / (Hq / Hkv).
    T = 19
    k, v, q, slots, NB = _inputs(T, Hkv, D, Hq, seed=D + Hkv)
    e = np.random.default_rng(7).integers(-4, 5, size=(Hkv, D))
    s = np.ldexp(np.ones((Hkv, D), np.float32), e).astype(np.float32)
    G = Hq // Hkv
    ks = wl.bf16_bits(wl.bf16_values(k) / s[None, :, :])
    qs = wl.bf16_bits(wl.bf16_values(q) * np.repeat(s, G, axis=0)[None, :, :])
    fused = orc.kv_rope_quant_write(k, v, slots, NB, BS, q=q, k_smooth=s)
    plain = orc.kv_quant_write(ks, v, slots, NB, BS, q=qs)
    _same(plain, fused, ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale"])


def test_smoothing_reduces_decode_error_on_channel_outliers():
    # K with 4 outlier channels x20 per KV head (the decode_outlier recipe, at a
    # shorter history): smoothing with s = sqrt(max |K_c|) per channel moves the
    # outliers' range half into Q; the quantized decode must come out closer to
    # fp64 attention on the unquantized values.
    L, Hq, Hkv, D = 2048, 8, 2, 128
    w = wl.DecodeWorkload("sm", Hq, Hkv, D, [L], seed=3, outlier_channels=4)
    k, v = w.kv(0)
    q = w.q()
    slots = w.slots(0)
    kf = wl.bf16_values(k).astype(np.float64)
    s = np.sqrt(np.abs(kf).max(axis=0)).astype(np.float32)   # [Hkv, D]
    errs = []
    for ks in (None, s):
        # history K/V through the producer; the query alone (slot -1 rows)
        c = orc.kv_rope_quant_write(k, v, slots, w.num_blocks, BS, k_smooth=ks)
        qq = orc.kv_rope_quant_write(np.zeros((1, Hkv, D), np.uint16), np.zeros((1, Hkv, D), np.uint16),
                                     np.array([-1], np.int32), w.num_blocks, BS, q=q, k_smooth=ks)
        out = orc.decode_attn(qq["q_i8"], qq["q_scale"], c, w.block_tables, w.seq_lens, BS)
        ref = orc.attention_fp64(orc.bf16_to_f64(q), kf, wl.bf16_values(v).astype(np.float64), np.array([L]),
                                 softmax_scale=float(np.float32(1) / np.sqrt(np.float32(D))))
        errs.append(np.abs(out - ref).mean())
    assert errs[1] < 0.8 * errs[0], errs
