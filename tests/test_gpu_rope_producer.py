"""GPU parity of the fused producer (kv_rope_quant_write): Q/K RMSNorm and RoPE
in fp32 with a fixed operation order, then the INT8 quantization and the paged
scatter.  Cache bytes, scales, the quantized query and the bf16 copies of the
transformed vectors must be bit-identical to the oracle on the same inputs."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

BS = wl.BLOCK_SIZE


def _assert_same(gpu: dict, ref: dict, keys):
    for k in keys:
        g = host(gpu[k])
        r = ref[k]
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        if g.dtype == np.int16:
            g = g.view(np.uint16)
        bad = np.flatnonzero(g.ravel() != r.ravel())
        assert bad.size == 0, f"{k}: {bad.size} mismatches, first at flat index {bad[:5]}"


def _run(k, v, slots, num_blocks, positions=None, cos_sin=None, rotary_dim=0, q=None, q_norm_weight=None,
         k_norm_weight=None, eps=1e-6, quantize_q=True, q_out=False, k_out=False, expect_error=0, k_smooth=None):
    T, Hkv, D = k.shape
    gc = i8.alloc_int8_cache(num_blocks, Hkv, D)
    extra = {}
    if q is not None:
        extra["q"] = dev(q)
        if quantize_q:
            extra.update(q_i8=torch.zeros(q.shape, dtype=torch.int8, device="cuda"),
                         q_scale=torch.zeros(q.shape[:2], dtype=torch.float32, device="cuda"))
        if q_out:
            extra["q_out"] = torch.zeros(q.shape, dtype=torch.int16, device="cuda")
    if k_out:
        extra["k_out"] = torch.zeros(k.shape, dtype=torch.int16, device="cuda")
    i8.kv_rope_quant_write(dev(k), dev(v), dev(slots), **gc,
                           positions=None if positions is None else dev(positions),
                           cos_sin=None if cos_sin is None else dev(cos_sin), rotary_dim=rotary_dim,
                           q_norm_weight=None if q_norm_weight is None else dev(q_norm_weight),
                           k_norm_weight=None if k_norm_weight is None else dev(k_norm_weight),
                           norm_eps=eps, k_smooth=None if k_smooth is None else dev(k_smooth), **extra)
    torch.cuda.synchronize()
    assert i8.device_error() == expect_error
    gc.update({kk: extra[kk] for kk in ("q_i8", "q_scale", "q_out", "k_out") if kk in extra})
    ref = orc.kv_rope_quant_write(k, v, slots, num_blocks, BS, positions=positions, cos_sin=cos_sin,
                                  rotary_dim=rotary_dim, q=q, q_norm_weight=q_norm_weight,
                                  k_norm_weight=k_norm_weight, eps=eps, quantize_q=quantize_q, q_out=q_out,
                                  k_out=k_out, k_smooth=k_smooth)
    return gc, ref


ALL = ["k_cache", "v_cache", "k_scale", "v_scale", "q_i8", "q_scale", "q_out", "k_out"]


def test_rope_producer_gqa_workload_bit_exact():
    # 8192 tokens at positions 0..8191, 32 / 8 heads, head_dim 128, full rotation,
    # both norms, 2% outliers x10, block-aligned slots (the transposed V path).
    p = wl.producer_rope_tokens()
    gc, ref = _run(p["k"], p["v"], p["slots"], p["num_blocks"], positions=p["positions"], cos_sin=p["cos_sin"],
                   rotary_dim=p["rotary_dim"], q=p["q"], q_norm_weight=p["q_norm_weight"],
                   k_norm_weight=p["k_norm_weight"], q_out=True, k_out=True)
    assert ref["status"] == 0
    _assert_same(gc, ref, ALL)


@pytest.mark.parametrize("D,rd,norm", [(128, 128, "qk"), (128, 64, "k"), (128, 32, ""), (128, 0, "qk"),
                                       (256, 256, "qk"), (256, 64, "q"), (256, 128, "qk"), (256, 0, "")])
def test_rope_producer_scattered_bit_exact(D, rd, norm):
    # random slots (byte-scatter V path) with a skipped token, ragged last tile,
    # random positions, partial rotations, norms on Q and/or K
    T, Hkv, Hq = 45, 4, 12
    rng = np.random.default_rng(D * 7 + rd)
    NB = (T + BS - 1) // BS + 3
    slots = rng.permutation(NB * BS)[:T].astype(np.int32)
    slots[T // 3] = -1
    k = wl.randn_bf16(rng, (T, Hkv, D))
    v = wl.randn_bf16(rng, (T, Hkv, D))
    q = wl.randn_bf16(rng, (T, Hq, D))
    pos = rng.integers(0, 5000, size=T).astype(np.int32) if rd else None
    cs = wl.rope_cos_sin(5000, rd, base=1e6) if rd else None
    qw = wl.norm_weight_bf16(rng, D) if "q" in norm else None
    kw = wl.norm_weight_bf16(rng, D) if "k" in norm else None
    gc, ref = _run(k, v, slots, NB, positions=pos, cos_sin=cs, rotary_dim=rd, q=q, q_norm_weight=qw,
                   k_norm_weight=kw, q_out=True, k_out=True)
    _assert_same(gc, ref, ALL)


@pytest.mark.parametrize("D,rd,Hkv,Hq,T", [(256, 192, 6, 18, 150), (128, 96, 3, 9, 400)])
def test_rope_producer_uneven_heads_partial_rotation_bit_exact(D, rd, Hkv, Hq, T):
    # Partial rotations whose rotary runs do not fill the lanes of a vector (the
    # lanes past them hold the unrotated tail) with head counts that leave
    # warps without a task in some units; block-aligned slots, both norms
    rng = np.random.default_rng(rd + Hkv)
    tables, NB = wl.paged_tables([T], perm_seed=rd)
    slots = wl.slot_mapping(tables[0], np.arange(T))
    k = wl.randn_bf16(rng, (T, Hkv, D))
    v = wl.randn_bf16(rng, (T, Hkv, D))
    q = wl.randn_bf16(rng, (T, Hq, D))
    pos = np.arange(T, dtype=np.int32)
    gc, ref = _run(k, v, slots, NB, positions=pos, cos_sin=wl.rope_cos_sin(T, rd), rotary_dim=rd, q=q,
                   q_norm_weight=wl.norm_weight_bf16(rng, D), k_norm_weight=wl.norm_weight_bf16(rng, D),
                   q_out=True, k_out=True)
    _assert_same(gc, ref, ALL)


def test_rope_producer_aligned_tiles_without_query():
    # one sequence, positions 32 .. 32+96: every tile fills one block; no query
    D, Hkv, rd = 256, 2, 256
    tables, NB = wl.paged_tables([160])
    positions = np.arange(32, 128, dtype=np.int32)
    slots = wl.slot_mapping(tables[0], positions)
    rng = np.random.default_rng(3)
    k = wl.randn_bf16(rng, (96, Hkv, D))
    v = wl.randn_bf16(rng, (96, Hkv, D))
    kw = wl.norm_weight_bf16(rng, D)
    gc, ref = _run(k, v, slots, NB, positions=positions, cos_sin=wl.rope_cos_sin(160, rd), rotary_dim=rd,
                   k_norm_weight=kw)
    _assert_same(gc, ref, ["k_cache", "v_cache", "k_scale", "v_scale"])


def test_rope_producer_query_copy_only():
    # q_i8 / q_scale omitted: only the transformed bf16 query is written
    D, Hkv, Hq, T, rd = 128, 2, 8, 20, 128
    rng = np.random.default_rng(8)
    NB = 3
    slots = np.arange(T, dtype=np.int32)
    k, v, q = (wl.randn_bf16(rng, (T, H, D)) for H in (Hkv, Hkv, Hq))
    gc, ref = _run(k, v, slots, NB, positions=np.arange(T, dtype=np.int32) * 3, cos_sin=wl.rope_cos_sin(64, rd),
                   rotary_dim=rd, q=q, q_norm_weight=wl.norm_weight_bf16(rng, D), quantize_q=False, q_out=True)
    _assert_same(gc, ref, ["k_cache", "v_cache", "k_scale", "v_scale", "q_out"])


def test_rope_producer_position_outside_table():
    # positions 10 and -1 lie outside a 10-row table: those tokens are skipped
    # (nothing written), error 4 is recorded, the others match the oracle.
    D, Hkv, Hq, rd = 128, 2, 4, 128
    rng = np.random.default_rng(4)
    T = 6
    slots = np.arange(T, dtype=np.int32)
    k, v, q = (wl.randn_bf16(rng, (T, H, D)) for H in (Hkv, Hkv, Hq))
    pos = np.array([0, 3, 10, 9, -1, 2], np.int32)
    gc, ref = _run(k, v, slots, 1, positions=pos, cos_sin=wl.rope_cos_sin(10, rd), rotary_dim=rd, q=q,
                   q_out=True, k_out=True, expect_error=4)
    assert ref["status"] == orc.BAD_POSITION
    _assert_same(gc, ref, ALL)


def test_rope_producer_identity_table_matches_plain_producer():
    # cos = 1, sin = 0, no norm: the fused kernel writes what the plain one writes
    D, Hkv, Hq, T, rd = 256, 4, 8, 33, 256
    rng = np.random.default_rng(12)
    NB = 4
    slots = rng.permutation(NB * BS)[:T].astype(np.int32)
    k, v, q = (wl.randn_bf16(rng, (T, H, D)) for H in (Hkv, Hkv, Hq))
    cs = np.concatenate([np.ones((4, rd // 2), np.float32), np.zeros((4, rd // 2), np.float32)], axis=1)
    a = i8.alloc_int8_cache(NB, Hkv, D)
    b = i8.alloc_int8_cache(NB, Hkv, D)
    qa = torch.zeros((T, Hq, D), dtype=torch.int8, device="cuda")
    qb = torch.zeros_like(qa)
    sa = torch.zeros((T, Hq), dtype=torch.float32, device="cuda")
    sb = torch.zeros_like(sa)
    i8.kv_quant_write(dev(k), dev(v), dev(slots), **a, q=dev(q), q_i8=qa, q_scale=sa)
    i8.kv_rope_quant_write(dev(k), dev(v), dev(slots), **b, positions=dev(np.full(T, 3, np.int32)),
                           cos_sin=dev(cs), rotary_dim=rd, q=dev(q), q_i8=qb, q_scale=sb)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    for key in a:
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(qa, qb) and torch.equal(sa, sb)


@pytest.mark.parametrize("D,rd", [(128, 128), (256, 64)])
def test_rope_producer_k_smoothing_bit_exact(D, rd):
    # per-channel K smoothing after norm and rotation: factors sqrt(max |K_c|)
    # of a channel-outlier K (not powers of two, so every product rounds)
    T, Hkv, Hq = 40, 4, 12
    w = wl.DecodeWorkload("sm", Hq, Hkv, D, [T], seed=D + rd, outlier_channels=4)
    k, v = w.kv(0)
    rng = np.random.default_rng(rd)
    q = wl.randn_bf16(rng, (T, Hq, D))
    smooth = np.sqrt(np.abs(wl.bf16_values(k)).max(axis=0)).astype(np.float32)
    slots = w.slots(0).copy()
    slots[5] = -1
    gc, ref = _run(k, v, slots, w.num_blocks, positions=np.arange(T, dtype=np.int32) * 7,
                   cos_sin=wl.rope_cos_sin(300, rd), rotary_dim=rd, q=q, q_norm_weight=wl.norm_weight_bf16(rng, D),
                   k_norm_weight=wl.norm_weight_bf16(rng, D), q_out=True, k_out=True, k_smooth=smooth)
    _assert_same(gc, ref, ALL)
