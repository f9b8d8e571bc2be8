"""The prefix kernel's integer contractions are exact.

The prefix chunk runs its INT8 contractions on the f16 tensor-core path
(tcgen05 kind::f16 with fp32 accumulation in tensor memory): every int8 code is
an exact f16, every product at most 127^2 and every partial sum below 2^24, so
the accumulators must come out as the exact int32 results the pages define
("gfx936 DCU上实现INT8 PV MMAC" §3: Wq x Vq accumulated in int32, at most
32 x 127 x 127 per group; §2: INT8 QK in int32).  i8kv_debug_prefix_i32 runs
the same kernel (its operand tiles, descriptors and tensor-memory reads) and
records S = Qq Kq^T, the probability codes Wq and each group's Wq x Vq as read
from tensor memory.  They are compared bit for bit with integer products
computed here from the cache bytes (numpy reshapes of the documented layouts;
float64 matmuls, exact below 2^53)."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import dev, host, gpu_quantize_rows
from tests.helpers import gather_int8

pytestmark = pytest.mark.gpu


def _debug_case(w: wl.PrefixWorkload):
    k, v = w.kv()
    H, C, Hq, Hkv, D = w.history, w.chunk, w.Hq, w.Hkv, w.D
    G = Hq // Hkv
    T = H + C
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    i8.kv_quant_write(dev(k), dev(v), dev(w.slots()), **cache)
    q_i8, q_s = gpu_quantize_rows(w.q(), Hkv, cache)
    bt = dev(w.block_table)
    s_acc, wq, pv, out_dbg = i8.debug_prefix_i32(q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                                 cache["v_scale"], bt, H)
    out = torch.empty((C, Hq, D), dtype=torch.float32, device="cuda")
    i8.int8_prefix_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"], cache["v_scale"], bt,
                        H)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    hc = {n: host(t) for n, t in cache.items()}
    oc = orc.kv_quant_write(k, v, w.slots(), w.num_blocks, w.block_size)
    assert all(np.array_equal(hc[n], oc[n]) for n in ("k_cache", "v_cache"))
    Kt, Vt, _, _ = gather_int8(hc, w.block_table, T, Hkv, D)
    qi = host(q_i8).astype(np.float64).reshape(C, Hkv, G, D)
    j = np.arange(C)[:, None]
    t = np.arange(T)[None, :]
    visible = t <= H + j  # [C, T]

    # S: int32 accumulators of every visible key, 0 elsewhere
    s_ref = np.einsum("ckgd,tkd->ckgt", qi, Kt.astype(np.float64), optimize=True).reshape(C, Hq, T)
    s_ref = np.where(visible[:, None, :], s_ref, 0.0)
    assert np.abs(s_ref).max() <= 4129024
    s_gpu = host(s_acc)
    assert np.array_equal(s_gpu.astype(np.float64), s_ref), \
        f"S differs at {np.argwhere(s_gpu != s_ref)[:5].tolist()}"

    # Wq: codes 0..127 on visible keys; the largest W of each group maps to 127
    ng = (T + 31) // 32
    codes = host(wq).reshape(C, Hq, ng * 32)
    vis_pad = np.zeros((C, ng * 32), bool)
    vis_pad[:, :T] = visible
    assert codes.max() <= 127 and not codes[~np.broadcast_to(vis_pad[:, None, :], codes.shape)].any()
    grp_vis = vis_pad.reshape(C, ng, 32).any(axis=2)  # [C, ng]
    gmax = codes.reshape(C, Hq, ng, 32).max(axis=3)
    assert np.all(gmax[np.broadcast_to(grp_vis[:, None, :], gmax.shape)] == 127)

    # PV: each group's sum_t Wq[t] Vq[t][d], as read from tensor memory
    Vp = np.zeros((ng * 32, Hkv, D))
    Vp[:T] = Vt
    wqf = codes.astype(np.float64).reshape(C, Hkv, G, ng, 32)
    pv_ref = np.einsum("ckgns,nskd->ckgnd", wqf, Vp.reshape(ng, 32, Hkv, D), optimize=True).reshape(C, Hq, ng, D)
    assert np.abs(pv_ref).max() <= 32 * 127 * 127
    pv_gpu = host(pv).astype(np.float64)
    assert np.array_equal(pv_gpu, pv_ref), f"PV differs at {np.argwhere(pv_gpu != pv_ref)[:5].tolist()}"

    # the recording instantiation computes the same output, bit for bit
    assert np.array_equal(host(out_dbg).view(np.uint32), host(out).view(np.uint32))
    return s_gpu, codes


@pytest.mark.parametrize("H,C,Hq,Hkv,D", [(0, 40, 8, 2, 128), (100, 37, 8, 1, 256), (300, 70, 24, 4, 256),
                                         (1000, 130, 32, 8, 128)])
def test_prefix_contractions_bit_exact(H, C, Hq, Hkv, D):
    _debug_case(wl.PrefixWorkload("dbg", Hq, Hkv, D, H, C, seed=H + C + D + 3))


def test_prefix_contractions_bit_exact_split_tail():
    # 650 chunk tokens x 32 q-heads over 8 KV heads = 168 row blocks: the last
    # wave's blocks are split over their key groups; every part records its own groups
    _debug_case(wl.PrefixWorkload("dbgsplit", 32, 8, 128, 64, 650, seed=17))


def test_prefix_contractions_at_the_int8_extremes():
    # every code +-127: S reaches D * 127^2 in magnitude (4,129,024 at head_dim
    # 256), still exact in the fp32 accumulator
    H, C, Hq, Hkv, D = 40, 24, 4, 1, 256
    w = wl.PrefixWorkload("extreme", Hq, Hkv, D, H, C, seed=9)
    rng = np.random.default_rng(10)
    sign = np.where(rng.random((H + C, Hkv, D)) < 0.5, -1.0, 1.0).astype(np.float32)
    k = wl.bf16_bits(sign)
    v = wl.bf16_bits(np.ones((H + C, Hkv, D), np.float32))
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    i8.kv_quant_write(dev(k), dev(v), dev(w.slots()), **cache)
    q = wl.bf16_bits(np.broadcast_to(sign[H:H + 1, :1, :], (C, Hq, D)).copy())
    q_i8, q_s = gpu_quantize_rows(q, Hkv, cache)
    s_acc, wq, pv, _ = i8.debug_prefix_i32(q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                           cache["v_scale"], dev(w.block_table), H)
    torch.cuda.synchronize()
    s = host(s_acc)
    # key H (the first chunk key) has q == k elementwise: S = D * 127^2
    assert np.all(s[:, :, H] == D * 127 * 127)
    Kt = sign[:, 0, :].astype(np.float64) * 127
    ref = (q_i8.cpu().numpy()[:, 0, :].astype(np.float64) @ Kt.T)
    j = np.arange(C)[:, None]
    ref = np.where(np.arange(H + C)[None, :] <= H + j, ref, 0)
    assert np.array_equal(s[:, 0, :].astype(np.float64), ref)
