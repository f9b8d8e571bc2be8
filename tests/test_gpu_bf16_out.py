"""BF16 attention outputs.

"gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §3.3: the decode merges
its partitions and writes BF16.  Every attention entry point takes an output
type; with bf16 the kernels round the same fp32 results to nearest even.  So
the bf16 output must equal RNE(fp32 output) bit for bit, on the same inputs,
for the decode (single-CTA pairs and pairs merged across CTAs, empty
sequences), the decode step, the UINT8-probability decode, the BF16-KV
comparison decode and both prefix paths (whole and split row blocks)."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from tests.gpu_helpers import dev, host, gpu_decode_cache, gpu_quantize_rows, gpu_bf16_cache

pytestmark = pytest.mark.gpu


def _rne_bits(x: np.ndarray) -> np.ndarray:
    return wl.bf16_bits(np.ascontiguousarray(x, np.float32))


def _same(out32: torch.Tensor, out16: torch.Tensor, what: str):
    a = host(out32)
    b = host(out16)
    assert np.isfinite(a).all(), what
    assert np.array_equal(b, _rne_bits(a)), f"{what}: {int((b != _rne_bits(a)).sum())} elements differ"


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([5000, 1, 0, 300], 24, 4, 256), ([32768, 777], 32, 8, 128)])
def test_decode_bf16_out(lens, Hq, Hkv, D):
    w = wl.DecodeWorkload("bo", Hq, Hkv, D, lens, seed=21)
    cache = gpu_decode_cache(w)
    q_i8, q_s = gpu_quantize_rows(w.q(), Hkv, cache)
    ws = i8.decode_workspace(w.B, Hq, Hkv, D, w.block_tables.shape[1])
    bt, sl = dev(w.block_tables), dev(w.seq_lens)
    for u8 in (False, True):
        o32 = torch.full((w.B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        o16 = torch.full((w.B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        for o in (o32, o16):
            i8.int8_paged_decode_attn(o, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                      cache["v_scale"], bt, sl, ws, u8_probs=u8)
        torch.cuda.synchronize()
        assert i8.device_error() == 0
        _same(o32, o16, f"decode u8={u8}")
        for b in np.flatnonzero(w.seq_lens == 0):
            assert not host(o16)[b].any()  # an empty sequence's rows are zeros


def test_decode_step_bf16_out():
    w = wl.DecodeWorkload("bs", 24, 4, 256, [3000, 17], seed=22)
    k_new = np.zeros((w.B, w.Hkv, w.D), np.uint16)
    v_new = np.zeros_like(k_new)
    caches = []
    for _ in range(2):
        c = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
        for b in range(w.B):
            L = int(w.seq_lens[b])
            k, v = w.kv(b)
            i8.kv_quant_write(dev(k[:L - 1]), dev(v[:L - 1]), dev(w.slots(b, 0, L - 1)), **c)
            k_new[b], v_new[b] = k[L - 1], v[L - 1]
        caches.append(c)
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
    bt, sl = dev(w.block_tables), dev(w.seq_lens)
    o32 = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    o16 = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    for o, c in zip((o32, o16), caches):
        i8.int8_decode_step(o, dev(w.q()), dev(k_new), dev(v_new), c["k_cache"], c["v_cache"], c["k_scale"],
                            c["v_scale"], bt, sl, ws)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    _same(o32, o16, "decode step")
    for n in caches[0]:
        assert torch.equal(caches[0][n], caches[1][n]), n


def test_bf16_kv_decode_bf16_out():
    w = wl.DecodeWorkload("bk", 24, 4, 256, [4000, 129], seed=23)
    cache = gpu_bf16_cache(w)
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
    bt, sl, q = dev(w.block_tables), dev(w.seq_lens), dev(w.q())
    o32 = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    o16 = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    for o in (o32, o16):
        i8.bf16_paged_decode_attn(o, q, cache["k_cache"], cache["v_cache"], bt, sl, ws)
    torch.cuda.synchronize()
    _same(o32, o16, "bf16-kv decode")


@pytest.mark.parametrize("H,C,Hq,Hkv,D", [(300, 70, 24, 4, 256), (100, 700, 32, 8, 128)])
def test_prefix_bf16_out(H, C, Hq, Hkv, D):
    # the second case has more row blocks than SMs: its last wave is split and merged
    w = wl.PrefixWorkload("bp", Hq, Hkv, D, H, C, seed=24)
    k, v = w.kv()
    cache = i8.alloc_int8_cache(w.num_blocks, Hkv, D)
    i8.kv_quant_write(dev(k), dev(v), dev(w.slots()), **cache)
    q_i8, q_s = gpu_quantize_rows(w.q(), Hkv, cache)
    bt = dev(w.block_table)
    o32 = torch.empty((C, Hq, D), dtype=torch.float32, device="cuda")
    o16 = torch.empty((C, Hq, D), dtype=torch.bfloat16, device="cuda")
    for o in (o32, o16):
        i8.int8_prefix_attn(o, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"], cache["v_scale"],
                            bt, H)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    _same(o32, o16, "int8 prefix")
    # the high-precision path over the same history and the chunk's bf16 K/V
    for o in (o32, o16):
        i8.bf16_prefix_attn(o, dev(w.q()), dev(k[H:]), dev(v[H:]), H, cache["k_cache"], cache["v_cache"],
                            cache["k_scale"], cache["v_scale"], bt)
    torch.cuda.synchronize()
    _same(o32, o16, "bf16 prefix")
