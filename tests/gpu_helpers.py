"""GPU-side test helpers: upload seeded inputs and fill caches through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor (uint16 bf16 bit patterns become torch.bfloat16)."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def gpu_decode_cache(w: wl.DecodeWorkload, seqs=None):
    """INT8 cache of a decode workload written by the CUDA producer, one call per sequence."""
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    for b in (range(w.B) if seqs is None else seqs):
        k, v = w.kv(b)
        i8.kv_quant_write(dev(k), dev(v), dev(w.slots(b)), **cache)
    return cache


def gpu_bf16_cache(w: wl.DecodeWorkload):
    cache = i8.alloc_bf16_cache(w.num_blocks, w.Hkv, w.D)
    for b in range(w.B):
        k, v = w.kv(b)
        i8.bf16_kv_write(dev(k), dev(v), dev(w.slots(b)), **cache)
    return cache


def gpu_quantize_rows(q: np.ndarray, Hkv: int, cache):
    """Quantize query rows [N, Hq, D] through the producer's query path (K/V writes skipped)."""
    N, Hq, D = q.shape
    dummy = torch.zeros((N, Hkv, D), dtype=torch.bfloat16, device="cuda")
    q_i8 = torch.empty((N, Hq, D), dtype=torch.int8, device="cuda")
    q_scale = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
    i8.kv_quant_write(dummy, dummy, torch.full((N,), -1, dtype=torch.int32, device="cuda"), **cache,
                      q=dev(q), q_i8=q_i8, q_scale=q_scale)
    return q_i8, q_scale


def gpu_decode(w: wl.DecodeWorkload, cache, q_i8, q_scale, workspace=None, out=None, u8_probs=False):
    if out is None:
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    if workspace is None:
        workspace = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
    i8.int8_paged_decode_attn(out, q_i8, q_scale, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                              cache["v_scale"], dev(w.block_tables), dev(w.seq_lens), workspace, u8_probs=u8_probs)
    return out
