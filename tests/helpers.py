"""Shared test helpers: oracle-side cache construction and golden-file parsing."""
from __future__ import annotations

import os

import numpy as np

import workloads as wl
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str):
    """Rows of a '|'-separated golden fixture, comment lines (#) skipped."""
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([part.split() for part in line.split("|")])
    return rows


def oracle_decode_cache(w: wl.DecodeWorkload, seqs=None):
    """Run the oracle producer over every token of the chosen sequences of a
    decode workload (all of them by default); returns the cache dict."""
    cache = None
    seqs = range(w.B) if seqs is None else seqs
    for b in seqs:
        k, v = w.kv(b)
        cache = orc.kv_quant_write(k, v, w.slots(b), w.num_blocks, w.block_size, **({} if cache is None else cache))
    return cache


def quantize_rows(q: np.ndarray):
    """Oracle quantization of every (token, head) row of a bf16 [N, H, D] array."""
    q_i8 = np.empty(q.shape, np.int8)
    q_scale = np.empty(q.shape[:2], np.float32)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            q_i8[b, h], q_scale[b, h] = orc.quantize_vector(q[b, h])
    return q_i8, q_scale


def oracle_query(w: wl.DecodeWorkload, seqs=None):
    """Quantized decode queries (q_i8 [B,Hq,D], q_scale [B,Hq]) through the oracle quantizer."""
    q = w.q()
    if seqs is not None:
        q = q[list(seqs)]
    return quantize_rows(q)


def dequant_decode_dense(w: wl.DecodeWorkload, b: int):
    """Raw (unquantized) bf16 K/V of sequence b as float64 [L, Hkv, D]."""
    k, v = w.kv(b)
    return orc.bf16_to_f64(k), orc.bf16_to_f64(v)


def gather_int8(cache, block_table_row, L, Hkv, D, bs=wl.BLOCK_SIZE):
    """Token-major int8 K, V [L, Hkv, D] and scales [L, Hkv] read from the paged
    cache with numpy reshapes of the documented layouts (independent of the
    oracle's own index arithmetic)."""
    NB = cache["k_cache"].shape[0]
    K5 = cache["k_cache"].reshape(NB, Hkv, D // 16, bs, 16)
    V4 = cache["v_cache"].reshape(NB, Hkv, D, bs)
    pos = np.arange(L)
    blk = block_table_row[pos // bs]
    off = pos % bs
    # K5[blk, h, c, off, i] -> [L, Hkv, D/16, 16] -> [L, Hkv, D]
    Kt = K5[blk, :, :, off, :].reshape(L, Hkv, D)
    Vt = V4[blk, :, :, off]  # advanced indices first: [L, Hkv, D]
    sK = cache["k_scale"][blk, off, :]
    sV = cache["v_scale"][blk, off, :]
    return Kt, Vt, sK, sV
