"""Seeded synthetic inputs for INT8 KV-cache paged attention.

This module draws inputs and lays out paging (block tables, slot mappings).
It holds none of the attention or quantization arithmetic, so both the CPU
oracle and the CUDA library can consume what it produces.

All tensors are numpy arrays; bf16 values are carried as uint16 bit patterns
(fp32 N(0,1) draws rounded to bf16 with round-to-nearest-even).  Every draw
comes from ``numpy.random.default_rng`` with an explicit seed (PCG64), so a
sequence's K/V can be regenerated on its own from ``(seed, sequence index)``.

Workloads (shaped like the pages' full-attention layer: 24 query heads, 4 KV
heads, head_dim 256, block size 16):

* ``decode_4k``      one sequence, history 4096, N(0,1).
* ``decode_outlier`` one sequence at history 8192 / 16384 / 32768; K has 4
  outlier channels per KV head scaled x20 (the stable channel outliers the
  part-1 page mentions when discussing KIVI), V is N(0,1).
* ``prefix_chunk``   2048 new query tokens after 16384 cached history tokens.
* ``decode_batch``   64 sequences, lengths uniform in [1024, 32768].
* ``producer_gqa``   8192 new tokens, 8 KV heads, head_dim 128, N(0,1) with 2%
  of elements x10; then batch-16 decode at 32768 with 32 / 8 heads.
* ``producer_rope_tokens``  the same tokens with their positions, a RoPE
  cos/sin table and per-head Q/K RMSNorm weights (model constants, drawn or
  tabulated here like any other input).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


# --------------------------------------------------------------------------- paging
def paged_tables(seq_lens, block_size: int = BLOCK_SIZE, perm_seed: int = 1, extra_blocks: int = 0):
    """One shared physical pool of sum(ceil(L_b / bs)) (+extra) blocks, permuted
    with ``perm_seed`` and handed out to the sequences in order.

    Returns (block_tables int32 [B, max_blocks] padded with -1, num_blocks)."""
    seq_lens = np.asarray(seq_lens, np.int64)
    nblk = (seq_lens + block_size - 1) // block_size
    num_blocks = int(nblk.sum()) + extra_blocks
    perm = np.random.default_rng(perm_seed).permutation(num_blocks).astype(np.int32)
    max_blocks = max(int(nblk.max()) if nblk.size else 1, 1)
    tables = np.full((len(seq_lens), max_blocks), -1, np.int32)
    pos = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[pos:pos + n]
        pos += n
    return tables, num_blocks


def slot_mapping(block_table_row: np.ndarray, positions, block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Slots of token positions of one sequence: block_table[p // bs] * bs + p % bs."""
    p = np.asarray(positions, np.int64)
    return (block_table_row[p // block_size].astype(np.int64) * block_size + p % block_size).astype(np.int32)


# --------------------------------------------------------------------------- workloads
@dataclass
class DecodeWorkload:
    """Decode batch: per-sequence K/V histories in a paged pool plus one query per sequence."""
    name: str
    Hq: int
    Hkv: int
    D: int
    seq_lens: np.ndarray
    seed: int = 0
    perm_seed: int = 1
    outlier_channels: int = 0       # per KV head, on K only
    outlier_scale: float = 20.0
    sparse_outlier_frac: float = 0.0  # i.i.d. elements of K and V scaled by sparse_outlier_scale
    sparse_outlier_scale: float = 10.0
    block_size: int = BLOCK_SIZE
    block_tables: np.ndarray = field(init=False)
    num_blocks: int = field(init=False)

    def __post_init__(self):
        self.seq_lens = np.asarray(self.seq_lens, np.int32)
        self.block_tables, self.num_blocks = paged_tables(self.seq_lens, self.block_size, self.perm_seed)

    @property
    def B(self) -> int:
        return int(self.seq_lens.size)

    def outlier_dims(self) -> np.ndarray:
        """[Hkv, outlier_channels] head-dims of K scaled by outlier_scale (seed 2)."""
        rng = np.random.default_rng(2)
        return np.stack([rng.permutation(self.D)[: self.outlier_channels] for _ in range(self.Hkv)]) \
            if self.outlier_channels else np.zeros((self.Hkv, 0), np.int64)

    def kv(self, b: int, start: int = 0, stop: int | None = None):
        """bf16 K, V [L_b, Hkv, D] of sequence b (rows start:stop), regenerated from (seed, b)."""
        L = int(self.seq_lens[b])
        rng = np.random.default_rng([self.seed, 1000 + b])
        k = rng.standard_normal((L, self.Hkv, self.D), dtype=np.float32)
        v = rng.standard_normal((L, self.Hkv, self.D), dtype=np.float32)
        if self.outlier_channels:
            dims = self.outlier_dims()
            for h in range(self.Hkv):
                k[:, h, dims[h]] *= np.float32(self.outlier_scale)
        if self.sparse_outlier_frac > 0:
            orng = np.random.default_rng([4, b])
            k[orng.random(k.shape) < self.sparse_outlier_frac] *= np.float32(self.sparse_outlier_scale)
            v[orng.random(v.shape) < self.sparse_outlier_frac] *= np.float32(self.sparse_outlier_scale)
        sl = slice(start, stop)
        return bf16_bits(k[sl]), bf16_bits(v[sl])

    def q(self) -> np.ndarray:
        """bf16 queries [B, Hq, D] (one decode token per sequence)."""
        return randn_bf16(np.random.default_rng([self.seed, 7]), (self.B, self.Hq, self.D))

    def slots(self, b: int, start: int = 0, stop: int | None = None) -> np.ndarray:
        L = int(self.seq_lens[b])
        stop = L if stop is None else stop
        return slot_mapping(self.block_tables[b], np.arange(start, stop), self.block_size)

    def kv_bytes_int8(self) -> int:
        """Algorithmic INT8 cache bytes one decode pass reads: Hkv*(2D + 8) per cached token."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * (2 * self.D + 8)

    def kv_bytes_bf16(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * 4 * self.D


@dataclass
class PrefixWorkload:
    """Prefix-prefill chunk: `history` cached tokens then `chunk` new tokens of one sequence."""
    name: str
    Hq: int
    Hkv: int
    D: int
    history: int
    chunk: int
    seed: int = 0
    perm_seed: int = 1
    block_size: int = BLOCK_SIZE
    block_table: np.ndarray = field(init=False)
    num_blocks: int = field(init=False)

    def __post_init__(self):
        tables, self.num_blocks = paged_tables([self.history + self.chunk], self.block_size, self.perm_seed)
        self.block_table = tables[0]

    @property
    def total(self) -> int:
        return self.history + self.chunk

    def kv(self):
        """bf16 K, V [history + chunk, Hkv, D]."""
        rng = np.random.default_rng([self.seed, 11])
        k = randn_bf16(rng, (self.total, self.Hkv, self.D))
        v = randn_bf16(rng, (self.total, self.Hkv, self.D))
        return k, v

    def q(self) -> np.ndarray:
        """bf16 chunk queries [chunk, Hq, D]."""
        return randn_bf16(np.random.default_rng([self.seed, 13]), (self.chunk, self.Hq, self.D))

    def slots(self, start: int = 0, stop: int | None = None) -> np.ndarray:
        stop = self.total if stop is None else stop
        return slot_mapping(self.block_table, np.arange(start, stop), self.block_size)

    def pairs(self) -> int:
        """(q-head, query, key) pairs the causal chunk attends over."""
        C, H = self.chunk, self.history
        return self.Hq * (C * H + C * (C + 1) // 2)

    def int8_ops(self) -> int:
        """QK and PV multiply-adds, 2 ops each: 4 * D per pair."""
        return self.pairs() * 4 * self.D


def decode_4k() -> DecodeWorkload:
    return DecodeWorkload("decode_4k", 24, 4, 256, [4096], seed=0)


def decode_outlier(L: int) -> DecodeWorkload:
    return DecodeWorkload(f"decode_outlier_{L}", 24, 4, 256, [L], seed=0, outlier_channels=4)


def prefix_chunk(history: int = 16384, chunk: int = 2048) -> PrefixWorkload:
    return PrefixWorkload(f"prefix_{history}+{chunk}", 24, 4, 256, history, chunk, seed=0)


def decode_batch(B: int = 64, lo: int = 1024, hi: int = 32768) -> DecodeWorkload:
    lens = np.random.default_rng(3).integers(lo, hi + 1, size=B)
    return DecodeWorkload("decode_batch64", 24, 4, 256, lens, seed=3)


def producer_gqa_decode(B: int = 16, L: int = 32768) -> DecodeWorkload:
    return DecodeWorkload("decode_gqa_b16", 32, 8, 128, [L] * B, seed=4, sparse_outlier_frac=0.02)


def producer_tokens(T: int = 8192, Hq: int = 32, Hkv: int = 8, D: int = 128, seed: int = 4):
    """Producer input: T new tokens (q, k, v bf16, 2% of elements x10) and their
    slots: consecutive positions of one sequence in a permuted block pool."""
    rng = np.random.default_rng([seed, 21])
    out = []
    for H in (Hq, Hkv, Hkv):
        x = rng.standard_normal((T, H, D), dtype=np.float32)
        x[rng.random(x.shape) < 0.02] *= np.float32(10.0)
        out.append(bf16_bits(x))
    q, k, v = out
    tables, num_blocks = paged_tables([T], BLOCK_SIZE, perm_seed=5)
    slots = slot_mapping(tables[0], np.arange(T))
    return dict(q=q, k=k, v=v, slots=slots, num_blocks=num_blocks, Hq=Hq, Hkv=Hkv, D=D)


def rope_cos_sin(max_position: int, rotary_dim: int, base: float = 10000.0) -> np.ndarray:
    """RoPE table float32 [max_position, rotary_dim]: row p holds cos(p f_i) for
    i < rotary_dim/2, then sin(p f_i), with f_i = base^(-2i / rotary_dim).  The
    angles and their cos/sin are taken in fp64 and rounded once to fp32; the
    table is a model constant handed to both the oracle and the kernels."""
    h = rotary_dim // 2
    f = base ** (-2.0 * np.arange(h, dtype=np.float64) / rotary_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * f[None, :]
    return np.ascontiguousarray(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


def norm_weight_bf16(rng: np.random.Generator, D: int) -> np.ndarray:
    """Per-head RMSNorm weight: 1 + 0.25 N(0,1), in bf16."""
    return bf16_bits(np.float32(1.0) + np.float32(0.25) * rng.standard_normal(D, dtype=np.float32))


def producer_rope_tokens(T: int = 8192, Hq: int = 32, Hkv: int = 8, D: int = 128, rotary_dim: int = 128,
                         max_position: int = 32768, seed: int = 4):
    """producer_tokens plus positions 0..T-1 (one sequence from its start), a
    RoPE table for max_position positions and Q / K RMSNorm weights."""
    p = producer_tokens(T, Hq, Hkv, D, seed)
    rng = np.random.default_rng([seed, 22])
    p.update(positions=np.arange(T, dtype=np.int32), cos_sin=rope_cos_sin(max_position, rotary_dim),
             rotary_dim=rotary_dim, q_norm_weight=norm_weight_bf16(rng, D), k_norm_weight=norm_weight_bf16(rng, D))
    return p
