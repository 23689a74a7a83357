"""Seeded synthetic inputs for the paged GQA decode path.

This module only builds inputs: block tables drawn from a shuffled physical
block pool (with reference counts for shared prefixes), context lengths,
attention windows, hole patterns, cold-tier selections and N(0,1) values.
It performs none of the method's arithmetic (no attention, no format
conversion, no quantisation, no row moves), so both the CPU oracle and the
CUDA path can consume the same inputs without sharing any computation.

Block model: "Tiered KV cache — architecture", section "The paged-attention
block model" (fixed-size physical blocks, a per-sequence logical-to-physical
table, reference-counted sharing, kInvalidBlockId holes).
Cell model: "KV Cache Design — cells, format, sessions", section 1
("Positions and cells": a position is a token index within its sequence, a
cell is the row that is written) and section 2 (copy-on-write of a shared
prefix before the first store lands in it).
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

INVALID_BLOCK_ID = -1

FORMATS = ("f32", "f16", "q8_0")


class BlockPool:
    """Physical block allocator with reference counts.

    Free ids are handed out in the order of a seeded random permutation, so
    a sequence's logical blocks land on scattered physical blocks.
    """

    def __init__(self, n_blocks: int, rng: np.random.Generator):
        self.n_blocks = int(n_blocks)
        self._free = list(rng.permutation(self.n_blocks)[::-1])
        self.refcount = np.zeros(self.n_blocks, dtype=np.int64)

    def alloc(self) -> int:
        if not self._free:
            raise RuntimeError("block pool exhausted")
        b = int(self._free.pop())
        self.refcount[b] = 1
        return b

    def incref(self, b: int) -> None:
        assert self.refcount[b] > 0
        self.refcount[b] += 1

    def decref(self, b: int) -> None:
        assert self.refcount[b] > 0
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self._free.append(int(b))

    @property
    def n_free(self) -> int:
        return len(self._free)


@dataclass
class Move:
    """A run of `len` rows to move from cell `src` to cell `dst`."""
    src: int
    dst: int
    len: int

    def as_tuple(self):
        return (self.src, self.dst, self.len)


class PagedSequences:
    """Host-side block tables for a batch of sequences over one BlockPool.

    `append(s, n)` grows sequence s by n positions, allocating blocks as
    needed. Appending into a block whose reference count is above one first
    copies that block into a fresh one (copy-on-write) and records the row
    move that does it; the caller applies the recorded moves with a mover
    before storing rows.
    """

    def __init__(self, pool: BlockPool, n_seqs: int, block_size: int):
        self.pool = pool
        self.bs = int(block_size)
        self.tables: list[list[int]] = [[] for _ in range(n_seqs)]
        self.lens = [0] * n_seqs
        self.cow_moves: list[Move] = []

    def append(self, s: int, n: int) -> None:
        for _ in range(n):
            pos = self.lens[s]
            lb = pos // self.bs
            if lb == len(self.tables[s]):
                self.tables[s].append(self.pool.alloc())
            else:
                b = self.tables[s][lb]
                if self.pool.refcount[b] > 1:
                    nb = self.pool.alloc()
                    self.cow_moves.append(Move(b * self.bs, nb * self.bs, self.bs))
                    self.pool.decref(b)
                    self.tables[s][lb] = nb
            self.lens[s] = pos + 1

    def fork(self, parent: int, child: int) -> None:
        """Child shares every block of parent (reference counts go up)."""
        assert not self.tables[child]
        for b in self.tables[parent]:
            self.pool.incref(b)
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]

    def cell_of(self, s: int, pos: int) -> int:
        b = self.tables[s][pos // self.bs]
        assert b != INVALID_BLOCK_ID
        return b * self.bs + pos % self.bs

    def table_array(self, max_blocks: int | None = None) -> np.ndarray:
        mb = max(1, max(len(t) for t in self.tables)) if max_blocks is None else max_blocks
        out = np.full((len(self.tables), mb), INVALID_BLOCK_ID, dtype=np.int32)
        for s, t in enumerate(self.tables):
            out[s, : len(t)] = t
        return out


@dataclass
class DecodeWorkload:
    """One layer of a paged decode step, plus the structure shared by all layers.

    Arrays are host numpy arrays. `k_hist`/`v_hist` hold the float32 values
    of every cell of the pool before the step (what earlier stores wrote);
    `k_new`/`v_new` are the decode token's freshly projected rows, to be
    stored at cell `new_cells[s]` (position context_lens[s]-1) before
    attention. `spans` is None (whole context) or int32 [n_seqs][2] [lo, hi).
    """
    name: str
    fmt: str
    n_seqs: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    n_phys_blocks: int
    block_table: np.ndarray
    context_lens: np.ndarray
    spans: np.ndarray | None
    q: np.ndarray
    k_hist: np.ndarray
    v_hist: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    new_cells: np.ndarray
    scale: float
    n_layers: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def n_cells(self) -> int:
        return self.n_phys_blocks * self.block_size

    @property
    def row_elems(self) -> int:
        return self.n_kv_heads * self.head_dim


def _values(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def _finish(name, fmt, seqs: PagedSequences, n_heads, n_kv_heads, head_dim, rng,
            spans=None, n_layers=1, max_blocks=None, extra=None, hist=True) -> DecodeWorkload:
    pool = seqs.pool
    bs = seqs.bs
    n = len(seqs.tables)
    table = seqs.table_array(max_blocks)
    lens = np.asarray(seqs.lens, dtype=np.int32)
    row = n_kv_heads * head_dim
    n_cells = pool.n_blocks * bs
    q = _values(rng, (n, n_heads, head_dim))
    k_hist = _values(rng, (n_cells, row)) if hist else None
    v_hist = _values(rng, (n_cells, row)) if hist else None
    k_new = _values(rng, (n, row))
    v_new = _values(rng, (n, row))
    new_cells = np.array([seqs.cell_of(s, int(lens[s]) - 1) if lens[s] > 0 else -1
                          for s in range(n)], dtype=np.int64)
    return DecodeWorkload(name=name, fmt=fmt, n_seqs=n, n_heads=n_heads,
                          n_kv_heads=n_kv_heads, head_dim=head_dim, block_size=bs,
                          n_phys_blocks=pool.n_blocks, block_table=table,
                          context_lens=lens, spans=spans, q=q, k_hist=k_hist,
                          v_hist=v_hist, k_new=k_new, v_new=v_new, new_cells=new_cells,
                          scale=1.0 / math.sqrt(head_dim), n_layers=n_layers,
                          extra=extra or {})


def tiny_f32(seed: int = 1001) -> DecodeWorkload:
    """Tiny paged decode, f32 KV: 2 sequences (ctx 37 and 100), 4/2 heads,
    d=64, bs=16, a pool of 32 blocks; sequence 1 has logical block 2 as a hole."""
    rng = np.random.default_rng(seed)
    pool = BlockPool(32, rng)
    seqs = PagedSequences(pool, 2, 16)
    seqs.append(0, 37)
    seqs.append(1, 100)
    w = _finish("tiny_f32", "f32", seqs, 4, 2, 64, rng)
    w.block_table[1, 2] = INVALID_BLOCK_ID
    return w


def llama3_f16(seed: int = 1003, n_seqs: int = 64, ctx_lo: int = 512, ctx_hi: int = 16384,
               fmt: str = "f16", block_size: int = 16, n_heads: int = 32,
               n_kv_heads: int = 8, head_dim: int = 128, pool_factor: float = 1.1,
               hist: bool = True, n_layers: int = 32) -> DecodeWorkload:
    """Llama-3-8B-shaped decode: 32/8 heads, d=128, bs=16, context lengths
    log-uniform in [ctx_lo, ctx_hi], tables drawn from a pool of
    pool_factor x the blocks needed."""
    rng = np.random.default_rng(seed)
    lens = np.round(np.exp(rng.uniform(math.log(ctx_lo), math.log(ctx_hi), n_seqs))).astype(np.int64)
    need = int(sum(-(-int(c) // block_size) for c in lens))
    pool = BlockPool(int(math.ceil(need * pool_factor)), rng)
    seqs = PagedSequences(pool, n_seqs, block_size)
    for s, c in enumerate(lens):
        seqs.append(s, int(c))
    return _finish("llama3_f16", fmt, seqs, n_heads, n_kv_heads, head_dim, rng,
                   n_layers=n_layers, hist=hist)


def smollm2_f32(seed: int = 1002, n_seqs: int = 8, ctx_lo: int = 2048, ctx_hi: int = 8192,
                hist: bool = True) -> DecodeWorkload:
    """SmolLM2-135M-shaped decode, f32 KV: 30 layers, 9/3 heads, d=64, bs=16,
    context lengths uniform in [ctx_lo, ctx_hi], pool = exactly the blocks
    needed, randomly permuted."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(ctx_lo, ctx_hi + 1, n_seqs)
    need = int(sum(-(-int(c) // 16) for c in lens))
    pool = BlockPool(need, rng)
    seqs = PagedSequences(pool, n_seqs, 16)
    for s, c in enumerate(lens):
        seqs.append(s, int(c))
    return _finish("smollm2_f32", "f32", seqs, 9, 3, 64, rng, n_layers=30, hist=hist)


def llama3_q8_prefix(seed: int = 1004, n_seqs: int = 32, prefix: int = 4096,
                     suffix_lo: int = 64, suffix_hi: int = 1024, block_size: int = 32,
                     windows: bool = True, hist: bool = True) -> DecodeWorkload:
    """Llama-3-8B-shaped q8_0 decode with a shared prefix and windows.

    Sequence 0 is prefilled with `prefix` positions and forked to all other
    sequences (the prefix blocks are then shared with reference count
    n_seqs); each sequence then appends a private suffix of U[suffix_lo,
    suffix_hi] positions. Appending into a shared, partly filled block copies
    it first (recorded in extra['cow_moves']). Each query gets a window
    [lo, hi) from two distinct uniform draws in [0, ctx].
    """
    rng = np.random.default_rng(seed)
    suffix = rng.integers(suffix_lo, suffix_hi + 1, n_seqs)
    n_prefix_blocks = -(-prefix // block_size)
    need = n_prefix_blocks + int(sum(-(-(prefix + int(x)) // block_size) - prefix // block_size
                                     for x in suffix))
    pool = BlockPool(need + 8, rng)
    seqs = PagedSequences(pool, n_seqs, block_size)
    seqs.append(0, prefix)
    for s in range(1, n_seqs):
        seqs.fork(0, s)
    for s in range(n_seqs):
        seqs.append(s, int(suffix[s]))
    spans = None
    if windows:
        spans = np.zeros((n_seqs, 2), dtype=np.int32)
        for s in range(n_seqs):
            ctx = seqs.lens[s]
            a, b = rng.choice(ctx + 1, size=2, replace=False)
            spans[s] = (min(a, b), max(a, b))
    extra = {"cow_moves": [m.as_tuple() for m in seqs.cow_moves],
             "refcount": pool.refcount.copy(), "prefix": prefix}
    return _finish("llama3_q8_prefix", "q8_0", seqs, 32, 8, 128, rng, spans=spans,
                   n_layers=32, extra=extra, hist=hist)


def longctx_f16_int4(seed: int = 1005, n_seqs: int = 16, ctx: int = 32768,
                     hole_frac: float = 0.05, cold_frac: float = 0.25,
                     pool_factor: float = 1.3, hist: bool = True) -> DecodeWorkload:
    """Long-context tiered decode, f16 KV: 16/4 heads, d=256, bs=16.

    A fraction `hole_frac` of logical blocks become holes (never the last
    block of a sequence). Of the remaining blocks other than the last (which
    takes the decode token's row), `cold_frac` are chosen for
    the cold round trip: extra['cold_src'] lists their current physical ids
    and extra['cold_dst'] the fresh ids (from the pool's spare blocks) that
    the dequantised data lands in; extra['cold_where'] holds the (seq,
    logical block) pairs whose table entries are retargeted.
    """
    rng = np.random.default_rng(seed)
    bs = 16
    nb = -(-ctx // bs)
    need = n_seqs * nb
    pool = BlockPool(int(math.ceil(need * pool_factor)), rng)
    seqs = PagedSequences(pool, n_seqs, bs)
    for s in range(n_seqs):
        seqs.append(s, ctx)
    table = seqs.table_array()
    holes = rng.random((n_seqs, nb)) < hole_frac
    holes[:, -1] = False
    for s in range(n_seqs):
        for lb in np.nonzero(holes[s])[0]:
            pool.decref(int(table[s, lb]))
            seqs.tables[s][lb] = INVALID_BLOCK_ID
    # the last block holds the position being written: it stays hot
    live = [(s, lb) for s in range(n_seqs) for lb in range(nb - 1) if not holes[s, lb]]
    pick = rng.random(len(live)) < cold_frac
    cold_where = [live[i] for i in np.nonzero(pick)[0]]
    cold_src = [seqs.tables[s][lb] for (s, lb) in cold_where]
    cold_dst = [pool.alloc() for _ in cold_where]
    extra = {"cold_where": cold_where, "cold_src": np.array(cold_src, dtype=np.int32),
             "cold_dst": np.array(cold_dst, dtype=np.int32)}
    w = _finish("longctx_f16_int4", "f16", seqs, 16, 4, 256, rng, extra=extra, hist=hist)
    return w


def retarget_cold(w: DecodeWorkload) -> np.ndarray:
    """Block table after the cold round trip: each cold (seq, logical block)
    entry points at its fresh physical id."""
    t = w.block_table.copy()
    for (s, lb), d in zip(w.extra["cold_where"], w.extra["cold_dst"]):
        t[s, lb] = d
    return t


def compaction_moves(seed: int = 1002, n_runs: int = 1000, len_lo: int = 8, len_hi: int = 64,
                     min_gap: int = 16, max_shift: int = 7):
    """Overlapping run moves for a compaction: each run of U[len_lo, len_hi]
    rows slides by a shift in [-max_shift, max_shift] minus 0 (so every move
    overlaps its own source); runs are separated by at least `min_gap` rows
    so their footprints stay disjoint. Returns (moves, n_cells) with moves in
    generation (ascending-address) order, roughly half up and half down."""
    rng = np.random.default_rng(seed)
    moves = []
    cursor = max_shift
    for _ in range(n_runs):
        cursor += min_gap + int(rng.integers(0, 8))
        ln = int(rng.integers(len_lo, len_hi + 1))
        d = 0
        while d == 0:
            d = int(rng.integers(-max_shift, max_shift + 1))
        moves.append((cursor, cursor + d, ln))
        cursor += ln
    n_cells = cursor + max_shift + min_gap
    return moves, n_cells
