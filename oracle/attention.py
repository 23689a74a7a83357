"""Paged grouped-query decode attention and the KV store, in float64.

TEST INFRASTRUCTURE: see the package docstring for who may import this.

What is computed (one decode query per sequence):
  * Block model — "Tiered KV cache — architecture", section "The
    paged-attention block model": position p of sequence s lives in
    physical block table[s][p // bs], slot p % bs, i.e. cell
    table[s][p//bs]*bs + p%bs of the layer's K and V pools.
  * Holes — same page, sections "The paged-attention block model" (item 3)
    and "Kernel dispatch": a table entry equal to kInvalidBlockId (-1)
    gives its positions a logit of -infinity, hence zero softmax weight.
  * Window — "KV Cache Design — cells, format, sessions", section 1: each
    query carries an allowed window [lo, hi); read here as logical
    positions of the sequence intersected with [0, ctx).
  * Grouped-query map: query head h reads KV head h // G, G = Hq / Hkv
    (contiguous groups; the pages do not state the map).

For each (s, h) the valid positions are gathered into dense K, V arrays
(decoded exactly as stored) and plain softmax attention is applied:
  t_p = scale * q . k_p,  w = exp(t - max t) / sum,  o = sum_p w_p v_p,
  lse = max t + log(sum exp(t - max t)).
With no valid position the output is 0 and lse is -infinity.
"""
from __future__ import annotations

import math

import numpy as np

from . import formats

INVALID_BLOCK_ID = -1


def kv_store(fmt: str, k_pool: np.ndarray, v_pool: np.ndarray, k_new, v_new, cells,
             n_kv_heads: int, head_dim: int) -> None:
    """Write freshly projected rows into resolved cells, converting to `fmt`.

    "KV Cache Design — cells, format, sessions", sections 1 and 3: the
    store writes the row to the cell the allocator resolved (not to the
    position) and quantises with the one store quantiser. Pools are uint8
    [n_cells][row_bytes]; a negative cell means "no row to store".
    """
    enc_k = formats.encode_rows(fmt, np.asarray(k_new, dtype=np.float32), n_kv_heads, head_dim)
    enc_v = formats.encode_rows(fmt, np.asarray(v_new, dtype=np.float32), n_kv_heads, head_dim)
    for r, c in enumerate(np.asarray(cells).tolist()):
        if c < 0:
            continue
        k_pool[c] = enc_k[r]
        v_pool[c] = enc_v[r]


def valid_positions(block_table, context_len: int, span, block_size: int):
    """Positions of one sequence that attention reads, with their cells."""
    lo, hi = 0, int(context_len)
    if span is not None:
        lo = max(int(span[0]), 0)
        hi = min(int(span[1]), int(context_len))
    pos, cells = [], []
    for p in range(lo, hi):
        b = int(block_table[p // block_size])
        if b == INVALID_BLOCK_ID:
            continue
        pos.append(p)
        cells.append(b * block_size + p % block_size)
    return np.array(pos, dtype=np.int64), np.array(cells, dtype=np.int64)


def attend_dense(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Textbook softmax attention of one query over dense rows, float64.

    q [d], k [n][d], v [n][d]. Returns (o [d], lse)."""
    d = q.shape[0]
    if k.shape[0] == 0:
        return np.zeros(d, dtype=np.float64), -math.inf
    t = scale * (k.astype(np.float64) @ q.astype(np.float64))
    m = np.max(t)
    e = np.exp(t - m)
    z = np.sum(e)
    o = (e / z) @ v.astype(np.float64)
    return o, float(m + math.log(z))


def gather_sequence(fmt, k_pool, v_pool, block_table_row, context_len, span,
                    n_kv_heads, head_dim, block_size):
    """Dense float64 K, V [n_valid][Hkv][d] of one sequence's valid positions."""
    _, cells = valid_positions(block_table_row, context_len, span, block_size)
    k = formats.decode_rows(fmt, k_pool[cells], n_kv_heads, head_dim)
    v = formats.decode_rows(fmt, v_pool[cells], n_kv_heads, head_dim)
    return (k.reshape(len(cells), n_kv_heads, head_dim),
            v.reshape(len(cells), n_kv_heads, head_dim))


def paged_attn_decode(fmt, q, k_pool, v_pool, block_table, context_lens, spans,
                      n_heads, n_kv_heads, head_dim, block_size, scale,
                      seqs=None, heads=None):
    """Decode attention for every (or the listed) sequence and query head.

    q float32/float64 [B][Hq][d]; pools uint8 [n_cells][row_bytes];
    block_table int32 [B][max_blocks]; context_lens int32 [B]; spans None or
    int32 [B][2]. Returns (out float64 [B][Hq][d], lse float64 [B][Hq]);
    entries outside `seqs` x `heads` are NaN.
    """
    B = q.shape[0]
    G = n_heads // n_kv_heads
    assert G * n_kv_heads == n_heads
    out = np.full((B, n_heads, head_dim), np.nan)
    lse = np.full((B, n_heads), np.nan)
    for s in (range(B) if seqs is None else seqs):
        span = None if spans is None else spans[s]
        k, v = gather_sequence(fmt, k_pool, v_pool, block_table[s], context_lens[s], span,
                               n_kv_heads, head_dim, block_size)
        for h in (range(n_heads) if heads is None else heads):
            g = h // G
            out[s, h], lse[s, h] = attend_dense(np.asarray(q[s, h], dtype=np.float64),
                                                k[:, g, :], v[:, g, :], scale)
    return out, lse
