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


# ------------------------------------------------- window modes, multi-query
#
# "KV Cache Design — cells, format, sessions", section 1: a backend takes a
# query's allowed window in one of three modes — causal positions, one
# [lo, hi) pair per query, or up to KV_MAP_MAX_SPANS (start, len) runs (the
# set-valued kv_map: a shared prefix plus a private run). Read here, as for
# the pair, as logical positions of the sequence; the pages give no value for
# KV_MAP_MAX_SPANS (the library fixes 8). The same section's multi-token
# (prefill) kernels take several queries per sequence; "Tiered KV cache —
# architecture", section "Kernel dispatch", passes per-sequence context and
# query lengths. Query j of the n queries of a sequence of context length
# ctx sits at position ctx - n + j and reads only positions up to its own.

def query_positions(context_len: int, span=None, runs=None, last=None) -> np.ndarray:
    """Sorted logical positions one query may read, before holes: [0, ctx)
    intersected with [0, last] (causal, when `last` is given) and with its
    window — the [lo, hi) `span`, or the union of the (start, len) `runs`."""
    hi = int(context_len) if last is None else min(int(context_len), int(last) + 1)
    hi = max(hi, 0)
    ok = np.zeros(hi, dtype=bool)
    if runs is not None:
        for start, n in np.asarray(runs).reshape(-1, 2).tolist():
            a, b = max(int(start), 0), min(int(start) + int(n), hi)
            if b > a:
                ok[a:b] = True
    else:
        lo, h2 = 0, hi
        if span is not None:
            lo, h2 = max(int(span[0]), 0), min(int(span[1]), hi)
        if h2 > lo:
            ok[lo:h2] = True
    return np.nonzero(ok)[0]


def cells_of(block_table_row, positions, block_size: int):
    """(positions kept, their cells): positions in holes are dropped."""
    keep, cells = [], []
    for p in np.asarray(positions).tolist():
        b = int(block_table_row[p // block_size])
        if b == INVALID_BLOCK_ID:
            continue
        keep.append(p)
        cells.append(b * block_size + p % block_size)
    return np.array(keep, dtype=np.int64), np.array(cells, dtype=np.int64)


def attend_positions(fmt, q_heads, k_pool, v_pool, block_table_row, positions, n_kv_heads,
                     head_dim, block_size, scale, G):
    """Attention of one query token (all its heads, q_heads [Hq][d]) over the
    listed positions of one sequence. Returns (out [Hq][d], lse [Hq])."""
    _, cells = cells_of(block_table_row, positions, block_size)
    k = formats.decode_rows(fmt, k_pool[cells], n_kv_heads, head_dim).reshape(
        len(cells), n_kv_heads, head_dim)
    v = formats.decode_rows(fmt, v_pool[cells], n_kv_heads, head_dim).reshape(
        len(cells), n_kv_heads, head_dim)
    Hq = q_heads.shape[0]
    out = np.zeros((Hq, head_dim))
    lse = np.zeros(Hq)
    for h in range(Hq):
        g = h // G
        out[h], lse[h] = attend_dense(np.asarray(q_heads[h], dtype=np.float64), k[:, g, :],
                                      v[:, g, :], scale)
    return out, lse


def paged_attn_decode_map(fmt, q, k_pool, v_pool, block_table, context_lens, kv_map,
                          n_heads, n_kv_heads, head_dim, block_size, scale):
    """Decode attention with set-valued windows: kv_map int32 [B][R][2] of
    (start, len) runs per sequence's query (len <= 0: unused run)."""
    B = q.shape[0]
    G = n_heads // n_kv_heads
    out = np.zeros((B, n_heads, head_dim))
    lse = np.zeros((B, n_heads))
    for s in range(B):
        pos = query_positions(context_lens[s], runs=kv_map[s])
        out[s], lse[s] = attend_positions(fmt, q[s], k_pool, v_pool, block_table[s], pos,
                                          n_kv_heads, head_dim, block_size, scale, G)
    return out, lse


def paged_attn_prefill(fmt, q, k_pool, v_pool, block_table, context_lens, q_start, spans,
                       kv_map, n_heads, n_kv_heads, head_dim, block_size, scale):
    """Multi-query (prefill) attention through the paged cache, float64.

    q [n_tokens][Hq][d]: the queries of sequence s are rows q_start[s] ..
    q_start[s+1]-1; query j of the n = q_start[s+1] - q_start[s] queries
    sits at position ctx - n + j and reads positions <= its own, within its
    window: spans [n_tokens][2] ([lo, hi) per query) or kv_map
    [n_tokens][R][2] ((start, len) runs per query), or neither. Returns
    (out [n_tokens][Hq][d], lse [n_tokens][Hq])."""
    B = len(context_lens)
    G = n_heads // n_kv_heads
    n_tok = q.shape[0]
    out = np.zeros((n_tok, n_heads, head_dim))
    lse = np.zeros((n_tok, n_heads))
    for s in range(B):
        a, b = int(q_start[s]), int(q_start[s + 1])
        n, ctx = b - a, int(context_lens[s])
        for j in range(n):
            i = a + j
            pos = query_positions(ctx, span=None if spans is None else spans[i],
                                  runs=None if kv_map is None else kv_map[i],
                                  last=ctx - n + j)
            out[i], lse[i] = attend_positions(fmt, q[i], k_pool, v_pool, block_table[s], pos,
                                              n_kv_heads, head_dim, block_size, scale, G)
    return out, lse
