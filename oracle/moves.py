"""Ordered row moves (cell compaction) and the grow-on-demand re-layout.

TEST INFRASTRUCTURE: see the package docstring for who may import this.

* "KV Cache Design — cells, format, sessions", section 2: a compaction
  changes only cells, so rows move verbatim; overlapping runs are copied
  one row at a time, ascending when the run slides down and descending
  when it slides up; callers order the moves with order_moves — upward
  moves top-down, downward bottom-up, upward first — because a destination
  may never land on a row that has not been copied yet.
* "KV cache" (sipllm), section "Design": the cache stores
  [layer][pos][kv_dim] with the live capacity as the per-layer stride;
  grow_to doubles the capacity (capped at max_ctx) and copies each layer's
  old rows verbatim to the new stride.

Readings: "top-down" sorts upward moves by source
descending, "bottom-up" sorts downward moves by source ascending, and
moves with dst == src are dropped. A move list is hazardous when some
move writes a row that a later move still has to read; such a list has no
meaning as a compaction and is rejected.
"""
from __future__ import annotations

import numpy as np


def order_moves(moves):
    """Upward moves (dst > src) by src descending, then downward moves
    (dst < src) by src ascending; zero-length and dst == src moves dropped."""
    ms = [tuple(int(v) for v in m) for m in moves if m[2] > 0 and m[0] != m[1]]
    up = sorted((m for m in ms if m[1] > m[0]), key=lambda m: -m[0])
    down = sorted((m for m in ms if m[1] < m[0]), key=lambda m: m[0])
    return up + down


def find_hazard(moves):
    """Index of the first move that writes a row some later move still
    reads (its original content would be lost), or None if there is none."""
    ms = [tuple(int(v) for v in m) for m in moves]
    for i, (s, d, n) in enumerate(ms):
        w0, w1 = d, d + n
        for (s2, _d2, n2) in ms[i + 1:]:
            if s2 < w1 and w0 < s2 + n2:
                return i
    return None


def move_rows(arena: np.ndarray, src: int, dst: int, n: int) -> None:
    """One move, one row at a time in slide order (descending when the run
    slides up, ascending when it slides down), so an overlapping run never
    reads a row it has already overwritten."""
    rows = range(n - 1, -1, -1) if dst > src else range(n)
    for r in rows:
        arena[dst + r] = arena[src + r]


def copy_cells(pools, moves) -> None:
    """Apply `moves` (already ordered) to every pool, in list order."""
    for pool in pools:
        for (s, d, n) in moves:
            move_rows(pool, int(s), int(d), int(n))


def grow_capacity(cap: int, need: int, max_ctx: int) -> int:
    """New capacity for a write at position need-1: double until it holds
    `need` positions, never above max_ctx."""
    nc = cap
    while nc < need:
        nc <<= 1
    return min(nc, max_ctx)


def initial_capacity(max_ctx: int, initial: int = 64) -> int:
    return min(initial, max_ctx)


def kv_relayout(src: np.ndarray, n_layers: int, old_cap: int, new_cap: int) -> np.ndarray:
    """Re-lay out a [layer][pos][row] store from stride old_cap to new_cap.

    src: array [n_layers*old_cap][...]. Returns [n_layers*new_cap][...] with
    layer l's rows [0, old_cap) copied verbatim; rows [old_cap, new_cap) of
    each layer are zero (never read before being written)."""
    dst = np.zeros((n_layers * new_cap,) + src.shape[1:], dtype=src.dtype)
    for l in range(n_layers):
        dst[l * new_cap: l * new_cap + old_cap] = src[l * old_cap: (l + 1) * old_cap]
    return dst
