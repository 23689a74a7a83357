"""Pins of the oracle's ordered mover and grow-on-demand re-layout (CPU only).

* "KV Cache Design — cells, format, sessions", section 2: rows move
  verbatim; order_moves puts upward moves first (top-down) and downward
  moves after (bottom-up) so that no destination lands on a row that has
  not been copied yet.
* "KV cache" (sipllm), section "Design": the capacity doubles, capped at
  max_ctx, and a re-layout copies each layer's rows verbatim, so reads are
  bitwise identical to a store preallocated at max_ctx.
"""
import itertools

import numpy as np
import pytest

from oracle import moves as om
from paged_kv_cache_gqa_gb300 import workloads


def _staged(arena, moves):
    """Simultaneous semantics: read every source first, then write every
    destination (the meaning a compaction's move set has)."""
    out = arena.copy()
    data = [arena[s:s + n].copy() for (s, d, n) in moves]
    for (s, d, n), rows in zip(moves, data):
        out[d:d + n] = rows
    return out


def test_order_moves_hand_example():
    ms = [(2, 0, 3), (8, 5, 2), (12, 15, 3), (20, 22, 2), (30, 30, 4), (40, 41, 0)]
    assert om.order_moves(ms) == [(20, 22, 2), (12, 15, 3), (2, 0, 3), (8, 5, 2)]


def test_order_moves_fixes_a_compaction_that_list_order_breaks():
    # runs slide down to close gaps: in list order the second move overwrites
    # the first move's source before it is read
    ms = [(20, 10, 5), (10, 5, 5)]
    assert om.find_hazard(ms) == 0
    ordered = om.order_moves(ms)
    assert ordered == [(10, 5, 5), (20, 10, 5)]
    assert om.find_hazard(ordered) is None
    arena = np.arange(32)
    a = arena.copy()
    om.copy_cells([a], ordered)
    assert np.array_equal(a, _staged(arena, ordered))


def test_crossing_swap_has_no_safe_order():
    ms = [(0, 10, 5), (10, 0, 5)]
    for perm in itertools.permutations(ms):
        assert om.find_hazard(list(perm)) is not None


def test_single_overlapping_move_is_memmove():
    for s, d, n in [(3, 5, 10), (5, 3, 10), (0, 1, 20), (1, 0, 20), (4, 11, 6)]:
        a = np.arange(40) * 7 + 1
        b = a.copy()
        om.move_rows(b, s, d, n)
        want = a.copy()
        want[d:d + n] = a[s:s + n]
        assert np.array_equal(b, want)


def test_validator_brute_force_small_arenas():
    """For every order of small move sets with disjoint destinations on an
    arena of distinct rows: the validator accepts exactly the orders whose
    sequential result equals the simultaneous one."""
    rng = np.random.default_rng(11)
    checked = accepted = 0
    for _ in range(300):
        k = int(rng.integers(2, 5))
        ms, dsts = [], set()
        while len(ms) < k:
            n = int(rng.integers(1, 4))
            s = int(rng.integers(0, 14))
            d = int(rng.integers(0, 14))
            rows = set(range(d, d + n))
            if s == d or rows & dsts:
                continue
            dsts |= rows
            ms.append((s, d, n))
        arena = np.arange(20) * 3 + 100
        for perm in itertools.permutations(ms):
            perm = list(perm)
            a = arena.copy()
            om.copy_cells([a], perm)
            same = np.array_equal(a, _staged(arena, perm))
            ok = om.find_hazard(perm) is None
            assert ok == same, perm
            checked += 1
            accepted += ok
    assert checked > 1000 and 0 < accepted < checked


def test_order_moves_on_generated_compaction():
    ms, n_cells = workloads.compaction_moves(seed=3, n_runs=60)
    ordered = om.order_moves(ms)
    assert om.find_hazard(ordered) is None
    ups = [m for m in ordered if m[1] > m[0]]
    assert ordered[:len(ups)] == ups  # upward first
    arena = np.arange(n_cells * 2).reshape(n_cells, 2)
    a = arena.copy()
    om.copy_cells([a], ordered)
    assert np.array_equal(a, _staged(arena, ordered))


def test_grow_capacity_doubles_and_caps():
    assert om.initial_capacity(8192) == 64 and om.initial_capacity(40) == 40
    assert om.grow_capacity(64, 65, 8192) == 128
    assert om.grow_capacity(64, 300, 8192) == 512
    assert om.grow_capacity(4096, 5000, 6000) == 6000
    assert om.grow_capacity(128, 100, 8192) == 128


def test_grow_on_demand_is_bitwise_full_preallocation():
    rng = np.random.default_rng(12)
    L, kv, max_ctx = 3, 6, 300
    rows = rng.standard_normal((L, max_ctx, kv)).astype(np.float32)
    full = np.zeros((L * max_ctx, kv), np.float32)
    cap = om.initial_capacity(max_ctx)
    grown = np.zeros((L * cap, kv), np.float32)
    relayouts = 0
    for pos in range(max_ctx):
        if pos >= cap:  # the write path grows before handing out the row
            nc = om.grow_capacity(cap, pos + 1, max_ctx)
            grown = om.kv_relayout(grown, L, cap, nc)
            cap = nc
            relayouts += 1
        for l in range(L):
            full[l * max_ctx + pos] = rows[l, pos]
            grown[l * cap + pos] = rows[l, pos]
    assert relayouts <= int(np.ceil(np.log2(max_ctx)))
    for l in range(L):
        assert np.array_equal(grown[l * cap:l * cap + max_ctx].view(np.uint32),
                              full[l * max_ctx:(l + 1) * max_ctx].view(np.uint32))
