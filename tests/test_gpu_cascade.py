"""GPU parity of the shared-prefix (cascade) decode against the oracle.

The cascade is an execution strategy: for any batch whose groups really
share their leading block-table entries, mt_paged_attn_decode_cascade must
give what the oracle's plain decode gives (f32 1e-4, f16 and q8_0 2e-3).
Groups are made by pointing the first k table entries of a run of sequences
at the same physical blocks, which is exactly what a refcounted fork does.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import moves as om
from oracle import formats as ofmt
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import (TOL, assert_close, assert_lse, oracle_decode, oracle_pools,
                            to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def share(table, groups):
    """Table in which each group's sequences use the first sequence's first
    n_prefix_blocks entries."""
    t = table.copy()
    for b, e, nb in groups:
        for s in range(b + 1, e):
            t[s, :nb] = t[b, :nb]
    return t


def cascade(mt, w, k_dev, v_dev, table, groups, spans="w"):
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda")
    sp = (None if w.spans is None else to_dev(w.spans)) if isinstance(spans, str) else \
        (None if spans is None else to_dev(spans))
    args = mt.paged_attn_args(w.fmt, q, k_dev, v_dev, to_dev(table), to_dev(w.context_lens), out,
                              n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                              n_phys_blocks=w.n_phys_blocks, scale=w.scale, spans=sp, lse=lse)
    nbytes = mt.mt_paged_attn_cascade_workspace_bytes(args, groups)
    assert nbytes > 0, mt.mt_last_error()
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_decode_cascade(args, groups, ws)
    st = mt.mt_check_device_status(ws)
    return out.cpu().numpy(), lse.cpu().numpy(), st


def check(mt, w, groups, table=None, expect_status=0):
    table = share(w.block_table if table is None else table, groups)
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    want, want_lse = oracle_decode(w, kp, vp, table=table)
    got, got_lse, st = cascade(mt, w, k_dev, v_dev, table, groups)
    assert st == expect_status, mt.mt_last_error()
    if expect_status == 0:
        assert_close(got, want, TOL[w.fmt], f"{w.name} cascade")
        assert_lse(got_lse, want_lse, TOL[w.fmt], f"{w.name} cascade")
    return got, want


@pytest.mark.parametrize("groups", [[(0, 6, 3)], [(0, 6, 3), (7, 10, 5)], [(2, 3, 4)],
                                    [(0, 10, 0)], [(0, 10, 6)]])
def test_cascade_llama3_f16(mt, groups):
    w = workloads.llama3_f16(seed=21, n_seqs=10, ctx_lo=30, ctx_hi=400)
    check(mt, w, groups)


def test_cascade_many_sequences_per_tile(mt):
    # 40 sequences with G = 4: tiles of 16 sequences, a ragged third tile
    w = workloads.llama3_f16(seed=22, n_seqs=40, ctx_lo=100, ctx_hi=300)
    check(mt, w, [(0, 40, 5)])
    check(mt, w, [(0, 17, 6), (20, 39, 2)])


def test_cascade_smollm2_f32(mt):
    # f32 (1e-4) through the three-product split, d = 64, G = 3 (padded to 4)
    w = workloads.smollm2_f32(seed=23, n_seqs=9, ctx_lo=60, ctx_hi=300)
    check(mt, w, [(0, 9, 3)])
    check(mt, w, [(1, 4, 2), (5, 9, 4)])


def test_cascade_q8_prefix_windows(mt):
    # the q8_0 shared-prefix configuration, small: windows cut the prefix
    w = workloads.llama3_q8_prefix(seed=24, n_seqs=20, prefix=320, suffix_lo=10, suffix_hi=90)
    kp, vp = oracle_pools(w)
    cow = om.order_moves(w.extra["cow_moves"])
    om.copy_cells([kp, vp], cow)  # no partial block here: prefix % 32 == 0
    assert not cow
    groups = [(0, w.n_seqs, w.extra["prefix"] // w.block_size)]
    # the generator's own tables already share the prefix blocks
    t = w.block_table
    assert (t[1:, :groups[0][2]] == t[0, :groups[0][2]]).all()
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    want, want_lse = oracle_decode(w, kp, vp)
    got, got_lse, st = cascade(mt, w, k_dev, v_dev, t, groups)
    assert st == 0
    assert_close(got, want, TOL["q8_0"], "q8_0 cascade")
    assert_lse(got_lse, want_lse, TOL["q8_0"], "q8_0 cascade")
    # and without windows
    got, got_lse, st = cascade(mt, w, k_dev, v_dev, t, groups, spans=None)
    assert st == 0
    import dataclasses
    want, want_lse = oracle_decode(dataclasses.replace(w, spans=None), kp, vp)
    assert_close(got, want, TOL["q8_0"], "q8_0 cascade, no windows")


@pytest.mark.parametrize("fmt,d,bs,hq,hkv", [("q8_0", 64, 16, 2, 2), ("q8_0", 128, 16, 16, 2),
                                             ("f16", 64, 32, 8, 1), ("f32", 128, 32, 4, 4),
                                             ("f16", 128, 16, 6, 2),
                                             # head_dim 256: Q rows kept in shared memory
                                             ("f16", 256, 16, 16, 4), ("q8_0", 256, 32, 8, 2),
                                             ("q8_0", 256, 16, 5, 1)])
def test_cascade_shape_grid(mt, fmt, d, bs, hq, hkv):
    w = workloads.llama3_f16(seed=25 + d + bs + hq, n_seqs=7, ctx_lo=20, ctx_hi=150, fmt=fmt,
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    check(mt, w, [(0, 7, 2)])


def test_cascade_holes_in_prefix_and_fallback_shape(mt):
    w = workloads.llama3_f16(seed=26, n_seqs=6, ctx_lo=120, ctx_hi=300)
    t = w.block_table.copy()
    t[:, 1] = -1  # a hole inside the shared prefix, in every sequence
    check(mt, w, [(0, 6, 4)], table=t)
    # the long-context shape (head_dim 256, f16) takes the prefix kernel too;
    # f32 pools of head_dim 256 have none and run the plain decode
    w2 = workloads.longctx_f16_int4(seed=27, n_seqs=3, ctx=400)
    check(mt, w2, [(0, 3, 5)])
    w3 = workloads.llama3_f16(seed=29, n_seqs=4, ctx_lo=100, ctx_hi=200, fmt="f32", n_heads=4,
                              n_kv_heads=2, head_dim=256)
    check(mt, w3, [(0, 4, 3)])


def test_cascade_broken_promise_is_flagged(mt):
    w = workloads.llama3_f16(seed=28, n_seqs=5, ctx_lo=100, ctx_hi=200)
    groups = [(0, 5, 3)]
    t = share(w.block_table, groups)
    t[3, 1] = w.block_table[3, 1] if w.block_table[3, 1] != t[0, 1] else t[0, 2]
    kp, vp = oracle_pools(w)
    _, _, st = cascade(mt, w, to_dev(kp), to_dev(vp), t, groups)
    assert st == mt.MT_ERR_DEVICE_CHECK


def test_cascade_rejects_bad_groups(mt):
    w = workloads.llama3_f16(seed=29, n_seqs=4, ctx_lo=40, ctx_hi=60)
    kp, vp = oracle_pools(w)
    q = to_dev(w.q)
    out = torch.zeros_like(q)
    args = mt.paged_attn_args(w.fmt, q, to_dev(kp), to_dev(vp), to_dev(w.block_table),
                              to_dev(w.context_lens), out, n_kv_heads=w.n_kv_heads,
                              block_size=w.block_size, n_phys_blocks=w.n_phys_blocks,
                              scale=w.scale)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for bad in ([(0, 3, 1), (2, 4, 1)], [(3, 2, 1)], [(0, 5, 1)], [(0, 2, -1)],
                [(0, 1, 1)] * 65):
        assert mt.mt_paged_attn_cascade_workspace_bytes(args, bad) == 0
        with pytest.raises(mt.MtError):
            mt.mt_paged_attn_decode_cascade(args, bad, ws)


def test_cascade_with_fused_store(mt):
    # the q8_0 shared-prefix configuration with a partly filled shared block:
    # copy on write first, then one call stores every new row and decodes
    w = workloads.llama3_q8_prefix(seed=30, n_seqs=9, prefix=100, suffix_lo=10, suffix_hi=90)
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    cow = om.order_moves(w.extra["cow_moves"])
    om.copy_cells([kp, vp], cow)
    rb = ofmt.row_bytes("q8_0", w.n_kv_heads, w.head_dim)
    mt.mt_copy_cells([k_dev, v_dev], rb, w.n_cells, cow)
    groups = [(0, w.n_seqs, w.extra["prefix"] // w.block_size)]
    from oracle import attention as oatt
    oatt.kv_store(w.fmt, kp, vp, w.k_new, w.v_new, w.new_cells, w.n_kv_heads, w.head_dim)
    want, want_lse = oracle_decode(w, kp, vp)
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda")
    args = mt.paged_attn_args(w.fmt, q, k_dev, v_dev, to_dev(w.block_table),
                              to_dev(w.context_lens), out, n_kv_heads=w.n_kv_heads,
                              block_size=w.block_size, n_phys_blocks=w.n_phys_blocks,
                              scale=w.scale, spans=to_dev(w.spans), lse=lse)
    ws = torch.zeros(mt.mt_paged_attn_cascade_workspace_bytes(args, groups), dtype=torch.uint8,
                     device="cuda")
    mt.mt_paged_attn_decode_cascade_append(args, groups, to_dev(w.k_new), to_dev(w.v_new), ws)
    assert mt.mt_check_device_status(ws) == 0
    assert np.array_equal(k_dev.cpu().numpy(), kp) and np.array_equal(v_dev.cpu().numpy(), vp)
    assert_close(out.cpu().numpy(), want, TOL["q8_0"], "cascade + fused store")
    assert_lse(lse.cpu().numpy(), want_lse, TOL["q8_0"], "cascade + fused store")


def _prefix_map(rng, lens, n_prefix, extra):
    """Set-valued windows: the shared prefix [0, n_prefix), one private run
    after it, and `extra` random runs anywhere (some reaching into the
    prefix, some past the context)."""
    mp = np.zeros((len(lens), 8, 2), dtype=np.int32)
    for s, c in enumerate(lens):
        c = int(c)
        mp[s, 0] = (0, n_prefix)
        a = int(rng.integers(n_prefix, max(c, n_prefix + 1)))
        mp[s, 1] = (a, int(rng.integers(1, max(c - a, 1) + 8)))
        for r in range(2, 2 + extra):
            mp[s, r] = (int(rng.integers(-4, c + 4)), int(rng.integers(-2, max(c // 4, 3))))
    return mp


@pytest.mark.parametrize("fmt,d,bs,hq,hkv,extra", [("f16", 128, 16, 32, 8, 0),
                                                   ("q8_0", 128, 32, 32, 8, 3),
                                                   ("f32", 64, 16, 9, 3, 2),
                                                   ("q8_0", 64, 16, 8, 2, 6)])
def test_cascade_kv_map_prefix_plus_private_run(mt, fmt, d, bs, hq, hkv, extra):
    # "KV Cache Design — cells, format, sessions", section 1: a set-valued
    # window (shared prefix + private run) goes through kv_map; the cascade
    # must equal the plain kv_map decode of the oracle
    rng = np.random.default_rng(90 + d + bs + extra)
    w = workloads.llama3_f16(seed=91 + extra, n_seqs=11, ctx_lo=100, ctx_hi=400, fmt=fmt,
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    nblk = 3
    groups = [(0, 6, nblk), (6, 11, nblk - 1)]
    table = share(w.block_table, groups)
    kp, vp = oracle_pools(w)
    mp = _prefix_map(rng, w.context_lens, nblk * bs, extra)
    mp[6:, 0] = ((nblk - 1) * bs) // 2, (nblk - 1) * bs  # the second group: part of its prefix
    want, want_lse = oatt.paged_attn_decode_map(w.fmt, w.q, kp, vp, table, w.context_lens, mp,
                                                w.n_heads, w.n_kv_heads, w.head_dim,
                                                w.block_size, w.scale)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda")
    args = mt.paged_attn_args(w.fmt, q, k_dev, v_dev, to_dev(table), to_dev(w.context_lens), out,
                              n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                              n_phys_blocks=w.n_phys_blocks, scale=w.scale, lse=lse,
                              kv_map=to_dev(mp))
    ws = torch.zeros(mt.mt_paged_attn_cascade_workspace_bytes(args, groups), dtype=torch.uint8,
                     device="cuda")
    mt.mt_paged_attn_decode_cascade(args, groups, ws)
    assert mt.mt_check_device_status(ws) == 0, mt.mt_last_error()
    assert_close(out.cpu().numpy(), want, TOL[w.fmt], f"{w.name} cascade kv_map")
    assert_lse(lse.cpu().numpy(), want_lse, TOL[w.fmt], f"{w.name} cascade kv_map")
