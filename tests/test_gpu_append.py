"""GPU parity of decode with the store fused in (mt_paged_attn_decode_append).

The oracle stores each sequence's new row into the cell of position ctx-1
(kv_store) and then runs the decode; the fused call must leave both pools
bit-identical to the oracle's and match its outputs within the decode
tolerances (f32 1e-4, f16 and q8_0 2e-3).
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import moves as om
from oracle import formats as ofmt
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, assert_lse, oracle_pools, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def _append_cells(w, table, lens):
    """Cell of position ctx-1 of every sequence (-1: nothing to store)."""
    cells = np.full(w.n_seqs, -1, dtype=np.int64)
    for s in range(w.n_seqs):
        c = int(lens[s])
        if c <= 0:
            continue
        blk = int(table[s, (c - 1) // w.block_size])
        if blk >= 0:
            cells[s] = blk * w.block_size + (c - 1) % w.block_size
    return cells


def _fused(mt, w, k_dev, v_dev, table=None, n_ctas=0, lens=None):
    table = w.block_table if table is None else table
    lens = w.context_lens if lens is None else lens
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda")
    sp = None if w.spans is None else to_dev(w.spans)
    args = mt.paged_attn_args(w.fmt, q, k_dev, v_dev, to_dev(table), to_dev(lens), out,
                              n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                              n_phys_blocks=w.n_phys_blocks, scale=w.scale, spans=sp, lse=lse,
                              n_ctas=n_ctas)
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args), dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_decode_append(args, to_dev(w.k_new), to_dev(w.v_new), ws)
    st = mt.mt_check_device_status(ws)
    return out.cpu().numpy(), lse.cpu().numpy(), st


def _check(mt, w, n_ctas=0, table=None, lens=None, expect_status=0, prepare=None):
    table = w.block_table if table is None else table
    lens = w.context_lens if lens is None else lens
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    if prepare is not None:
        prepare(kp, vp, k_dev, v_dev)
    cells = _append_cells(w, table, lens)
    oatt.kv_store(w.fmt, kp, vp, w.k_new, w.v_new, cells, w.n_kv_heads, w.head_dim)
    want, want_lse = oatt.paged_attn_decode(w.fmt, w.q, kp, vp, table, lens, w.spans, w.n_heads,
                                            w.n_kv_heads, w.head_dim, w.block_size, w.scale)
    got, got_lse, st = _fused(mt, w, k_dev, v_dev, table=table, n_ctas=n_ctas, lens=lens)
    assert st == expect_status, mt.mt_last_error()
    assert np.array_equal(k_dev.cpu().numpy(), kp), "K pool differs from the oracle's store"
    assert np.array_equal(v_dev.cpu().numpy(), vp), "V pool differs from the oracle's store"
    assert_close(got, want, TOL[w.fmt], w.name)
    assert_lse(got_lse, want_lse, TOL[w.fmt], w.name)


def test_append_tiny_f32(mt):
    w = workloads.tiny_f32()
    _check(mt, w)
    _check(mt, w, n_ctas=3)


@pytest.mark.parametrize("n_ctas", [0, 1, 5, 64])
def test_append_llama3_f16(mt, n_ctas):
    w = workloads.llama3_f16(seed=13, n_seqs=6, ctx_lo=20, ctx_hi=700)
    _check(mt, w, n_ctas=n_ctas)


def test_append_smollm2_f32(mt):
    w = workloads.smollm2_f32(seed=12, n_seqs=4, ctx_lo=50, ctx_hi=400)
    _check(mt, w, n_ctas=7)


def test_append_q8_prefix_windows(mt):
    # random windows: many sequences' position ctx-1 lies outside their
    # window, so their rows are written by the "read by no CTA" path
    w = workloads.llama3_q8_prefix(seed=14, n_seqs=6, prefix=100, suffix_lo=10, suffix_hi=80)
    assert (w.spans[:, 1] < w.context_lens).any()
    cow = om.order_moves(w.extra["cow_moves"])
    rb = ofmt.row_bytes("q8_0", w.n_kv_heads, w.head_dim)

    def prepare(kp, vp, k_dev, v_dev):
        om.copy_cells([kp, vp], cow)
        mt.mt_copy_cells([k_dev, v_dev], rb, w.n_cells, cow)

    for n_ctas in (0, 4):
        _check(mt, w, n_ctas=n_ctas, prepare=prepare)


def test_append_longctx_wide_rows(mt):
    # head_dim 256 f16 (2 KB rows), holes elsewhere in the table
    w = workloads.longctx_f16_int4(seed=15, n_seqs=3, ctx=600)
    _check(mt, w)


def test_append_hole_and_empty_sequence(mt):
    w = workloads.llama3_f16(seed=16, n_seqs=4, ctx_lo=40, ctx_hi=300)
    table = w.block_table.copy()
    lens = w.context_lens.copy()
    # sequence 1: the block of position ctx-1 is a hole -> nothing stored,
    # flagged; sequence 2: empty context -> nothing stored, output 0
    table[1, (int(lens[1]) - 1) // w.block_size] = -1
    lens[2] = 0
    _check(mt, w, table=table, lens=lens, expect_status=mt.MT_ERR_DEVICE_CHECK)
