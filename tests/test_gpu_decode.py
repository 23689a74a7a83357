"""GPU parity of paged decode attention (and the store that precedes it)
against the CPU oracle, through the C ABI.

Tolerances: f32 KV max |err| <= 1e-4, f16 and q8_0 KV <= 2e-3 (the oracle
reads the identical stored values in float64). Sizes span several blocks
per CTA range, ragged tails, and forced split counts so every sequence is
cut into several partials.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import formats as ofmt
from oracle import moves as om
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import (TOL, assert_close, assert_lse, gpu_decode, oracle_decode,
                            oracle_pools, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def _store_both(mt, w, kp, vp, k_dev, v_dev, cells=None, k_new=None, v_new=None):
    cells = w.new_cells if cells is None else cells
    k_new = w.k_new if k_new is None else k_new
    v_new = w.v_new if v_new is None else v_new
    oatt.kv_store(w.fmt, kp, vp, k_new, v_new, cells, w.n_kv_heads, w.head_dim)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.mt_kv_store(w.fmt, k_dev, v_dev, w.n_kv_heads, w.head_dim, to_dev(k_new), to_dev(v_new),
                   to_dev(np.asarray(cells, dtype=np.int64)), status=status)
    assert mt.mt_check_device_status(status) == 0


def _run(mt, w, n_ctas=0, table=None, store=True):
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    if store:
        _store_both(mt, w, kp, vp, k_dev, v_dev)
        assert np.array_equal(k_dev.cpu().numpy(), kp) and np.array_equal(v_dev.cpu().numpy(), vp)
    want, want_lse = oracle_decode(w, kp, vp, table=table)
    got, got_lse, st = gpu_decode(mt, w, k_dev, v_dev, table=table, n_ctas=n_ctas)
    assert st == 0, mt.mt_last_error()
    tol = TOL[w.fmt]
    assert_close(got, want, tol, w.name)
    assert_lse(got_lse, want_lse, tol, w.name)
    return got, want


def test_tiny_f32_config(mt):
    w = workloads.tiny_f32()
    assert list(w.context_lens) == [37, 100] and w.block_table[1, 2] == -1
    _run(mt, w)


@pytest.mark.parametrize("n_ctas", [0, 1, 2, 3, 7, 64, 1000])
def test_llama3_f16_small(mt, n_ctas):
    w = workloads.llama3_f16(seed=3, n_seqs=6, ctx_lo=20, ctx_hi=700)
    _run(mt, w, n_ctas=n_ctas)


def test_smollm2_f32_small(mt):
    w = workloads.smollm2_f32(seed=2, n_seqs=4, ctx_lo=50, ctx_hi=400)
    _run(mt, w)
    _run(mt, w, n_ctas=5)


def test_q8_prefix_windows_and_cow(mt):
    # prefix of 100 positions at block size 32: the fourth prefix block is
    # shared and partly filled, so each fork's first append copies it
    w = workloads.llama3_q8_prefix(seed=4, n_seqs=5, prefix=100, suffix_lo=10, suffix_hi=80)
    cow = w.extra["cow_moves"]
    assert len(cow) == w.n_seqs - 1
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    shared_block = cow[0][0] // w.block_size
    n_shared_rows = w.extra["prefix"] % w.block_size  # prefix rows in that block
    before = kp[shared_block * 32:shared_block * 32 + n_shared_rows].copy()
    # copy-on-write: oracle mover on the host, libmtkv mover on the device
    ordered = om.order_moves(cow)
    assert om.find_hazard(ordered) is None
    om.copy_cells([kp, vp], ordered)
    rb = ofmt.row_bytes("q8_0", w.n_kv_heads, w.head_dim)
    mt.mt_copy_cells([k_dev, v_dev], rb, w.n_cells, mt.mt_order_moves(cow))
    _store_both(mt, w, kp, vp, k_dev, v_dev)
    assert np.array_equal(k_dev.cpu().numpy(), kp) and np.array_equal(v_dev.cpu().numpy(), vp)
    # the shared prefix rows were never written in place
    assert np.array_equal(kp[shared_block * 32:shared_block * 32 + n_shared_rows], before)
    assert (w.spans[:, 0] < w.spans[:, 1]).all()
    want, want_lse = oracle_decode(w, kp, vp)
    for n_ctas in (0, 3):
        got, got_lse, st = gpu_decode(mt, w, k_dev, v_dev, n_ctas=n_ctas)
        assert st == 0
        assert_close(got, want, TOL["q8_0"], "q8_0 windows")
        assert_lse(got_lse, want_lse, TOL["q8_0"], "q8_0 windows")


def test_longctx_holes_and_int4_round_trip(mt):
    w = workloads.longctx_f16_int4(seed=5, n_seqs=3, ctx=600)
    hkv, d, bs = w.n_kv_heads, w.head_dim, w.block_size
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    _store_both(mt, w, kp, vp, k_dev, v_dev)
    src, dst = w.extra["cold_src"], w.extra["cold_dst"]
    assert len(src) > 4 and (w.block_table == -1).sum() > 0
    n_elts = bs * hkv * d
    for pool_host, pool_dev in ((kp, k_dev), (vp, v_dev)):
        scales = torch.empty(len(src), dtype=torch.float32, device="cuda")
        nib = torch.empty(len(src), n_elts // 2, dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        mt.mt_kv_quant_int4("f16", pool_dev, bs, hkv, d, w.n_phys_blocks, to_dev(src), scales,
                            nib, status=status)
        mt.mt_kv_dequant_int4("f16", pool_dev, bs, hkv, d, w.n_phys_blocks, to_dev(dst), scales,
                              nib, status=status)
        assert mt.mt_check_device_status(status) == 0
        g_scales, g_nib = scales.cpu().numpy(), nib.cpu().numpy()
        for i, (b_src, b_dst) in enumerate(zip(src, dst)):
            blk = pool_host[b_src * bs:(b_src + 1) * bs].view(np.float16)
            s, n = ofmt.int4_quantize_block(blk)
            assert g_scales[i].view(np.uint32) == np.float32(s).view(np.uint32)
            assert np.array_equal(g_nib[i], n)
            back = ofmt.int4_dequantize_block(s, n, n_elts, "f16")
            pool_host[b_dst * bs:(b_dst + 1) * bs] = back.view(np.uint8).reshape(bs, -1)
        assert np.array_equal(pool_dev.cpu().numpy(), pool_host)
    table = workloads.retarget_cold(w)
    want, want_lse = oracle_decode(w, kp, vp, table=table)
    got, got_lse, st = gpu_decode(mt, w, k_dev, v_dev, table=table)
    assert st == 0
    assert_close(got, want, TOL["f16"], "longctx")
    assert_lse(got_lse, want_lse, TOL["f16"], "longctx")


SHAPES = [  # fmt, head_dim, block_size, n_heads, n_kv_heads
    ("f32", 64, 16, 4, 2), ("f32", 128, 32, 8, 8), ("f32", 256, 16, 2, 1),
    # f32 rows of 8 x 128 floats: 8-row tensor-core stages (query groups 4, 1)
    ("f32", 128, 16, 32, 8), ("f32", 128, 16, 7, 7),
    ("f16", 64, 32, 8, 1), ("f16", 128, 16, 32, 8), ("f16", 256, 16, 16, 4),
    ("f16", 128, 32, 24, 4), ("f16", 64, 16, 21, 3), ("f16", 128, 16, 5, 5),
    ("q8_0", 64, 16, 6, 2), ("q8_0", 128, 32, 32, 8), ("q8_0", 256, 16, 16, 4),
    ("q8_0", 128, 16, 8, 1), ("q8_0", 64, 32, 9, 3),
    # head_dim 128 q8_0 on the direct-operand consumer: paired 16-row blocks
    # (32-byte chunks at 8 heads, 16-byte chunks at 2), whole 32-row blocks
    # through the 16-byte-chunk map (6 heads), query groups 1, 4 and 8
    ("q8_0", 128, 16, 32, 8), ("q8_0", 128, 16, 16, 2), ("q8_0", 128, 32, 6, 6),
    ("q8_0", 128, 16, 12, 4),
]


@pytest.mark.parametrize("fmt,d,bs,hq,hkv", SHAPES)
def test_shape_grid(mt, fmt, d, bs, hq, hkv):
    w = workloads.llama3_f16(seed=7 + d + bs + hq, n_seqs=5, ctx_lo=1, ctx_hi=300, fmt=fmt,
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    _run(mt, w, n_ctas=0)
    _run(mt, w, n_ctas=4, store=False)


def test_edge_cases(mt):
    w = workloads.llama3_f16(seed=9, n_seqs=8, ctx_lo=40, ctx_hi=200)
    bs = w.block_size
    ctx = w.context_lens.copy()
    ctx[0] = 0          # empty sequence
    ctx[1] = 1          # one position
    ctx[2] = 2 * bs     # block aligned
    w.context_lens = ctx
    w.new_cells[0] = -1
    w.new_cells[1] = w.block_table[1, 0] * bs
    w.new_cells[2] = w.block_table[2, 1] * bs + bs - 1
    w.block_table[3, :] = -1          # every block a hole
    nb4 = -(-int(ctx[4]) // bs)
    w.block_table[4, 0:nb4 - 1] = -1  # all but the last block are holes
    spans = np.zeros((8, 2), dtype=np.int32)
    spans[:, 1] = ctx
    spans[5] = (10, 10)               # empty window
    spans[6] = (-7, bs)               # starts below 0, ends on a block edge
    spans[7] = (bs + 3, 10 ** 6)      # ends past the context
    w.spans = spans
    w.new_cells[3] = -1
    got, want = _run(mt, w)
    assert (got[0] == 0).all() and (got[3] == 0).all() and (got[5] == 0).all()
    _run(mt, w, n_ctas=2, store=False)


def test_out_of_range_ids_are_flagged_not_read(mt):
    w = workloads.llama3_f16(seed=10, n_seqs=3, ctx_lo=60, ctx_hi=90)
    kp, vp = oracle_pools(w)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    table = w.block_table.copy()
    table[1, 1] = w.n_phys_blocks + 5
    table[2, 0] = -3
    _, _, st = gpu_decode(mt, w, k_dev, v_dev, table=table)
    assert st == mt.MT_ERR_DEVICE_CHECK
    # the flagged entries were skipped: they read as holes
    t2 = table.copy()
    t2[1, 1] = -1
    t2[2, 0] = -1
    want, _ = oracle_decode(w, kp, vp, table=t2)
    got, _, st = gpu_decode(mt, w, k_dev, v_dev, table=table)
    assert_close(got, want, TOL["f16"], "flagged ids")
    # a context length beyond the table is clamped and flagged
    ctx = w.context_lens.copy()
    ctx[0] = w.max_blocks * w.block_size + 50
    _, _, st = gpu_decode(mt, w, k_dev, v_dev, context_lens=ctx)
    assert st == mt.MT_ERR_DEVICE_CHECK


def test_store_formats_bit_exact(mt):
    rng = np.random.default_rng(30)
    for fmt in ("f32", "f16", "q8_0"):
        for hkv, d in ((2, 64), (8, 128), (3, 96)):
            n_cells = 64
            rb = ofmt.row_bytes(fmt, hkv, d)
            kp = rng.integers(0, 256, (n_cells, rb), dtype=np.uint8)
            vp = rng.integers(0, 256, (n_cells, rb), dtype=np.uint8)
            rows = (rng.standard_normal((20, hkv * d)) * rng.uniform(0.01, 100)).astype(np.float32)
            rows[3, :32] = 0.0                    # an all-zero q8_0 group
            rows[4, :32] = np.float32(2.5)        # ties after division
            # scale 3: x / d = k + 1/2 exactly, while x * fl(1/3) misses the tie
            ks = rng.integers(-127, 127, 32)
            rows[6, :32] = (3.0 * (ks + 0.5)).astype(np.float32)
            rows[6, 0] = np.float32(381.0)        # amax = 3 * 127
            # a group whose scale is subnormal (its reciprocal overflows)
            rows[7, :32] = (rng.standard_normal(32) * 1e-38).astype(np.float32)
            cells = rng.permutation(n_cells)[:20].astype(np.int64)
            cells[5] = -1                         # skipped row
            k_dev, v_dev = to_dev(kp), to_dev(vp)
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            mt.mt_kv_store(fmt, k_dev, v_dev, hkv, d, to_dev(rows), to_dev(-rows), to_dev(cells),
                           status=status)
            oatt.kv_store(fmt, kp, vp, rows, -rows, cells, hkv, d)
            assert mt.mt_check_device_status(status) == 0
            assert np.array_equal(k_dev.cpu().numpy(), kp), (fmt, hkv, d)
            assert np.array_equal(v_dev.cpu().numpy(), vp), (fmt, hkv, d)
    # a cell past the pool is skipped and flagged
    k_dev = torch.zeros(4, 256, dtype=torch.uint8, device="cuda")
    v_dev = torch.zeros_like(k_dev)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    row = torch.ones(1, 64, dtype=torch.float32, device="cuda")
    mt.mt_kv_store("f32", k_dev, v_dev, 1, 64, row, row,
                   torch.tensor([7], dtype=torch.int64, device="cuda"), status=status)
    assert mt.mt_check_device_status(status) == mt.MT_ERR_DEVICE_CHECK
    assert int(k_dev.sum()) == 0


def test_store_q8_0_hand_worked_blocks(mt):
    # The GPU quantiser against the hand-worked blocks themselves (not only
    # against the oracle): among them, groups whose f16 scale differs from the
    # float32 amax/127 in either direction, one subnormal, and ties.
    from tests import golden
    blocks = golden.q8_0_blocks()
    rows = np.array([x for x, _ in blocks], dtype=np.float32)      # [n][32]: 1 head, d 32
    n = rows.shape[0]
    k_dev = torch.zeros(n, 36, dtype=torch.uint8, device="cuda")
    v_dev = torch.zeros_like(k_dev)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cells = torch.arange(n, dtype=torch.int64, device="cuda")
    mt.mt_kv_store("q8_0", k_dev, v_dev, 1, 32, to_dev(rows), to_dev(-rows), cells, status=status)
    assert mt.mt_check_device_status(status) == 0
    k = k_dev.cpu().numpy()
    for i, (_, want) in enumerate(blocks):
        assert list(k[i, :34]) == want, i
        assert list(k[i, 34:]) == [0, 0]
