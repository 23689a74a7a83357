"""GPU parity of the tcgen05 prefill kernel (f16 pools; q8_0 pools staged as
f16 rows, f32 pools staged as high / low f16 pairs) at sizes that drive its
pipeline: contexts of many 128-token chunks, more tiles than CTAs (tile
changes with the next tile's query staged during the current one), running
maxima that grow past the lazy-rescale threshold in every chunk, and more
sequences than one launch takes. The oracle and tolerances are those of the
other prefill tests (f16 and q8_0: 2e-3, f32: 1e-4, on outputs and
log-sum-exp).
"""
import dataclasses

import numpy as np
import pytest

from oracle import attention as oatt
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, assert_lse, oracle_pools
from tests.test_gpu_prefill import make_queries, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def check_pools(mt, w, q, q_start, kp, vp):
    want, want_lse = oatt.paged_attn_prefill(w.fmt, q, kp, vp, w.block_table, w.context_lens,
                                             q_start, None, None, w.n_heads, w.n_kv_heads,
                                             w.head_dim, w.block_size, w.scale)
    got, got_lse, st = run_prefill(mt, w, q, q_start, kp, vp)
    assert st == 0, mt.mt_last_error()
    assert_close(got, want, TOL[w.fmt], f"{w.name} prefill")
    assert_lse(got_lse, want_lse, TOL[w.fmt], f"{w.name} prefill")


def test_prefill_tc_long_contexts_many_tiles(mt):
    # Llama-3 heads (GP = 4: 32 queries per tile), contexts of 6-9 chunks and
    # up to 300 queries per sequence: ~200 tiles, so CTAs take several
    # tiles and the staging rings wrap many times
    rng = np.random.default_rng(81)
    w = workloads.llama3_f16(seed=81, n_seqs=3, ctx_lo=700, ctx_hi=1100)
    q, q_start = make_queries(w, rng, 300)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)


@pytest.mark.parametrize("fmt", ["f16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_tc_rescales_growing_maxima(mt, d, fmt):
    # scores that grow by ~8.5 (base 2) per 128 tokens: every chunk raises the
    # running maximum past the 2^8 threshold, so the output row in tensor
    # memory is rescaled in every chunk (f32: probabilities up to 2^8 as
    # high / low f16 pairs)
    rng = np.random.default_rng(82 + d)
    w = workloads.llama3_f16(seed=82 + d, n_seqs=2, ctx_lo=500, ctx_hi=640, n_heads=4,
                             n_kv_heads=1, head_dim=d, fmt=fmt)
    u = np.ones(d, dtype=np.float32) / np.sqrt(d)
    k_hist = w.k_hist.copy()
    for s in range(w.n_seqs):
        for t in range(int(w.context_lens[s])):
            cell = int(w.block_table[s, t // w.block_size]) * w.block_size + t % w.block_size
            # q ~ sqrt(d) u, so q.k * scale * log2(e) ~ gamma * log2(e) = 8.5 t / 128
            gamma = (8.5 / 128.0) * t / 1.4426950408889634
            k_hist[cell] = gamma * u + 0.3 * rng.standard_normal(d).astype(np.float32)
    w = dataclasses.replace(w, k_hist=k_hist)
    q, q_start = make_queries(w, rng, 200)
    q = (np.sqrt(d) * u[None, None, :] + 0.3 * q).astype(np.float32)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)


def test_prefill_tc_more_sequences_than_one_launch(mt):
    # 1100 short sequences: the call runs two launches of at most 1024
    rng = np.random.default_rng(83)
    w = workloads.llama3_f16(seed=83, n_seqs=1100, ctx_lo=1, ctx_hi=12, n_heads=4, n_kv_heads=2,
                             head_dim=64)
    q, q_start = make_queries(w, rng, 6)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)


@pytest.mark.parametrize("hq,hkv,d", [(12, 2, 128), (6, 2, 128), (16, 8, 64), (8, 8, 128)])
def test_prefill_tc_output_boxes(mt, hq, hkv, d):
    # a softmax warp's 32 rows are 32 / GP whole queries; when all are queries
    # of the sequence they leave by tensor stores of box (32 dims, G heads,
    # 32 / GP queries), else by the threads' own stores: query groups of 6
    # and 3 (padded to 8 and 4: the box packs the real heads), 2 and 1, with
    # query counts that end sequences inside a warp's block
    rng = np.random.default_rng(84 + hq + d)
    w = workloads.llama3_f16(seed=84 + hq + d, n_seqs=4, ctx_lo=300, ctx_hi=700, n_heads=hq,
                             n_kv_heads=hkv, head_dim=d)
    q, q_start = make_queries(w, rng, 150)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)


@pytest.mark.parametrize("d,bs,hq,hkv", [(128, 16, 32, 8), (128, 32, 12, 2), (64, 16, 8, 2)])
def test_prefill_tc_q8_0_staged(mt, d, bs, hq, hkv):
    # q8_0 pools run the tcgen05 kernel on rows staged as f16 (code * scale
    # rounded once to f16): contexts of several 128-token chunks, many tiles,
    # a hole, against the oracle's exact dequantisation at the q8_0 tolerance
    rng = np.random.default_rng(86 + d + bs + hq)
    w = workloads.llama3_f16(seed=86 + d + bs, n_seqs=3, ctx_lo=500, ctx_hi=900, fmt="q8_0",
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    table = w.block_table.copy()
    table[1, 2] = -1
    w = dataclasses.replace(w, block_table=table)
    q, q_start = make_queries(w, rng, 260)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)


def test_prefill_tc_q8_0_staged_flags_bad_ids(mt):
    # an out-of-range block id is flagged by the staging pass and read as a
    # hole; the other sequence's rows are unaffected
    rng = np.random.default_rng(87)
    w = workloads.llama3_f16(seed=87, n_seqs=2, ctx_lo=300, ctx_hi=400, fmt="q8_0")
    q, q_start = make_queries(w, rng, 40)
    kp, vp = oracle_pools(w)
    table = w.block_table.copy()
    table[0, 3] = w.n_phys_blocks + 5
    got, _, st = run_prefill(mt, w, q, q_start, kp, vp, table=table)
    assert st == mt.MT_ERR_DEVICE_CHECK
    holed = table.copy()
    holed[0, 3] = -1
    want, _ = oatt.paged_attn_prefill(w.fmt, q, kp, vp, holed, w.context_lens, q_start, None,
                                      None, w.n_heads, w.n_kv_heads, w.head_dim, w.block_size,
                                      w.scale)
    assert_close(got, want, TOL[w.fmt], "q8_0 staged prefill with a bad id")


def test_prefill_tc_q8_0_staged_flags_f16_overflow(mt):
    # a q8_0 group whose values reach past the f16 range (scale 600, codes
    # 127: 76 200) cannot be staged as f16: the staging pass flags it
    rng = np.random.default_rng(88)
    w = workloads.llama3_f16(seed=88, n_seqs=2, ctx_lo=100, ctx_hi=200, fmt="q8_0")
    q, q_start = make_queries(w, rng, 20)
    kp, vp = oracle_pools(w)
    cell = int(w.block_table[0, 0]) * w.block_size  # position 0 of sequence 0
    kp = kp.copy()
    kp[cell, 0:2] = np.frombuffer(np.float16(600.0).tobytes(), dtype=np.uint8)
    kp[cell, 2:34] = 127
    _, _, st = run_prefill(mt, w, q, q_start, kp, vp)
    assert st == mt.MT_ERR_DEVICE_CHECK


@pytest.mark.parametrize("d,bs,hq,hkv", [(128, 16, 32, 8), (128, 32, 12, 2), (64, 16, 8, 2),
                                         (64, 32, 9, 3)])
def test_prefill_tc_f32_paired(mt, d, bs, hq, hkv):
    # f32 pools run the tcgen05 kernel on rows staged as high / low f16
    # pairs (x = high + low to ~2^-22), scores and P.V each from three
    # products: contexts of several 128-token chunks, many tiles, a hole,
    # against the oracle at the f32 tolerance
    rng = np.random.default_rng(90 + d + bs + hq)
    w = workloads.llama3_f16(seed=90 + d + bs, n_seqs=3, ctx_lo=500, ctx_hi=900, fmt="f32",
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    table = w.block_table.copy()
    table[1, 2] = -1
    w = dataclasses.replace(w, block_table=table)
    q, q_start = make_queries(w, rng, 260)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)


def test_prefill_tc_f32_staged_flags_bad_ids(mt):
    # an out-of-range block id is flagged by the f32 staging pass and read as
    # a hole; the other rows are unaffected
    rng = np.random.default_rng(92)
    w = workloads.llama3_f16(seed=92, n_seqs=2, ctx_lo=300, ctx_hi=400, fmt="f32")
    q, q_start = make_queries(w, rng, 40)
    kp, vp = oracle_pools(w)
    table = w.block_table.copy()
    table[1, 4] = w.n_phys_blocks + 7
    got, _, st = run_prefill(mt, w, q, q_start, kp, vp, table=table)
    assert st == mt.MT_ERR_DEVICE_CHECK
    holed = table.copy()
    holed[1, 4] = -1
    want, _ = oatt.paged_attn_prefill(w.fmt, q, kp, vp, holed, w.context_lens, q_start, None,
                                      None, w.n_heads, w.n_kv_heads, w.head_dim, w.block_size,
                                      w.scale)
    assert_close(got, want, TOL[w.fmt], "f32 staged prefill with a bad id")


def test_prefill_tc_f32_flags_f16_overflow(mt):
    # an f32 value outside the f16 range (1e5) has no high / low f16 pair:
    # the staging pass flags it
    rng = np.random.default_rng(91)
    w = workloads.llama3_f16(seed=91, n_seqs=2, ctx_lo=100, ctx_hi=200, fmt="f32")
    q, q_start = make_queries(w, rng, 20)
    kp, vp = oracle_pools(w)
    cell = int(w.block_table[1, 0]) * w.block_size + 3  # position 3 of sequence 1
    vp = vp.copy()
    vp[cell, 5 * 4:6 * 4] = np.frombuffer(np.float32(1.0e5).tobytes(), dtype=np.uint8)
    _, _, st = run_prefill(mt, w, q, q_start, kp, vp)
    assert st == mt.MT_ERR_DEVICE_CHECK


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "f32"])
def test_prefill_tc_split_long_context(mt, fmt):
    # one chunk of a long prompt: ~100 queries at the end of a context of
    # 3000-4000 positions leave 32 tiles for 152 CTAs, so each tile's ~30
    # chunks are cut into pieces whose records the combine merges (f16, and
    # q8_0 and f32 through their staged rows)
    rng = np.random.default_rng(89)
    w = workloads.llama3_f16(seed=89, n_seqs=1, ctx_lo=3000, ctx_hi=4000, fmt=fmt)
    n = 100
    q_start = np.array([0, n], dtype=np.int32)
    q = rng.standard_normal((n, w.n_heads, w.head_dim)).astype(np.float32)
    kp, vp = oracle_pools(w)
    check_pools(mt, w, q, q_start, kp, vp)
