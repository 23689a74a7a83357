"""GPU parity of multi-query (prefill) paged attention against the oracle.

Each sequence's last n positions are queries (chunked prefill; n = ctx is a
full prefill); query j sees positions <= its own, within its optional window
(a [lo, hi) pair or kv_map runs). Tolerances as the decode: f32 1e-4, f16
and q8_0 2e-3 (the oracle reads the identical stored values in float64).
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, assert_lse, oracle_pools, to_dev

pytestmark = pytest.mark.gpu
MAXR = 8  # MT_KV_MAP_MAX_SPANS


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def make_queries(w, rng, max_q, full=()):
    """q_start and random queries: n_s in [0, min(ctx, max_q)] (ctx for `full`)."""
    n = []
    for s in range(w.n_seqs):
        c = int(w.context_lens[s])
        n.append(c if s in full else int(rng.integers(0, min(c, max_q) + 1)))
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = rng.standard_normal((int(q_start[-1]), w.n_heads, w.head_dim)).astype(np.float32)
    return q, q_start


def random_spans(rng, w, q_start):
    sp = np.zeros((int(q_start[-1]), 2), dtype=np.int32)
    for s in range(w.n_seqs):
        c = int(w.context_lens[s])
        for i in range(q_start[s], q_start[s + 1]):
            a, b = sorted(rng.integers(0, c + 1, 2).tolist())
            sp[i] = (a, b)
    return sp


def random_map(rng, w, q_start):
    mp = np.zeros((int(q_start[-1]), MAXR, 2), dtype=np.int32)
    for s in range(w.n_seqs):
        c = int(w.context_lens[s])
        for i in range(q_start[s], q_start[s + 1]):
            for r in range(int(rng.integers(0, MAXR + 1))):
                a = int(rng.integers(-5, c + 5))
                mp[i, r] = (a, int(rng.integers(-2, max(c // 3, 2))))
    return mp


def run_prefill(mt, w, q, q_start, kp, vp, table=None, spans=None, kv_map=None, ctx=None):
    table = w.block_table if table is None else table
    ctx = w.context_lens if ctx is None else ctx
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    qd = to_dev(q)
    n_tok = q.shape[0]
    out = torch.full((n_tok, w.n_heads, w.head_dim), float("nan"), device="cuda")
    lse = torch.full((n_tok, w.n_heads), float("nan"), device="cuda")
    args = mt.prefill_args(w.fmt, qd, k_dev, v_dev, to_dev(table), to_dev(ctx), to_dev(q_start),
                           out, n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                           n_phys_blocks=w.n_phys_blocks, scale=w.scale,
                           spans=None if spans is None else to_dev(spans),
                           kv_map=None if kv_map is None else to_dev(kv_map), lse=lse)
    ws = torch.zeros(mt.mt_paged_prefill_workspace_bytes(args), dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_prefill(args, ws)
    st = mt.mt_check_device_status(ws)
    return out.cpu().numpy(), lse.cpu().numpy(), st


def check(mt, w, q, q_start, table=None, spans=None, kv_map=None, ctx=None, expect_status=0):
    kp, vp = oracle_pools(w)
    table = w.block_table if table is None else table
    ctx = w.context_lens if ctx is None else ctx
    want, want_lse = oatt.paged_attn_prefill(w.fmt, q, kp, vp, table, ctx, q_start, spans, kv_map,
                                             w.n_heads, w.n_kv_heads, w.head_dim, w.block_size,
                                             w.scale)
    got, got_lse, st = run_prefill(mt, w, q, q_start, kp, vp, table, spans, kv_map, ctx)
    assert st == expect_status, mt.mt_last_error()
    assert_close(got, want, TOL[w.fmt], f"{w.name} prefill")
    assert_lse(got_lse, want_lse, TOL[w.fmt], f"{w.name} prefill")


def test_prefill_f16_chunked_and_full(mt):
    rng = np.random.default_rng(51)
    w = workloads.llama3_f16(seed=51, n_seqs=6, ctx_lo=20, ctx_hi=300)
    q, q_start = make_queries(w, rng, 40, full=(2,))
    check(mt, w, q, q_start)


def test_prefill_f32_gqa3(mt):
    rng = np.random.default_rng(52)
    w = workloads.smollm2_f32(seed=52, n_seqs=4, ctx_lo=30, ctx_hi=200)
    q, q_start = make_queries(w, rng, 30, full=(1,))
    check(mt, w, q, q_start)


def test_prefill_q8_with_spans(mt):
    rng = np.random.default_rng(53)
    w = workloads.llama3_q8_prefix(seed=53, n_seqs=5, prefix=64, suffix_lo=10, suffix_hi=90)
    q, q_start = make_queries(w, rng, 24)
    check(mt, w, q, q_start, spans=random_spans(rng, w, q_start))


def test_prefill_f32_with_spans(mt):
    # f32 pools (staged as high / low f16 pairs) with a random [lo, hi)
    # window per query, contexts of a few chunks
    rng = np.random.default_rng(60)
    w = workloads.llama3_f16(seed=60, n_seqs=4, ctx_lo=100, ctx_hi=400, fmt="f32",
                             n_heads=8, n_kv_heads=2, head_dim=128)
    q, q_start = make_queries(w, rng, 40)
    check(mt, w, q, q_start, spans=random_spans(rng, w, q_start))


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "f32"])
def test_prefill_kv_map_runs(mt, fmt):
    rng = np.random.default_rng(54)
    w = workloads.llama3_f16(seed=54, n_seqs=4, ctx_lo=30, ctx_hi=200, fmt=fmt, block_size=16,
                             n_heads=8, n_kv_heads=2, head_dim=64)
    q, q_start = make_queries(w, rng, 20)
    check(mt, w, q, q_start, kv_map=random_map(rng, w, q_start))


@pytest.mark.parametrize("fmt,d,bs,hq,hkv", [("f16", 64, 32, 8, 1), ("q8_0", 64, 16, 2, 2),
                                             ("f16", 128, 16, 5, 5), ("f32", 128, 32, 4, 2),
                                             ("q8_0", 128, 32, 24, 4),
                                             # head_dim 256 (the (256, 16) dispatch tuple of
                                             # "Tiered KV cache — architecture", "Kernel
                                             # dispatch"): Q rows kept in shared memory
                                             ("f16", 256, 16, 16, 4), ("q8_0", 256, 16, 8, 2),
                                             ("f16", 256, 32, 6, 2), ("q8_0", 256, 32, 3, 3)])
def test_prefill_shape_grid(mt, fmt, d, bs, hq, hkv):
    rng = np.random.default_rng(55 + d + bs + hq)
    w = workloads.llama3_f16(seed=55 + d + hq, n_seqs=4, ctx_lo=1, ctx_hi=160, fmt=fmt,
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    q, q_start = make_queries(w, rng, 70)
    check(mt, w, q, q_start)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "f32"])
def test_prefill_holes_and_empty(mt, fmt):
    rng = np.random.default_rng(56)
    w = workloads.llama3_f16(seed=56, n_seqs=5, ctx_lo=40, ctx_hi=200, fmt=fmt)
    table = w.block_table.copy()
    table[0, 1] = -1
    table[3, 0] = -1
    ctx = w.context_lens.copy()
    ctx[4] = 0  # an empty sequence with no queries
    q, q_start = make_queries(dataclass_ctx(w, ctx), rng, 30)
    check(mt, w, q, q_start, table=table, ctx=ctx)


def dataclass_ctx(w, ctx):
    import dataclasses
    return dataclasses.replace(w, context_lens=ctx)


def test_prefill_flags_bad_query_counts(mt):
    rng = np.random.default_rng(57)
    w = workloads.llama3_f16(seed=57, n_seqs=2, ctx_lo=20, ctx_hi=30)
    # sequence 0 claims more queries than positions: flagged, its rows are
    # read as having no position before the context start
    n = [int(w.context_lens[0]) + 3, 2]
    q_start = np.array([0, n[0], n[0] + n[1]], dtype=np.int32)
    q = rng.standard_normal((q_start[-1], w.n_heads, w.head_dim)).astype(np.float32)
    kp, vp = oracle_pools(w)
    _, _, st = run_prefill(mt, w, q, q_start, kp, vp)
    assert st == mt.MT_ERR_DEVICE_CHECK


def test_prefill_rejects_bad_arguments(mt):
    rng = np.random.default_rng(58)
    w = workloads.llama3_f16(seed=58, n_seqs=2, ctx_lo=20, ctx_hi=30)
    q, q_start = make_queries(w, rng, 5)
    kp, vp = oracle_pools(w)
    sp = random_spans(rng, w, q_start)
    mp = random_map(rng, w, q_start)
    with pytest.raises(mt.MtError):
        run_prefill(mt, w, q, q_start, kp, vp, spans=sp, kv_map=mp)
    # f32 pools of head_dim 256 have no multi-query kernel
    w2 = workloads.llama3_f16(seed=59, n_seqs=1, ctx_lo=40, ctx_hi=64, fmt="f32", n_heads=4,
                              n_kv_heads=2, head_dim=256)
    q2, qs2 = make_queries(w2, rng, 4)
    kp2, vp2 = oracle_pools(w2)
    with pytest.raises(mt.MtError) as e:
        run_prefill(mt, w2, q2, qs2, kp2, vp2)
    assert e.value.status == mt.MT_ERR_UNSUPPORTED
