"""GPU parity of decode with set-valued (kv_map) windows against the oracle.

Each sequence's query reads the union of up to 8 (start, len) runs of
logical positions, intersected with [0, ctx) and with holes removed
("KV Cache Design — cells, format, sessions", section 1: the third window
mode). Tolerances as the decode: f32 1e-4, f16 and q8_0 2e-3.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, assert_lse, oracle_pools, to_dev

pytestmark = pytest.mark.gpu
MAXR = 8


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def random_map(rng, lens, n_runs=None):
    mp = np.zeros((len(lens), MAXR, 2), dtype=np.int32)
    for s, c in enumerate(lens):
        k = int(rng.integers(0, MAXR + 1)) if n_runs is None else n_runs
        for r in range(k):
            a = int(rng.integers(-8, int(c) + 8))
            mp[s, r] = (a, int(rng.integers(-3, max(int(c) // 3, 3))))
    return mp


def decode_map(mt, w, kp, vp, kv_map, table=None, n_ctas=0, spans=None, k_new=None):
    table = w.block_table if table is None else table
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda")
    args = mt.paged_attn_args(w.fmt, q, k_dev, v_dev, to_dev(table), to_dev(w.context_lens), out,
                              n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                              n_phys_blocks=w.n_phys_blocks, scale=w.scale, lse=lse,
                              n_ctas=n_ctas, kv_map=to_dev(kv_map),
                              spans=None if spans is None else to_dev(spans))
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args) or 256, dtype=torch.uint8,
                     device="cuda")
    if k_new is None:
        mt.mt_paged_attn_decode(args, ws)
    else:
        mt.mt_paged_attn_decode_append(args, to_dev(k_new[0]), to_dev(k_new[1]), ws)
    st = mt.mt_check_device_status(ws)
    return out.cpu().numpy(), lse.cpu().numpy(), st, (k_dev, v_dev)


def check(mt, w, kv_map, table=None, n_ctas=0):
    table = w.block_table if table is None else table
    kp, vp = oracle_pools(w)
    want, want_lse = oatt.paged_attn_decode_map(w.fmt, w.q, kp, vp, table, w.context_lens, kv_map,
                                                w.n_heads, w.n_kv_heads, w.head_dim,
                                                w.block_size, w.scale)
    got, got_lse, st, _ = decode_map(mt, w, kp, vp, kv_map, table=table, n_ctas=n_ctas)
    assert st == 0, mt.mt_last_error()
    assert_close(got, want, TOL[w.fmt], f"{w.name} kv_map")
    assert_lse(got_lse, want_lse, TOL[w.fmt], f"{w.name} kv_map")


@pytest.mark.parametrize("n_ctas", [0, 1, 7])
def test_kv_map_f16_tensor_core_path(mt, n_ctas):
    rng = np.random.default_rng(61)
    w = workloads.llama3_f16(seed=61, n_seqs=8, ctx_lo=20, ctx_hi=500)
    check(mt, w, random_map(rng, w.context_lens), n_ctas=n_ctas)


def test_kv_map_q8_and_f32(mt):
    rng = np.random.default_rng(62)
    w = workloads.llama3_q8_prefix(seed=62, n_seqs=6, prefix=96, suffix_lo=10, suffix_hi=120,
                                   windows=False)
    check(mt, w, random_map(rng, w.context_lens))
    w2 = workloads.smollm2_f32(seed=62, n_seqs=5, ctx_lo=40, ctx_hi=300)
    check(mt, w2, random_map(rng, w2.context_lens))


@pytest.mark.parametrize("fmt,d,bs,hq,hkv", [("f16", 256, 16, 16, 4), ("q8_0", 256, 16, 16, 4),
                                             ("f32", 256, 16, 2, 1), ("q8_0", 64, 32, 9, 3),
                                             ("f16", 64, 32, 8, 1), ("f32", 128, 32, 8, 8)])
def test_kv_map_shape_grid(mt, fmt, d, bs, hq, hkv):
    rng = np.random.default_rng(63 + d + bs + hq)
    w = workloads.llama3_f16(seed=63 + d + hq, n_seqs=5, ctx_lo=1, ctx_hi=300, fmt=fmt,
                             block_size=bs, n_heads=hq, n_kv_heads=hkv, head_dim=d)
    check(mt, w, random_map(rng, w.context_lens))
    check(mt, w, random_map(rng, w.context_lens), n_ctas=3)


def test_kv_map_reduces_to_plain_decode_and_empty(mt):
    rng = np.random.default_rng(64)
    w = workloads.llama3_f16(seed=64, n_seqs=5, ctx_lo=30, ctx_hi=200)
    t = w.block_table.copy()
    t[1, 1] = -1  # a hole inside a run
    mp = np.zeros((w.n_seqs, MAXR, 2), dtype=np.int32)
    mp[:, 3] = np.stack([np.zeros(w.n_seqs), w.context_lens], axis=1)  # one run = [0, ctx)
    mp[2] = 0  # no run at all: output 0, lse -inf
    check(mt, w, mp, table=t)
    # duplicated and overlapping runs read each position once
    mp2 = np.zeros((w.n_seqs, MAXR, 2), dtype=np.int32)
    mp2[:, 0] = (0, 20)
    mp2[:, 1] = (10, 20)
    mp2[:, 2] = (0, 20)
    check(mt, w, mp2, table=t)


def test_kv_map_with_fused_store(mt):
    rng = np.random.default_rng(65)
    w = workloads.llama3_f16(seed=65, n_seqs=6, ctx_lo=40, ctx_hi=300)
    mp = random_map(rng, w.context_lens, n_runs=3)
    mp[0, 0] = (int(w.context_lens[0]) - 5, 5)  # sequence 0 reads its new row
    kp, vp = oracle_pools(w)
    oatt.kv_store(w.fmt, kp, vp, w.k_new, w.v_new, w.new_cells, w.n_kv_heads, w.head_dim)
    want, want_lse = oatt.paged_attn_decode_map(w.fmt, w.q, kp, vp, w.block_table,
                                                w.context_lens, mp, w.n_heads, w.n_kv_heads,
                                                w.head_dim, w.block_size, w.scale)
    kp0, vp0 = oracle_pools(w)
    got, got_lse, st, (k_dev, v_dev) = decode_map(mt, w, kp0, vp0, mp, k_new=(w.k_new, w.v_new))
    assert st == 0
    assert np.array_equal(k_dev.cpu().numpy(), kp) and np.array_equal(v_dev.cpu().numpy(), vp)
    assert_close(got, want, TOL[w.fmt], "kv_map + fused store")
    assert_lse(got_lse, want_lse, TOL[w.fmt], "kv_map + fused store")


def test_kv_map_rejected_with_spans(mt):
    rng = np.random.default_rng(66)
    w = workloads.llama3_f16(seed=66, n_seqs=3, ctx_lo=30, ctx_hi=60)
    kp, vp = oracle_pools(w)
    mp = random_map(rng, w.context_lens)
    sp = np.stack([np.zeros(3), w.context_lens], axis=1).astype(np.int32)
    with pytest.raises(mt.MtError):
        decode_map(mt, w, kp, vp, mp, spans=sp)
