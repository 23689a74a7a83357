"""Pins of the oracle's paged decode attention (CPU only).

The oracle is checked against things fixed outside it:
  * torch's scaled_dot_product_attention (float64, CPU) on the dense
    sequence — a library routine — with the grouped-query map expanded by
    repeat_interleave, on paged layouts with scattered physical blocks;
  * invariants the block model fixes ("Tiered KV cache — architecture",
    section "The paged-attention block model"): the result does not depend
    on which physical blocks hold a sequence; a kInvalidBlockId hole is the
    same as deleting its positions; a window [lo, hi) is the same as slicing
    ("KV Cache Design — cells, format, sessions", section 1);
  * closed forms: one valid position gives o = v; equal keys or a zero
    query give the mean of v and lse = log(n) (+ the common logit);
  * the degenerate case with no valid position: o = 0, lse = -inf.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, formats
from paged_kv_cache_gqa_gb300 import workloads


def _paged_layout(rng, lens, bs, n_phys, row, fmt="f32", n_kv_heads=None, head_dim=None):
    """Scatter dense per-sequence rows over a shuffled pool; returns the pool
    bytes, the table and the dense float32 rows per sequence."""
    perm = rng.permutation(n_phys)
    mb = max(-(-c // bs) for c in lens)
    table = np.full((len(lens), mb), -1, dtype=np.int32)
    k_cells = rng.standard_normal((n_phys * bs, row)).astype(np.float32)
    v_cells = rng.standard_normal((n_phys * bs, row)).astype(np.float32)
    nxt = 0
    for s, c in enumerate(lens):
        for lb in range(-(-c // bs)):
            table[s, lb] = perm[nxt]
            nxt += 1
    kp = formats.encode_rows(fmt, k_cells, n_kv_heads, head_dim)
    vp = formats.encode_rows(fmt, v_cells, n_kv_heads, head_dim)
    return kp, vp, table


def _dense(kp, vp, table_row, ctx, bs, fmt, hkv, d):
    cells = [table_row[p // bs] * bs + p % bs for p in range(ctx)]
    k = formats.decode_rows(fmt, kp[cells], hkv, d).reshape(ctx, hkv, d)
    v = formats.decode_rows(fmt, vp[cells], hkv, d).reshape(ctx, hkv, d)
    return k, v


def _sdpa(q, k, v, scale, G):
    """q [Hq][d], k/v [n][Hkv][d] -> torch SDPA float64 with kv heads expanded."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, :, None, :]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("fmt,hq,hkv,d,bs", [
    ("f32", 4, 2, 64, 16), ("f16", 8, 2, 64, 16), ("q8_0", 8, 2, 64, 32),
    ("f32", 9, 3, 64, 16), ("f16", 4, 4, 32, 16), ("f32", 8, 1, 64, 32),
])
def test_matches_library_sdpa_on_paged_layout(fmt, hq, hkv, d, bs):
    rng = np.random.default_rng(10)
    lens = [1, 37, 100, 16]
    kp, vp, table = _paged_layout(rng, lens, bs, 24, hkv * d, fmt, hkv, d)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    out, lse = attention.paged_attn_decode(fmt, q, kp, vp, table, np.array(lens), None,
                                           hq, hkv, d, bs, scale)
    for s, c in enumerate(lens):
        k, v = _dense(kp, vp, table[s], c, bs, fmt, hkv, d)
        want = _sdpa(q[s], k, v, scale, hq // hkv)
        assert np.allclose(out[s], want, rtol=0, atol=1e-12)
        # lse against a library log-sum-exp of the same logits
        for h in range(hq):
            t = scale * k[:, h // (hq // hkv), :] @ q[s, h].astype(np.float64)
            assert lse[s, h] == pytest.approx(float(torch.logsumexp(torch.from_numpy(t), 0)),
                                              abs=1e-12)


def test_physical_placement_does_not_matter():
    w = workloads.tiny_f32()
    kp = formats.encode_rows("f32", w.k_hist, 2, 64)
    vp = formats.encode_rows("f32", w.v_hist, 2, 64)
    out1, lse1 = attention.paged_attn_decode("f32", w.q, kp, vp, w.block_table,
                                             w.context_lens, None, 4, 2, 64, 16, w.scale)
    # move every physical block b to perm[b] and renumber the table
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.n_phys_blocks)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    for b in range(w.n_phys_blocks):
        kp2[perm[b] * 16:(perm[b] + 1) * 16] = kp[b * 16:(b + 1) * 16]
        vp2[perm[b] * 16:(perm[b] + 1) * 16] = vp[b * 16:(b + 1) * 16]
    t2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    out2, lse2 = attention.paged_attn_decode("f32", w.q, kp2, vp2, t2, w.context_lens, None,
                                             4, 2, 64, 16, w.scale)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_hole_equals_deleting_its_positions():
    w = workloads.tiny_f32()
    assert w.block_table[1, 2] == -1
    kp = formats.encode_rows("f32", w.k_hist, 2, 64)
    vp = formats.encode_rows("f32", w.v_hist, 2, 64)
    out, lse = attention.paged_attn_decode("f32", w.q, kp, vp, w.block_table, w.context_lens,
                                           None, 4, 2, 64, 16, w.scale)
    # dense rows of sequence 1 without positions 32..47, through the library routine
    cells = [w.block_table[1, p // 16] * 16 + p % 16 for p in range(100) if not 32 <= p < 48]
    k = formats.decode_rows("f32", kp[cells], 2, 64).reshape(-1, 2, 64)
    v = formats.decode_rows("f32", vp[cells], 2, 64).reshape(-1, 2, 64)
    assert len(cells) == 84
    assert np.allclose(out[1], _sdpa(w.q[1], k, v, w.scale, 2), atol=1e-12, rtol=0)


def test_window_equals_slicing():
    rng = np.random.default_rng(6)
    lens = [100, 64, 50, 33]
    kp, vp, table = _paged_layout(rng, lens, 16, 20, 2 * 64, "f32", 2, 64)
    q = rng.standard_normal((4, 4, 64)).astype(np.float32)
    # windows: interior, clipped at ctx, starting below 0, empty
    spans = np.array([[17, 83], [40, 999], [-5, 20], [10, 10]], dtype=np.int32)
    out, lse = attention.paged_attn_decode("f32", q, kp, vp, table, np.array(lens), spans,
                                           4, 2, 64, 16, 0.125)
    for s, (lo, hi) in enumerate(spans):
        lo, hi = max(lo, 0), min(hi, lens[s])
        k, v = _dense(kp, vp, table[s], lens[s], 16, "f32", 2, 64)
        if hi <= lo:
            assert (out[s] == 0).all() and (lse[s] == -np.inf).all()
        else:
            want = _sdpa(q[s], k[lo:hi], v[lo:hi], 0.125, 2)
            assert np.allclose(out[s], want, atol=1e-12, rtol=0)


def test_closed_forms():
    rng = np.random.default_rng(7)
    d = 64
    v = rng.standard_normal((5, d))
    # one position: o = v
    o, lse = attention.attend_dense(rng.standard_normal(d), rng.standard_normal((1, d)), v[:1], 0.3)
    assert np.array_equal(o, v[0])
    # equal keys: mean of v, lse = logit + log n
    q = rng.standard_normal(d)
    k = np.tile(rng.standard_normal(d), (5, 1))
    o, lse = attention.attend_dense(q, k, v, 0.125)
    assert np.allclose(o, v.mean(0), atol=1e-14)
    assert lse == pytest.approx(0.125 * float(k[0] @ q) + math.log(5), abs=1e-12)
    # zero query: mean of v, lse = log n
    o, lse = attention.attend_dense(np.zeros(d), rng.standard_normal((5, d)), v, 0.125)
    assert np.allclose(o, v.mean(0), atol=1e-14) and lse == pytest.approx(math.log(5))
    # no position: zero output, lse -inf
    o, lse = attention.attend_dense(q, np.zeros((0, d)), np.zeros((0, d)), 0.125)
    assert (o == 0).all() and lse == -math.inf


def test_all_hole_sequence_and_empty_context():
    rng = np.random.default_rng(8)
    kp, vp, table = _paged_layout(rng, [40, 5], 16, 8, 64, "f32", 1, 64)
    table[0, :] = -1
    q = rng.standard_normal((3, 2, 64)).astype(np.float32)
    table = np.vstack([table, np.full((1, table.shape[1]), -1, np.int32)])
    out, lse = attention.paged_attn_decode("f32", q, kp, vp, table, np.array([40, 5, 0]), None,
                                           2, 1, 64, 16, 0.125)
    assert (out[0] == 0).all() and (lse[0] == -np.inf).all()
    assert (out[2] == 0).all() and (lse[2] == -np.inf).all()
    assert np.isfinite(out[1]).all()


def test_store_writes_resolved_cells_only():
    rng = np.random.default_rng(9)
    kp = np.zeros((32, 68), dtype=np.uint8)
    vp = np.zeros((32, 68), dtype=np.uint8)
    rows = rng.standard_normal((3, 64)).astype(np.float32)
    attention.kv_store("q8_0", kp, vp, rows, -rows, np.array([5, -1, 17]), 2, 32)
    touched = sorted(set(np.nonzero(kp.any(1))[0].tolist()))
    assert touched == [5, 17]
    assert np.array_equal(kp[5], formats.encode_rows("q8_0", rows[:1], 2, 32)[0])
    assert np.array_equal(vp[17], formats.encode_rows("q8_0", -rows[2:3], 2, 32)[0])
