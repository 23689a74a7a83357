"""Pins of the oracle's multi-query (prefill) attention and set-valued
(kv_map) windows (CPU only).

Fixed outside the oracle:
  * torch's scaled_dot_product_attention (float64, CPU), a library routine,
    with an explicit boolean mask: full causal prefill (is_causal), chunked
    prefill (the queries are the last n positions: query j sees t <= ctx-n+j),
    and kv_map runs (mask = union of the runs);
  * special cases that reduce to the decode oracle, itself pinned to SDPA:
    one query per sequence; a single run (lo, hi - lo) equals the pair
    [lo, hi) ("KV Cache Design — cells, format, sessions", section 1);
  * brute force on tiny inputs with plain Python loops and math.exp;
  * invariants of the block model ("Tiered KV cache — architecture", section
    "The paged-attention block model"): holes equal deletion, physical
    placement does not matter;
  * empty windows: output 0, lse -infinity.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, formats


def _layout(rng, lens, bs, fmt, hkv, d, extra_blocks=3):
    """Shuffled paged layout of `lens` sequences; returns pools, table, the
    number of physical blocks."""
    nb = [-(-c // bs) for c in lens]
    n_phys = sum(nb) + extra_blocks
    perm = rng.permutation(n_phys)
    table = np.full((len(lens), max(nb)), -1, dtype=np.int32)
    nxt = 0
    for s, n in enumerate(nb):
        table[s, :n] = perm[nxt:nxt + n]
        nxt += n
    k = rng.standard_normal((n_phys * bs, hkv * d)).astype(np.float32)
    v = rng.standard_normal((n_phys * bs, hkv * d)).astype(np.float32)
    return formats.encode_rows(fmt, k, hkv, d), formats.encode_rows(fmt, v, hkv, d), table


def _dense(kp, vp, row, ctx, bs, fmt, hkv, d):
    cells = [row[p // bs] * bs + p % bs for p in range(ctx)]
    k = formats.decode_rows(fmt, kp[cells], hkv, d).reshape(ctx, hkv, d)
    v = formats.decode_rows(fmt, vp[cells], hkv, d).reshape(ctx, hkv, d)
    return k, v


def _sdpa_masked(q, k, v, scale, G, mask):
    """q [n][Hq][d], k/v [ctx][Hkv][d], mask [n][ctx] bool -> [n][Hq][d]."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    m = torch.from_numpy(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("fmt,hq,hkv,d,bs", [("f32", 4, 2, 64, 16), ("f16", 8, 2, 32, 16),
                                             ("q8_0", 6, 3, 64, 32), ("f32", 3, 3, 32, 16)])
def test_chunked_prefill_matches_library_sdpa(fmt, hq, hkv, d, bs):
    rng = np.random.default_rng(40)
    lens = [50, 37, 70]
    n_q = [50, 5, 17]  # a full prefill, then two chunks at the end of the context
    kp, vp, table = _layout(rng, lens, bs, fmt, hkv, d)
    q_start = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
    q = rng.standard_normal((q_start[-1], hq, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    out, lse = attention.paged_attn_prefill(fmt, q, kp, vp, table, np.array(lens), q_start,
                                            None, None, hq, hkv, d, bs, scale)
    for s, c in enumerate(lens):
        n = n_q[s]
        k, v = _dense(kp, vp, table[s], c, bs, fmt, hkv, d)
        j = np.arange(n)[:, None]
        t = np.arange(c)[None, :]
        mask = t <= c - n + j
        want = _sdpa_masked(q[q_start[s]:q_start[s + 1]], k, v, scale, hq // hkv, mask)
        assert np.allclose(out[q_start[s]:q_start[s + 1]], want, rtol=0, atol=1e-12)
        if n == c:  # a full prefill is the library's own causal attention
            qt = torch.from_numpy(q[q_start[s]:q_start[s + 1]].astype(np.float64)).permute(
                1, 0, 2)[None]
            kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)[None]
            vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)[None]
            o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                                 scale=scale)
            assert np.allclose(out[q_start[s]:q_start[s + 1]], o[0].permute(1, 0, 2).numpy(),
                               rtol=0, atol=1e-12)


def test_one_query_per_sequence_is_the_decode():
    rng = np.random.default_rng(41)
    lens = [40, 17, 64, 1]
    hq, hkv, d, bs = 4, 2, 32, 16
    kp, vp, table = _layout(rng, lens, bs, "f16", hkv, d)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float32)
    spans = np.array([[3, 30], [0, 17], [60, 64], [0, 0]], dtype=np.int32)
    q_start = np.arange(len(lens) + 1, dtype=np.int32)
    scale = 0.17
    out, lse = attention.paged_attn_prefill("f16", q, kp, vp, table, np.array(lens), q_start,
                                            spans, None, hq, hkv, d, bs, scale)
    want, want_lse = attention.paged_attn_decode("f16", q, kp, vp, table, np.array(lens), spans,
                                                 hq, hkv, d, bs, scale)
    assert np.array_equal(out, want) and np.array_equal(lse, want_lse)


def test_prefill_brute_force_with_holes_and_windows():
    rng = np.random.default_rng(42)
    bs, hq, hkv, d = 4, 2, 1, 3
    lens = [11, 6]
    n_q = [3, 6]
    kp, vp, table = _layout(rng, lens, bs, "f32", hkv, d)
    table[0, 1] = -1  # positions 4..7 of sequence 0 are a hole
    q_start = np.array([0, 3, 9], dtype=np.int32)
    q = rng.standard_normal((9, hq, d)).astype(np.float32)
    spans = np.array([[0, 11], [2, 9], [5, 6], [0, 6], [1, 3], [2, 2], [0, 6], [4, 5], [3, 6]],
                     dtype=np.int32)
    scale = 0.5
    out, lse = attention.paged_attn_prefill("f32", q, kp, vp, table, np.array(lens), q_start,
                                            spans, None, hq, hkv, d, bs, scale)
    kf = formats.decode_rows("f32", kp, hkv, d)
    vf = formats.decode_rows("f32", vp, hkv, d)
    for s in range(2):
        for j in range(n_q[s]):
            i = q_start[s] + j
            pos = lens[s] - n_q[s] + j
            for h in range(hq):
                logits, rows = [], []
                for t in range(lens[s]):
                    blk = table[s, t // bs]
                    if t > pos or blk < 0 or not spans[i][0] <= t < spans[i][1]:
                        continue
                    cell = blk * bs + t % bs
                    logits.append(scale * sum(float(q[i, h, e]) * float(kf[cell, e])
                                              for e in range(d)))
                    rows.append(cell)
                if not logits:
                    assert np.all(out[i, h] == 0) and lse[i, h] == -math.inf
                    continue
                m = max(logits)
                w = [math.exp(x - m) for x in logits]
                z = sum(w)
                for e in range(d):
                    o = sum(w[r] * float(vf[rows[r], e]) for r in range(len(rows))) / z
                    assert out[i, h, e] == pytest.approx(o, abs=1e-12)
                assert lse[i, h] == pytest.approx(m + math.log(z), abs=1e-12)


def test_kv_map_single_run_is_the_pair_and_union_matches_sdpa():
    rng = np.random.default_rng(43)
    lens = [90, 33]
    hq, hkv, d, bs = 4, 2, 32, 16
    kp, vp, table = _layout(rng, lens, bs, "q8_0", hkv, d)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    scale = 0.2
    # a single run equals the [lo, hi) pair
    spans = np.array([[7, 61], [0, 20]], dtype=np.int32)
    runs = np.zeros((2, 8, 2), dtype=np.int32)
    runs[:, 0, 0] = spans[:, 0]
    runs[:, 0, 1] = spans[:, 1] - spans[:, 0]
    o1, l1 = attention.paged_attn_decode_map("q8_0", q, kp, vp, table, np.array(lens), runs,
                                             hq, hkv, d, bs, scale)
    o2, l2 = attention.paged_attn_decode("q8_0", q, kp, vp, table, np.array(lens), spans,
                                         hq, hkv, d, bs, scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # overlapping and out-of-range runs: the union within [0, ctx)
    runs = np.zeros((2, 8, 2), dtype=np.int32)
    runs[0, :4] = [[0, 16], [10, 12], [70, 40], [-5, 2]]  # {0..21} U {70..89}
    runs[1, :2] = [[30, 3], [5, 0]]                        # {30, 31, 32}
    out, lse = attention.paged_attn_decode_map("q8_0", q, kp, vp, table, np.array(lens), runs,
                                               hq, hkv, d, bs, scale)
    for s, c in enumerate(lens):
        k, v = _dense(kp, vp, table[s], c, bs, "q8_0", hkv, d)
        mask = np.zeros((1, c), dtype=bool)
        if s == 0:
            mask[0, :22] = True
            mask[0, 70:90] = True
        else:
            mask[0, 30:33] = True
        want = _sdpa_masked(q[s][None], k, v, scale, hq // hkv, mask)[0]
        assert np.allclose(out[s], want, rtol=0, atol=1e-12)


def test_empty_windows_and_holes_as_deletion():
    rng = np.random.default_rng(44)
    lens = [40]
    hq, hkv, d, bs = 2, 1, 16, 8
    kp, vp, table = _layout(rng, lens, bs, "f32", hkv, d)
    q = rng.standard_normal((1, hq, d)).astype(np.float32)
    runs = np.zeros((1, 8, 2), dtype=np.int32)  # no run: nothing to read
    out, lse = attention.paged_attn_decode_map("f32", q, kp, vp, table, np.array(lens), runs,
                                               hq, hkv, d, bs, 1.0)
    assert np.all(out == 0) and np.all(lse == -math.inf)
    # a hole inside a run: same as a map that skips the hole's positions
    t2 = table.copy()
    t2[0, 2] = -1
    runs[0, 0] = (0, 40)
    a, la = attention.paged_attn_decode_map("f32", q, kp, vp, t2, np.array(lens), runs,
                                            hq, hkv, d, bs, 1.0)
    runs2 = np.zeros((1, 8, 2), dtype=np.int32)
    runs2[0, :2] = [(0, 16), (24, 16)]
    b, lb = attention.paged_attn_decode_map("f32", q, kp, vp, table, np.array(lens), runs2,
                                            hq, hkv, d, bs, 1.0)
    assert np.allclose(a, b, rtol=0, atol=1e-13) and np.allclose(la, lb, rtol=0, atol=1e-13)
