"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times.

At these sizes the float64 oracle cannot check every (sequence, head) of a
decode call in seconds, so each decode test runs the whole call on the GPU
and compares a seeded sample of sequences — always including the longest
and the shortest — with all their heads (f32 KV 1e-4, f16 and q8_0 2e-3);
where the oracle is cheap enough (SmolLM2-shaped f32, the q8_0 shared
prefix) every sequence is compared; the chunked prefill call compares a
seeded sample of its query rows. Everything whose result must be
bit-exact is compared in full: the stored rows (the whole pools after the
call, so nothing else was written), the int4 scales, nibbles and
dequantised blocks of every cold block, the 60 pools after the 1000-move
compaction and the 30-layer buffer after the 64 -> 8192 grow.

Pool contents are seeded N(0,1) values drawn by torch's generator on the
device (f32/f16) or stored by the oracle's q8_0 quantiser on the host:
inputs, never results of this library. The oracle reads a host copy.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import formats as ofmt
from oracle import moves as om
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, assert_lse, oracle_decode, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _randn_pools(w, g, dtype):
    row = w.n_kv_heads * w.head_dim
    return tuple(torch.randn(w.n_cells, row, generator=g, device="cuda", dtype=dtype)
                 for _ in range(2))


def _host_bytes(t):
    """uint8 [rows][row bytes] host copy of a device pool."""
    return t.cpu().numpy().view(np.uint8).reshape(t.shape[0], -1)


def _sample(w, n, seed):
    lens = w.context_lens
    rng = np.random.default_rng(seed)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    pick.update(int(s) for s in rng.choice(w.n_seqs, size=min(n, w.n_seqs), replace=False))
    return sorted(pick)


def _args(mt, w, k_dev, v_dev, table=None, lse=False):
    q = to_dev(w.q)
    out = torch.full_like(q, float("nan"))
    lse_t = torch.full((w.n_seqs, w.n_heads), float("nan"), device="cuda") if lse else None
    sp = None if w.spans is None else to_dev(w.spans)
    args = mt.paged_attn_args(w.fmt, q, k_dev, v_dev,
                              to_dev(w.block_table if table is None else table),
                              to_dev(w.context_lens), out, n_kv_heads=w.n_kv_heads,
                              block_size=w.block_size, n_phys_blocks=w.n_phys_blocks,
                              scale=w.scale, spans=sp, lse=lse_t)
    return args, out, lse_t


def _check(w, got, want, seqs, what, got_lse=None, want_lse=None):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert_close(got[seqs], want[seqs], TOL[w.fmt], what)
    if got_lse is not None:
        assert_lse(got_lse[seqs], want_lse[seqs], TOL[w.fmt], what)


def _fused_step(mt, w, seed, n_sample):
    """One layer of the decode step as the benchmark runs it: the new rows
    stored inside the decode launch (mt_paged_attn_decode_append), default
    grid, workspace from mt_paged_attn_workspace_bytes."""
    dtype = torch.float32 if w.fmt == "f32" else torch.float16
    k_dev, v_dev = _randn_pools(w, _gen(seed), dtype)
    kp, vp = _host_bytes(k_dev), _host_bytes(v_dev)
    args, out, _ = _args(mt, w, k_dev, v_dev)
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args), dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_decode_append(args, to_dev(w.k_new), to_dev(w.v_new), ws)
    assert mt.mt_check_device_status(ws) == 0, mt.mt_last_error()
    oatt.kv_store(w.fmt, kp, vp, w.k_new, w.v_new, w.new_cells, w.n_kv_heads, w.head_dim)
    # the new rows are bit-exact and no other cell was written
    assert np.array_equal(_host_bytes(k_dev), kp)
    assert np.array_equal(_host_bytes(v_dev), vp)
    seqs = list(range(w.n_seqs)) if n_sample is None else _sample(w, n_sample, seed)
    want, _ = oracle_decode(w, kp, vp, seqs=seqs)
    _check(w, out.cpu().numpy(), want, seqs, f"{w.name} full size")


def test_full_llama3_f16_step(mt):
    # 64 sequences, context log-uniform in [512, 16384], 32/8 heads, d 128,
    # bs 16, pool 1.1x the blocks needed
    w = workloads.llama3_f16(hist=False)
    assert w.n_seqs == 64 and w.context_lens.max() > 8192
    _fused_step(mt, w, 3001, 6)


def test_full_smollm2_f32_step(mt):
    # 8 sequences, context uniform in [2048, 8192], 9/3 heads, d 64: every
    # sequence is checked
    w = workloads.smollm2_f32(hist=False)
    _fused_step(mt, w, 3002, None)


@pytest.mark.parametrize("bs", [16, 32])
def test_full_llama3_q8_0_decode(mt, bs):
    # the Llama-3-shaped batch (64 sequences, context log-uniform in
    # [512, 16384], 32/8 heads, d 128) with q8_0 pools, one decode call in the
    # launch configuration the per-format benchmark times (default grid,
    # paired 16-row blocks at block size 16). The sampled sequences' blocks
    # hold N(0,1) rows stored by the oracle's quantiser; the other blocks are
    # zero (scale 0, codes 0: valid q8_0 cells)
    w = workloads.llama3_f16(fmt="q8_0", block_size=bs, hist=False)
    seqs = _sample(w, 4, 3010 + bs)
    rb = ofmt.row_bytes("q8_0", w.n_kv_heads, w.head_dim)
    kp = np.zeros((w.n_cells, rb), np.uint8)
    vp = np.zeros((w.n_cells, rb), np.uint8)
    rng = np.random.default_rng(3011 + bs)
    row = w.n_kv_heads * w.head_dim
    for s in seqs:
        nb = -(-int(w.context_lens[s]) // bs)
        cells = (w.block_table[s, :nb].astype(np.int64)[:, None] * bs + np.arange(bs)).reshape(-1)
        x = rng.standard_normal((2, nb * bs, row), dtype=np.float32)
        kp[cells] = ofmt.encode_rows("q8_0", x[0], w.n_kv_heads, w.head_dim)
        vp[cells] = ofmt.encode_rows("q8_0", x[1], w.n_kv_heads, w.head_dim)
    args, out, lse = _args(mt, w, to_dev(kp), to_dev(vp), lse=True)
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args), dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_decode(args, ws)
    assert mt.mt_check_device_status(ws) == 0, mt.mt_last_error()
    want, want_lse = oracle_decode(w, kp, vp, seqs=seqs)
    _check(w, out.cpu().numpy(), want, seqs, f"q8_0 bs {bs} full size", lse.cpu().numpy(),
           want_lse)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "f32"])
def test_full_llama3_prefill(mt, fmt):
    # the chunked-prefill benchmark's call: 16 sequences at context 2048 whose
    # last 512 positions are queries (8192 query rows), 32/8 heads, d 128,
    # bs 16, in its launch configuration (f16 pools directly, q8_0 and f32
    # through their staging passes). A seeded sample of query rows of four
    # sequences (always each one's first and last query) is checked with all
    # heads: sampled row j of sequence s is the oracle's one-query sequence
    # at context ctx - n + j + 1 over the same blocks
    n_q = 512
    w = workloads.llama3_f16(seed=3020, n_seqs=16, ctx_lo=2048, ctx_hi=2048, hist=False, fmt=fmt)
    g = _gen(3021)
    rng = np.random.default_rng(3023)
    seqs = sorted({0, w.n_seqs - 1} | set(rng.choice(w.n_seqs, 2, replace=False).tolist()))
    if fmt == "q8_0":
        # the sampled sequences' blocks hold N(0,1) rows stored by the
        # oracle's quantiser; the other blocks are zero (valid q8_0 cells)
        rb = ofmt.row_bytes("q8_0", w.n_kv_heads, w.head_dim)
        kp = np.zeros((w.n_cells, rb), np.uint8)
        vp = np.zeros((w.n_cells, rb), np.uint8)
        xr = np.random.default_rng(3022)
        bs = w.block_size
        for s in seqs:
            nb = -(-int(w.context_lens[s]) // bs)
            cells = (w.block_table[s, :nb].astype(np.int64)[:, None] * bs
                     + np.arange(bs)).reshape(-1)
            x = xr.standard_normal((2, nb * bs, w.n_kv_heads * w.head_dim), dtype=np.float32)
            kp[cells] = ofmt.encode_rows("q8_0", x[0], w.n_kv_heads, w.head_dim)
            vp[cells] = ofmt.encode_rows("q8_0", x[1], w.n_kv_heads, w.head_dim)
        k_dev, v_dev = to_dev(kp), to_dev(vp)
    else:
        k_dev, v_dev = _randn_pools(w, g, torch.float32 if fmt == "f32" else torch.float16)
        kp, vp = _host_bytes(k_dev), _host_bytes(v_dev)
    q = torch.randn(n_q * w.n_seqs, w.n_heads, w.head_dim, generator=g, device="cuda")
    q_start = torch.arange(0, n_q * w.n_seqs + 1, n_q, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], w.n_heads), float("nan"), device="cuda")
    a = mt.prefill_args(fmt, q, k_dev, v_dev, to_dev(w.block_table), to_dev(w.context_lens),
                        q_start, out, n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                        n_phys_blocks=w.n_phys_blocks, scale=w.scale, lse=lse)
    ws = torch.zeros(mt.mt_paged_prefill_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_prefill(a, ws)
    assert mt.mt_check_device_status(ws) == 0, mt.mt_last_error()
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(got).all(), f"{fmt} prefill full size: non-finite output"
    rows, ctx_sub, tab_sub = [], [], []
    for s in seqs:
        c = int(w.context_lens[s])
        for j in sorted({0, n_q - 1} | set(rng.choice(n_q, 4, replace=False).tolist())):
            rows.append(s * n_q + j)
            ctx_sub.append(c - n_q + j + 1)
            tab_sub.append(w.block_table[s])
    q_sub = q.cpu().numpy()[rows]
    want, want_lse = oatt.paged_attn_prefill(
        fmt, q_sub, kp, vp, np.stack(tab_sub), np.array(ctx_sub, np.int32),
        np.arange(len(rows) + 1, dtype=np.int32), None, None, w.n_heads, w.n_kv_heads,
        w.head_dim, w.block_size, w.scale)
    assert_close(got[rows], want, TOL[fmt], f"{fmt} prefill full size")
    assert_lse(got_lse[rows], want_lse, TOL[fmt], f"{fmt} prefill full size")


@pytest.mark.parametrize("prefix", ["cascade", "plain"])
def test_full_q8_prefix_windows(mt, prefix):
    # 32 sequences sharing a 4096-token prefix (refcount 32) plus private
    # suffixes U[64, 1024], random windows, bs 32; the store runs as its own
    # launch and the decode reads the prefix once per group (cascade) or per
    # sequence (plain); every sequence is checked
    w = workloads.llama3_q8_prefix()
    kp = ofmt.encode_rows("q8_0", w.k_hist, w.n_kv_heads, w.head_dim)
    vp = ofmt.encode_rows("q8_0", w.v_hist, w.n_kv_heads, w.head_dim)
    k_dev, v_dev = to_dev(kp), to_dev(vp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.mt_kv_store("q8_0", k_dev, v_dev, w.n_kv_heads, w.head_dim, to_dev(w.k_new),
                   to_dev(w.v_new), to_dev(w.new_cells), status=status)
    assert mt.mt_check_device_status(status) == 0, mt.mt_last_error()
    oatt.kv_store("q8_0", kp, vp, w.k_new, w.v_new, w.new_cells, w.n_kv_heads, w.head_dim)
    assert np.array_equal(_host_bytes(k_dev), kp) and np.array_equal(_host_bytes(v_dev), vp)
    args, out, lse = _args(mt, w, k_dev, v_dev, lse=True)
    if prefix == "cascade":
        groups = [(0, w.n_seqs, w.extra["prefix"] // w.block_size)]
        ws = torch.zeros(mt.mt_paged_attn_cascade_workspace_bytes(args, groups),
                         dtype=torch.uint8, device="cuda")
        mt.mt_paged_attn_decode_cascade(args, groups, ws)
    else:
        ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args), dtype=torch.uint8,
                         device="cuda")
        mt.mt_paged_attn_decode(args, ws)
    assert mt.mt_check_device_status(ws) == 0, mt.mt_last_error()
    seqs = list(range(w.n_seqs))
    want, want_lse = oracle_decode(w, kp, vp)
    got_lse = lse.cpu().numpy()
    _check(w, out.cpu().numpy(), want, seqs, f"q8_0 prefix {prefix}", got_lse, want_lse)


def test_full_longctx_int4_round_trip(mt):
    # 16 sequences x 32768, 16/4 heads, d 256, bs 16, 5 % holes; 25 % of the
    # other blocks go through int4 (K and V separately) into fresh ids from a
    # 1.3x pool. Every cold block's scale, nibbles and dequantised rows are
    # compared bit for bit; the decode over the retargeted table is compared
    # on a sample of sequences.
    w = workloads.longctx_f16_int4(hist=False)
    hkv, d, bs = w.n_kv_heads, w.head_dim, w.block_size
    n_el = bs * hkv * d
    src, dst = w.extra["cold_src"], w.extra["cold_dst"]
    assert len(src) > 7000
    k_dev, v_dev = _randn_pools(w, _gen(3005), torch.float16)
    kp, vp = _host_bytes(k_dev), _host_bytes(v_dev)
    src_d, dst_d = to_dev(src), to_dev(dst)
    for pool_host, pool_dev in ((kp, k_dev), (vp, v_dev)):
        scales = torch.empty(len(src), dtype=torch.float32, device="cuda")
        nib = torch.empty(len(src), n_el // 2, dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        mt.mt_kv_quant_int4("f16", pool_dev, bs, hkv, d, w.n_phys_blocks, src_d, scales, nib,
                            status=status)
        mt.mt_kv_dequant_int4("f16", pool_dev, bs, hkv, d, w.n_phys_blocks, dst_d, scales, nib,
                              status=status)
        assert mt.mt_check_device_status(status) == 0, mt.mt_last_error()
        g_scales, g_nib = scales.cpu().numpy(), nib.cpu().numpy()
        want_scales = np.empty(len(src), dtype=np.float32)
        for i, (b_src, b_dst) in enumerate(zip(src, dst)):
            s, n = ofmt.int4_quantize_block(pool_host[b_src * bs:(b_src + 1) * bs].view(np.float16))
            want_scales[i] = s
            assert np.array_equal(g_nib[i], n), f"nibbles of cold block {i}"
            back = ofmt.int4_dequantize_block(s, n, n_el, "f16")
            pool_host[b_dst * bs:(b_dst + 1) * bs] = back.view(np.uint8).reshape(bs, -1)
        assert np.array_equal(g_scales.view(np.uint32), want_scales.view(np.uint32))
        assert np.array_equal(_host_bytes(pool_dev), pool_host)
    table = workloads.retarget_cold(w)
    args, out, lse = _args(mt, w, k_dev, v_dev, table=table, lse=True)
    ws = torch.zeros(mt.mt_paged_attn_workspace_bytes(args), dtype=torch.uint8, device="cuda")
    mt.mt_paged_attn_decode(args, ws)
    assert mt.mt_check_device_status(ws) == 0, mt.mt_last_error()
    seqs = _sample(w, 3, 3005)
    want, want_lse = oracle_decode(w, kp, vp, table=table, seqs=seqs)
    _check(w, out.cpu().numpy(), want, seqs, "long-context int4", lse.cpu().numpy(), want_lse)


def test_full_compaction_60_pools(mt):
    # 1000 overlapping run moves ordered by order_moves, applied to 60 pools
    # (30 layers x K and V) of 768-byte rows in one call
    moves, n_cells = workloads.compaction_moves()
    assert len(moves) == 1000
    ordered = mt.mt_order_moves(moves)
    assert ordered == om.order_moves(moves) and om.find_hazard(ordered) is None
    g = _gen(3006)
    devs = [torch.randint(0, 256, (n_cells, 768), generator=g, device="cuda",
                          dtype=torch.uint8) for _ in range(60)]
    before = [d.cpu().numpy() for d in devs]
    mt.mt_copy_cells(devs, 768, n_cells, ordered)
    for i, (host, dev) in enumerate(zip(before, devs)):
        om.copy_cells([host], ordered)
        assert np.array_equal(dev.cpu().numpy(), host), f"pool {i}"


def test_full_grow_64_to_8192(mt):
    # grow-on-demand from capacity 64 to max_ctx 8192 (seven doublings), 30
    # layers of f32 kv_dim 192 rows; each doubling's new positions are then
    # written, and the final buffer must equal a store preallocated at 8192
    L, rb, max_ctx = 30, 192 * 4, 8192
    g = _gen(3007)
    rows = torch.randint(0, 256, (L, max_ctx, rb), generator=g, device="cuda",
                         dtype=torch.uint8)
    rows_h = rows.cpu().numpy()
    cap = om.initial_capacity(max_ctx)
    dev = rows[:, :cap].reshape(L * cap, rb).clone()
    host = rows_h[:, :cap].reshape(L * cap, rb).copy()
    n_grow = 0
    while cap < max_ctx:
        nc = mt.mt_kv_grow_capacity(cap, cap + 1, max_ctx)
        assert nc == om.grow_capacity(cap, cap + 1, max_ctx) == 2 * cap
        new = torch.empty(L * nc, rb, dtype=torch.uint8, device="cuda")
        mt.mt_kv_relayout(dev, new, L, cap, nc, rb)
        host = om.kv_relayout(host, L, cap, nc)
        assert np.array_equal(new.view(L, nc, rb)[:, :cap].cpu().numpy(),
                              host.reshape(L, nc, rb)[:, :cap])
        new.view(L, nc, rb)[:, cap:] = rows[:, cap:nc]
        host.reshape(L, nc, rb)[:, cap:] = rows_h[:, cap:nc]
        dev, cap = new, nc
        n_grow += 1
    assert n_grow == 7
    assert np.array_equal(dev.view(L, cap, rb).cpu().numpy(), rows_h)
