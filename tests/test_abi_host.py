"""The C-ABI library loads, exports every entry point the header declares,
and its host-side logic agrees with the oracle (no GPU needed).

Host-side entry points tested here: mt_kv_row_bytes, mt_order_moves,
mt_check_moves, mt_kv_grow_capacity, mt_paged_prefill_workspace_bytes, and
the argument checks that run before any launch.
"""
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import formats as ofmt
from oracle import moves as om
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def mt():
    from paged_kv_cache_gqa_gb300 import mtkv
    if not os.path.exists(mtkv.LIB_PATH):
        from paged_kv_cache_gqa_gb300 import build as b
        try:
            b.build()
        except RuntimeError as e:  # pragma: no cover - no toolkit
            pytest.skip(f"cannot build libmtkv here: {e}")
    mtkv.lib()
    return mtkv


def _declared():
    txt = open(os.path.join(ROOT, "include", "mtkv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(mt_[a-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(mt):
    names = _declared()
    assert "mt_paged_attn_decode" in names and len(names) >= 14
    nm = subprocess.run(["nm", "-D", "--defined-only", mt.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r" T (mt_\w+)", nm))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(mt.lib(), n)
    assert set(mt.EXPORTED) <= set(names)


def test_row_bytes_matches_oracle(mt):
    for fmt in ("f32", "f16", "q8_0"):
        for hkv in (1, 2, 3, 8):
            for d in (32, 64, 96, 128, 256):
                assert mt.mt_kv_row_bytes(fmt, hkv, d) == ofmt.row_bytes(fmt, hkv, d)
    assert mt.mt_kv_row_bytes("q8_0", 2, 48) == 0
    assert mt.mt_kv_row_bytes(7, 2, 64) == 0
    assert mt.mt_kv_row_bytes("f16", 0, 64) == 0


def test_order_moves_matches_oracle(mt):
    rng = np.random.default_rng(20)
    for _ in range(200):
        n = int(rng.integers(0, 12))
        ms = [(int(rng.integers(0, 50)), int(rng.integers(0, 50)), int(rng.integers(0, 6)))
              for _ in range(n)]
        assert mt.mt_order_moves(ms) == om.order_moves(ms)


def test_check_moves_matches_oracle(mt):
    rng = np.random.default_rng(21)
    n_hazard = 0
    for _ in range(400):
        n = int(rng.integers(1, 8))
        ms = [(int(rng.integers(0, 40)), int(rng.integers(0, 40)), int(rng.integers(1, 6)))
              for _ in range(n)]
        st, bad = mt.mt_check_moves(ms, 64)
        want = om.find_hazard(ms)
        if want is None:
            assert st == mt.MT_OK and bad == -1
        else:
            n_hazard += 1
            assert st == mt.MT_ERR_ORDER and bad == want
    assert n_hazard > 50
    # runs outside the arena are invalid arguments
    st, bad = mt.mt_check_moves([(0, 5, 3), (60, 10, 8)], 64)
    assert st == mt.MT_ERR_INVALID_ARG and bad == 1


def test_generated_compaction_orders_cleanly(mt):
    from paged_kv_cache_gqa_gb300 import workloads
    ms, n_cells = workloads.compaction_moves(seed=1002)
    ordered = mt.mt_order_moves(ms)
    assert ordered == om.order_moves(ms)
    assert mt.mt_check_moves(ordered, n_cells) == (mt.MT_OK, -1)
    assert len(ordered) == 1000


def test_grow_capacity_matches_oracle(mt):
    for cap, need, mx in [(64, 65, 8192), (64, 300, 8192), (4096, 5000, 6000), (128, 100, 8192),
                          (1, 1 << 20, 1 << 30), (64, 8192, 8192)]:
        assert mt.mt_kv_grow_capacity(cap, need, mx) == om.grow_capacity(cap, need, mx)
    assert mt.mt_kv_grow_capacity(0, 5, 10) == -1


def test_host_checks_reject_before_launch(mt):
    # no device memory or GPU is touched: these fail in host validation
    with pytest.raises(mt.MtError) as e:
        mt.lib()
        st = mt.lib().mt_kv_store(9, None, None, 0, 2, 64, None, None, None, 1, None, None)
        mt._check(st, "mt_kv_store")
    assert e.value.status == mt.MT_ERR_INVALID_ARG
    a = mt.mt_paged_attn_args()
    a.fmt, a.n_seqs, a.n_heads, a.n_kv_heads, a.head_dim = 1, 4, 32, 8, 96
    a.block_size, a.max_blocks, a.n_phys_blocks, a.n_ctas = 16, 8, 64, 4
    assert mt.mt_paged_attn_workspace_bytes(a) == 0  # head_dim 96 is not built
    a.head_dim = 128
    assert mt.mt_paged_attn_workspace_bytes(a) > 0
    a.n_heads = 30  # not a multiple of n_kv_heads
    assert mt.mt_paged_attn_workspace_bytes(a) == 0
    a.n_heads, a.block_size = 32, 8
    assert mt.mt_paged_attn_workspace_bytes(a) == 0
    st = mt.lib().mt_kv_relayout(None, None, 2, 8, 4, 64, None)
    assert st == mt.MT_ERR_INVALID_ARG and "old_cap" in mt.mt_last_error()
    st = mt.lib().mt_kv_quant_int4(2, None, 16, 4, 256, 10, None, 1, None, None, None, None)
    assert st == mt.MT_ERR_UNSUPPORTED


def _prefill_ws(mt, fmt, n_seqs, n_tokens, hq, hkv, d, bs, max_blocks):
    a = mt.mt_paged_prefill_args()
    a.fmt = mt._fmt(fmt)
    a.n_seqs, a.n_tokens, a.n_heads, a.n_kv_heads, a.head_dim = n_seqs, n_tokens, hq, hkv, d
    a.block_size, a.max_blocks, a.n_phys_blocks = bs, max_blocks, n_seqs * max_blocks
    return mt.mt_paged_prefill_workspace_bytes(a)


def test_prefill_workspace_holds_the_staged_rows(mt):
    # the header's contract: q8_0 and f32 pools of head_dim 64 / 128 add the
    # staging of the call's blocks, n_seqs x max_blocks x block_size rows of
    # n_kv_heads x head_dim values as f16 (q8_0) or high / low f16 pairs
    # (f32), for K and for V, plus a table of n_seqs x max_blocks ids; f16
    # pools and head_dim 256 stage nothing
    B, mb, bs, hq, hkv = 16, 128, 16, 32, 8
    for d in (64, 128):
        rows = B * mb * bs
        base = _prefill_ws(mt, "f16", B, 8192, hq, hkv, d, bs, mb)
        assert 0 < base <= 4096
        q8 = _prefill_ws(mt, "q8_0", B, 8192, hq, hkv, d, bs, mb)
        f32 = _prefill_ws(mt, "f32", B, 8192, hq, hkv, d, bs, mb)
        need_q8 = 2 * rows * hkv * d * 2 + B * mb * 4
        need_f32 = 2 * rows * hkv * d * 4 + B * mb * 4
        assert need_q8 <= q8 - base < need_q8 + 4096
        assert need_f32 <= f32 - base < need_f32 + 4096
    d256 = [_prefill_ws(mt, f, B, 8192, 16, 4, 256, bs, mb) for f in ("f16", "q8_0")]
    assert d256[0] == d256[1] == base
    # few query rows (fewer tiles than SMs can take): room for the split
    # records, 2 x 160 units of 128 rows x (head_dim + 4) floats
    few = _prefill_ws(mt, "f16", 1, 100, hq, hkv, 128, bs, mb)
    assert few - base >= 2 * 160 * 128 * (128 + 4) * 4
