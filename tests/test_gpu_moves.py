"""GPU parity of the ordered row mover (copy_cells) and the grow-on-demand
re-layout against the oracle: both bit-exact."""
import numpy as np
import pytest
import torch

from oracle import moves as om
from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


@pytest.mark.parametrize("row_bytes", [768, 68, 1088])
def test_compaction_moves_bit_exact(mt, row_bytes):
    moves, n_cells = workloads.compaction_moves(seed=40 + row_bytes, n_runs=150)
    ordered = mt.mt_order_moves(moves)
    assert ordered == om.order_moves(moves)
    rng = np.random.default_rng(41)
    pools = [rng.integers(0, 256, (n_cells, row_bytes), dtype=np.uint8) for _ in range(5)]
    devs = [to_dev(p) for p in pools]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.mt_copy_cells(devs, row_bytes, n_cells, ordered, status=status)
    om.copy_cells(pools, ordered)
    # a normal call (staged runs for 16-byte rows) leaves the status word clear
    assert mt.mt_check_device_status(status) == mt.MT_OK
    for p, d in zip(pools, devs):
        assert np.array_equal(d.cpu().numpy(), p)


def test_dependent_moves_and_shared_sources(mt):
    # a compaction whose moves depend on each other (must run in order), one
    # move read by several later copies (copy-on-write fan-out), and
    # single-row shifts (a chunk per row)
    rb, n_cells = 48, 200
    moves = [(20, 10, 5), (10, 5, 5), (40, 41, 30), (100, 150, 4), (100, 160, 4),
             (100, 170, 4), (120, 119, 25)]
    ordered = om.order_moves(moves)
    assert om.find_hazard(ordered) is None
    assert mt.mt_order_moves(moves) == ordered
    rng = np.random.default_rng(42)
    pools = [rng.integers(0, 256, (n_cells, rb), dtype=np.uint8) for _ in range(3)]
    devs = [to_dev(p) for p in pools]
    mt.mt_copy_cells(devs, rb, n_cells, ordered)
    om.copy_cells(pools, ordered)
    for p, d in zip(pools, devs):
        assert np.array_equal(d.cpu().numpy(), p)


def test_hazardous_list_is_rejected_before_launch(mt):
    dev = torch.arange(64 * 16, dtype=torch.int32, device="cuda").view(torch.uint8).reshape(64, -1)
    before = dev.clone()
    with pytest.raises(mt.MtError) as e:
        mt.mt_copy_cells([dev], 64, 64, [(20, 10, 5), (10, 5, 5)])
    assert e.value.status == mt.MT_ERR_ORDER
    torch.cuda.synchronize()
    assert torch.equal(dev, before)


def test_grow_on_demand_relayout_bit_exact(mt):
    L, rb, max_ctx = 3, 192 * 4, 1000
    rng = np.random.default_rng(43)
    rows = rng.integers(0, 256, (L, max_ctx, rb), dtype=np.uint8)
    cap = om.initial_capacity(max_ctx)
    host = np.zeros((L * cap, rb), np.uint8)
    dev = torch.zeros(L * cap, rb, dtype=torch.uint8, device="cuda")
    for pos in range(max_ctx):
        if pos >= cap:
            nc = mt.mt_kv_grow_capacity(cap, pos + 1, max_ctx)
            assert nc == om.grow_capacity(cap, pos + 1, max_ctx)
            new = torch.empty(L * nc, rb, dtype=torch.uint8, device="cuda")
            mt.mt_kv_relayout(dev, new, L, cap, nc, rb)
            host = om.kv_relayout(host, L, cap, nc)
            dev, cap = new, nc
        for l in range(L):
            host[l * cap + pos] = rows[l, pos]
        dev.view(L, cap, rb)[:, pos] = to_dev(rows[:, pos])
    got = dev.view(L, cap, rb)[:, :max_ctx].cpu().numpy()
    assert np.array_equal(got, host.reshape(L, cap, rb)[:, :max_ctx])
    assert np.array_equal(got, rows)  # identical to a store preallocated at max_ctx


def test_relayout_word_rows(mt):
    L, rb = 4, 36  # q8_0 row of one 32-dim head: 4-byte words, not 16-byte
    src = torch.randint(0, 256, (L * 50, rb), dtype=torch.uint8, device="cuda")
    dst = torch.zeros(L * 128, rb, dtype=torch.uint8, device="cuda")
    mt.mt_kv_relayout(src, dst, L, 50, 128, rb)
    assert torch.equal(dst.view(L, 128, rb)[:, :50], src.view(L, 50, rb))
    assert int(dst.view(L, 128, rb)[:, 50:].sum()) == 0
