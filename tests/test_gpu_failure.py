"""Failure detection without faulting the GPU.

Every pipeline wait in libmtkv is bounded: when it runs out it records
MT_STATUS_BIT_TIMEOUT in a status word and the kernel returns. These tests
make a wait run out on purpose (a barrier nothing completes, short limit),
read the status back on the host, and check the context still works; they
also check that bad inputs are turned into statuses on the host or in the
kernels rather than faults.
"""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_gqa_gb300 import workloads
from tests.gpu_util import TOL, assert_close, gpu_decode, oracle_decode, oracle_pools, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_gqa_gb300 import mtkv
    return mtkv


def test_bounded_wait_times_out_and_reports(mt):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    mt.mt_selftest_bounded_wait(10_000_000, status)  # 10 ms
    st = mt.mt_check_device_status(status)
    dt = time.perf_counter() - t0
    assert st == mt.MT_ERR_TIMEOUT
    assert dt < 1.5
    # the status word was cleared and the context is usable
    assert mt.mt_check_device_status(status) == mt.MT_OK
    w = workloads.tiny_f32()
    kp, vp = oracle_pools(w)
    want, _ = oracle_decode(w, kp, vp)
    got, _, st = gpu_decode(mt, w, to_dev(kp), to_dev(vp))
    assert st == mt.MT_OK
    assert_close(got, want, TOL["f32"], "after timeout")


def test_bad_arguments_are_refused_before_launch(mt):
    w = workloads.llama3_f16(seed=70, n_seqs=2, ctx_lo=20, ctx_hi=40)
    kp, vp = oracle_pools(w)
    q = to_dev(w.q)
    out = torch.empty_like(q)
    args = mt.paged_attn_args("f16", q, to_dev(kp), to_dev(vp), to_dev(w.block_table),
                              to_dev(w.context_lens), out, n_kv_heads=w.n_kv_heads,
                              block_size=w.block_size, n_phys_blocks=w.n_phys_blocks,
                              scale=w.scale)
    need = mt.mt_paged_attn_workspace_bytes(args)
    small = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(mt.MtError) as e:
        mt.mt_paged_attn_decode(args, small)
    assert e.value.status == mt.MT_ERR_INVALID_ARG and "workspace" in str(e.value)
    args.fmt = 7
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(mt.MtError) as e:
        mt.mt_paged_attn_decode(args, ws)
    assert e.value.status == mt.MT_ERR_INVALID_ARG
    args.fmt = 1
    args.block_size = 8
    with pytest.raises(mt.MtError) as e:
        mt.mt_paged_attn_decode(args, ws)
    assert e.value.status == mt.MT_ERR_UNSUPPORTED
    torch.cuda.synchronize()
