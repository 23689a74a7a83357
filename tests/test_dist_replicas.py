"""The multi-GPU path of bench.py on CPU: two gloo ranks.

The method has no exchange step, so N GPUs run N independent replicas; the
only cross-rank logic is the barrier, the max over ranks of the measured
time, and the whole-job aggregate. These run here as two processes over the
gloo backend (127.0.0.1)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        # rank r "measured" (r + 1) * 10 ms for 1 GB
        t = bench.max_over_ranks((rank + 1) * 0.010, world)
        out[rank] = (t, bench.whole_job_rate(1e9, t, world))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        t, v = out[r]
        assert t == pytest.approx(0.020)        # max over the two ranks
        assert v == pytest.approx(2 * 1e9 / 0.020 / 1e9)  # both replicas' bytes


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(2e9, 0.5, 1) == pytest.approx(4.0)
    bench.barrier(1)
