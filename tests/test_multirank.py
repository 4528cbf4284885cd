"""The N > 1 bench path on CPU: two gloo ranks, each with its own copy of the workload
(weak scaling), aggregate the timing the way bench.py does."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        ms_local = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(ms_local, world)
        val = bench.whole_job_tflops(1.0e12, world, ms)
        q.put((rank, ms, val))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_and_weak_scaling():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, ms, val in res:
        assert ms == 5.0                       # the slowest rank's time, seen by every rank
        assert abs(val - 2 * 1.0e12 / 5e-3 / 1e12) < 1e-9   # both ranks' work / that time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(4.2, 1) == 4.2
    assert abs(bench.whole_job_tflops(2e12, 1, 1.0) - 2000.0) < 1e-9
