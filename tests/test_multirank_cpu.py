"""The benchmark's multi-rank path on CPU: two gloo ranks (replicas) agree on the
slowest rank's step time and report the whole-job value."""
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
        t = bench.reduce_step_time(0.001 * (rank + 1), dist, torch.device("cpu"))
        out[rank] = t
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(0.002) and out[1] == pytest.approx(0.002)
    import bench
    assert bench.job_value(2, 0.002) == pytest.approx(2 * bench.STEP_FLOPS / 0.002 / 1e12)
    assert bench.reduce_step_time(0.5, None, None) == 0.5
