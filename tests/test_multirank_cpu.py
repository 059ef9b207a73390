"""The N > 1 benchmark path on CPU: two gloo ranks, each timing its own replica
of the workload; the job's time is the slowest rank's and the throughput counts
every rank's bytes (weak scaling, no data-path collective)."""

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


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = 10.0 + 5.0 * rank              # rank 1 is the slow one
    mx = bench.max_over_ranks(my_ms, world)
    val = bench.job_throughput_gbs(1_000_000_000, 4, mx, world)
    results[rank] = (mx, val)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 1 GB x 4 steps in 15 ms
    assert abs(res[0][1] - 2 * 1.0 * 4 / 0.015) < 1e-6


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.job_throughput_gbs(2_000_000_000, 10, 20.0, 1) - 1000.0) < 1e-9
