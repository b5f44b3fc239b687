"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own
replica; the job's time is the slowest rank's and the value counts both."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.slowest_rank_ms([2.0, 5.0][rank], dist, torch.device("cpu"))
    q.put((rank, ms, bench.job_throughput(world, 1 << 27, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    assert res[0][2] == pytest.approx(2 * (1 << 27) / 5e-3 / 1e9)


def test_single_rank_needs_no_group():
    import bench
    assert bench.slowest_rank_ms(3.5) == 3.5
    assert bench.job_throughput(1, 1000, 1.0) == pytest.approx(1e-3)
