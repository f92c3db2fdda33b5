"""The multi-rank bench path on CPU: two gloo ranks, weak scaling, max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                     # rank 1 is the slowest
    m = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    dist.barrier()
    q.put((rank, m, bench.whole_job_rate(world, 128, m / 4)))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_ranks_take_the_slowest_time(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, rate in res:
        assert m == 15.0
        assert rate == pytest.approx(world * 128 / (15.0 / 4 * 1e-3))


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.whole_job_rate(1, 128, 1.0) == 128_000
