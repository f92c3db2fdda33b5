"""Multi-rank host paths on CPU (two gloo ranks): the bench's weak scaling and max over
ranks, and EPLB planning from the loads of all ranks."""
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


def _eplb_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    from combine_moe_route_03_gb300 import api
    rec = api.EplbRecorder(32, 40, period=2, n_group=4, n_nodes=2, n_gpus=4, max_rep=4)
    rng = np.random.default_rng(rank)
    for _ in range(2):
        rec.observe(rng.integers(0, 100 * (rank + 1), 32).astype(np.int32))
    mine = rec.load.copy()
    m, bal = rec.plan(group=dist.group.WORLD)
    q.put((rank, mine, [a.tolist() for a in m], bal))
    dist.destroy_process_group()


def test_eplb_plan_from_all_ranks_loads():
    """Each rank records its own loads; planning sums them across ranks, so both
    ranks install the same map — the oracle's plan of the summed loads."""
    import numpy as np
    from combine_moe_route_03_gb300 import build
    build.build()
    from oracle import eplb as oeplb
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_eplb_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    total = res[0][1] + res[1][1]
    ref, rbal = oeplb.plan(total, 32, 40, 4, 2, 4, 4)
    for _, _, m, bal in res:
        assert m[0] == ref[0] and m[1] == ref[1] and m[2] == ref[2]
        assert abs(bal - rbal) < 1e-12
    assert not np.array_equal(res[0][1], res[1][1])   # the ranks saw different loads


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the reference arm's other ranks exit at once, with no output and no
    process group (rank 0 alone times the oracle and prints the line)."""
    import argparse

    import bench
    from combine_moe_route_03_gb300 import configs
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(argparse.Namespace(steps=1, warmup=1, gpus=2), configs.DECODE)
    assert capsys.readouterr().out == ""
    assert bench.run_config(configs.DECODE, 2)["global_batch"] == 2 * configs.DECODE.B


def _eplb_dead_peer_rank(rank, world, port, q):
    import datetime
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        dist.barrier()
        os._exit(0)                      # leaves between steps, never plans
    import numpy as np
    from combine_moe_route_03_gb300 import api
    rec = api.EplbRecorder(32, 40, period=1, n_group=4, n_nodes=2, n_gpus=4, max_rep=4)
    rec.observe(np.arange(32, dtype=np.int32))
    dist.barrier()
    time.sleep(1.0)
    t0 = time.time()
    try:
        rec.plan(group=dist.group.WORLD)
        q.put(("planned", 0.0, None, None))
    except Exception:                    # the peer is gone: the collective fails
        q.put(("error", time.time() - t0, rec.load.tolist(), rec.steps))
        m, _ = rec.plan()                # the kept window still plans locally
        q.put(("local", 0.0, [a.tolist() for a in m], None))
    q.close()
    q.join_thread()                      # flush before leaving without cleanup
    os._exit(0)


def test_cross_rank_plan_with_a_departed_rank_fails_and_keeps_the_window():
    """A rank that left between steps makes the other rank's cross-rank plan raise
    within the process group's timeout instead of waiting for ever; the recorder keeps
    the loads it recorded, so the caller can re-plan (here: locally)."""
    from combine_moe_route_03_gb300 import build
    build.build()
    from oracle import eplb as oeplb
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_eplb_dead_peer_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        kind, dt, load, steps = q.get(timeout=90)
        assert kind == "error" and dt < 30.0
        assert load == list(range(32)) and steps == 1
        kind, _, m, _ = q.get(timeout=60)
        ref, _ = oeplb.plan(list(range(32)), 32, 40, 4, 2, 4, 4)
        assert kind == "local" and m == [[list(map(int, r)) for r in ref[0]],
                                         list(map(int, ref[1])), list(map(int, ref[2]))]
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
