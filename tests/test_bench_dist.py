"""Multi-process rank logic of bench.py on the CPU (gloo, world size 2):
rendezvous, barrier, max over ranks, per-rank seeds and the whole-job value."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), SA_BENCH_BACKEND="gloo")
    import bench
    import torch.distributed as dist
    r, wsz = bench.dist_setup()
    bench.barrier(wsz)
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, wsz)
    dist.destroy_process_group()
    q.put((r, wsz, slowest))


def test_two_ranks_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in results] == [0, 1]
    assert all(x[1] == 2 for x in results)
    assert all(x[2] == 15.0 for x in results)   # every rank sees the slowest time


def test_rank_seeds_and_job_value():
    import bench
    from sparse_long_context_banded_gb300 import inputs
    w = inputs.workload(5)
    seeds = [bench.rank_seed(w, r) for r in range(8)]
    assert seeds[0] == 1005 and len(set(seeds)) == 8
    # 2 ranks, 1 TFLOP each per step, 10 steps in 20 ms on the slowest rank
    assert bench.job_value(1e12, 10, 20.0, 2) == pytest.approx(1000.0)
    assert bench.job_value(1e12, 10, 20.0, 1) == pytest.approx(500.0)
