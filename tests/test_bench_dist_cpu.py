"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, each with
its own step time; both must see the slowest rank's time, and the job
throughput must count every rank's drafted tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [0.25, 0.75][rank]
    got = bench.max_over_ranks(local_ms, dist, "cpu")
    env = bench.dist_env()
    q.put((rank, got, env, bench.job_throughput(world, 1, 4, got)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, env, thr in out:
        assert got == pytest.approx(0.75)
        assert env == (rank, 2, rank)
        assert thr == pytest.approx(2 * 1 * 4 / 0.75e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.job_throughput(1, 64, 8, 2.0) == pytest.approx(256000.0)
