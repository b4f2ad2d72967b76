"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks, replicas with
different per-rank times; the job time is the slowest rank's and the job
value counts every rank's bytes (weak scaling)."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    bench.barrier(world)
    my_seconds = 0.5 + rank                       # rank 1 is the slow one
    worst = bench.reduce_max(my_seconds, world, "cpu")
    gbs = bench.job_gbs(10 ** 9, 4, worst, world)
    q.put((rank, worst, gbs))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, worst, gbs in got:
        assert worst == 1.5
        assert gbs == pytest.approx(2 * 4 * 1e9 / 1.5 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.0, 1, "cpu") == 3.0
    assert bench.job_gbs(2 * 10 ** 9, 10, 2.0, 1) == pytest.approx(10.0)
