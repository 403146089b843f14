"""CPU checks of the benchmark's multi-replica logic with two gloo ranks:
each rank times its own replica, the job's time is the slowest rank's and
the throughput counts every replica's work."""
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
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    t = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
    v = bench.whole_job_throughput(100.0, w, t)
    q.put((r, w, lr, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, w, lr, t, v) in enumerate(res):
        assert (r, w, lr) == (rank, 2, rank)
        assert t == 2.5                       # max over ranks
        assert v == pytest.approx(200.0 / 2.5)
