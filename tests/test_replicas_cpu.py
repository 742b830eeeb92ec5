"""The multi-GPU form of this path is replicas only (each GPU decodes its own
sequences; there is no exchange step).  The benchmark's N-rank bookkeeping --
max of the ranks' times, job throughput = ranks x units / slowest time -- is
checked here on 2 CPU ranks over gloo."""
import os

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(1.0 + rank, world, "cpu")  # rank 1 is the slower replica
        q.put((rank, t, bench.replica_throughput(100.0, world, t)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t, thr in got:
        assert t == pytest.approx(2.0)      # every rank sees the slowest replica's time
        assert thr == pytest.approx(100.0)  # 2 ranks x 100 units / 2.0 s
