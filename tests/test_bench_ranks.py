"""bench.py's multi-process path (replicas only: no collective on the data
path) on CPU: two gloo ranks reduce their timings with a max, and the
whole-job throughput counts every replica's work."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    vals = bench.max_over_ranks([10.0 + rank, 5.0 - rank], world, "cpu")
    q.put((rank, vals))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == [11.0, 5.0]


def test_job_throughput_counts_every_replica():
    import bench
    assert bench.job_throughput(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.job_throughput(1e12, 4, 1000.0) == pytest.approx(4.0)
    assert bench.max_over_ranks([1.0, 2.0], 1, "cpu") == [1.0, 2.0]
