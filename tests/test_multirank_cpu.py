"""The benchmark's multi-rank plumbing on CPU with gloo (world size 2):
rendezvous from the torchrun environment variables, barrier, the max-over-
ranks timing reduction and the weak-scaling whole-job rate.  Every (batch,
channel) of the scan is independent, so ranks exchange no data."""
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
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    torch.cuda.is_available = lambda: False          # CPU test: force the gloo backend
    import bench
    w, r, local = bench.dist_init(world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)            # rank 1 is slower
    rate = bench.whole_job_rate(w, 1000, 4, slowest)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, slowest, rate))


def test_two_ranks_gloo():
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
    for r, w, slowest, rate in res:
        assert w == 2 and slowest == 15.0
        assert rate == pytest.approx(2 * 1000 * 4 / 15e-3)


def test_single_rank_rate():
    import bench
    assert bench.whole_job_rate(1, 10, 2, 4.0) == pytest.approx(5000.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
