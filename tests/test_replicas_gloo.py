"""The N > 1 path of bench.py on CPU: two gloo ranks.

The path shards by replica (every rank runs its own batch, no data-path
collective); the only cross-rank step is the max-over-ranks of the timed
region and the whole-job throughput built from it.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 5.0][rank]
    worst = bench.max_over_ranks(ms, world)
    out[rank] = (worst, bench.job_throughput(1000.0, worst, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        worst, thr = out[r]
        assert worst == 5.0
        assert thr == pytest.approx(2 * 1000.0 / 5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(10.0, 2.0, 1) == pytest.approx(5000.0)
