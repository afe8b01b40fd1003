"""The multi-replica plumbing of bench.py on CPU: two gloo ranks (world size 2) take
the maximum of their timings, the reference arm works on rank 0 only, and the
whole-job figure counts every replica's bytes.  No GPU: the kernels are not run."""

import os
import socket
import sys
from types import SimpleNamespace

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, torch.device("cpu"))
    dist.barrier()
    ref = bench.run_reference(SimpleNamespace(m=1, steps=1, warmup=0), rank, world) if rank != 0 else "rank 0"
    queue.put((rank, got, ref))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_timing_and_only_rank0_runs_the_reference():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict((r, (got, ref)) for r, got, ref in (queue.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert results[r][0] == [2.0, 10.0]   # each entry: the maximum over the two ranks
    assert results[1][1] is None               # rank 1 does no reference work


def test_job_figure_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_gbs(1e9, 1.0, 1) == pytest.approx(1000.0)
    assert bench.job_gbs(1e9, 1.0, 4) == pytest.approx(4000.0)
    assert bench.max_over_ranks([3, 4.5], None, None) == [3.0, 4.5]
