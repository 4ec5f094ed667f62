"""The N > 1 host path of bench.py on CPU: two gloo ranks (the path shards by
sequence into independent replicas, so timing is the only cross-rank
exchange).  The job's time is the slowest rank's, its rate counts every
rank's units, and the reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import argparse

    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench._max_over_ranks(dist, 10.0 + 5.0 * rank, torch.device("cpu"))
        rate = bench._whole_job_rate(world, 100, 4, slowest / 1e3)
        # the reference arm: rank 0 alone does the work and prints
        args = argparse.Namespace(workload=0, steps=1, warmup=0, gpus=world)
        ref_rc = bench.run_reference(args) if rank != 0 else 0
        q.put((rank, slowest, rate, ref_rc))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_and_count_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate, ref_rc in got:
        assert slowest == 15.0                      # max over ranks, seen by every rank
        assert rate == pytest.approx(2 * 100 * 4 / 0.015)
        assert ref_rc == 0                          # rank 1 returns without work


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(None, 3.5, None) == 3.5
    assert bench._whole_job_rate(1, 10, 2, 0.5) == 40.0
