"""bench.py's multi-rank aggregation on CPU: two gloo ranks, each with its own
step time; both must see the slowest rank's time, and the job's rate counts
the work of every rank (weak scaling). No GPU is involved."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = 2.0 + 3.0 * rank                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world, torch.device("cpu"))
        results[rank] = (slowest, bench.job_rate(1000.0, world, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    world = 2
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(results) == {0: (5.0, 2 * 1000.0 / 5e-3), 1: (5.0, 2 * 1000.0 / 5e-3)}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_rate(10.0, 1, 1.0) == 10.0 / 1e-3
