"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, max over ranks
and whole-job rates (no GPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local = {"pre_s": 1.0 + rank, "dec_s": 2.0 - rank, "total_ms": 10.0 * (rank + 1)}
        agg = bench.aggregate_ranks(local, world, "cpu")
        out[rank] = agg
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    # spawn, not fork: earlier tests may have started the oracle's threads
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    for rank in range(world):
        assert res[rank] == {"pre_s": 2.0, "dec_s": 2.0, "total_ms": 20.0}


def test_whole_job_rate_counts_every_rank():
    import bench

    assert bench.whole_job_rate(100.0, 2.0, 1) == 50.0
    assert bench.whole_job_rate(100.0, 2.0, 4) == 200.0
    assert bench.aggregate_ranks({"a": 1.5}, 1, None) == {"a": 1.5}
