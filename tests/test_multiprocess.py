"""Replicas on several ranks (the benchmark's N > 1 path), with the gloo
backend on CPU: each rank runs its own sequences; the job's throughput is the
tokens of all ranks over the slowest rank's time, with no collective on the
data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, tokens, seconds, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    assert bench.dist_env() == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.job_throughput(tokens[rank], seconds[rank], world)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_job_throughput_sums_tokens_over_the_slowest_rank(world):
    tokens, seconds = [100.0, 300.0], [1.0, 2.5]
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a multi-threaded process
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), tokens, seconds, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        tps, slowest = res[r]
        assert slowest == 2.5
        assert abs(tps - 400.0 / 2.5) < 1e-12


def test_single_rank_needs_no_process_group():
    assert bench.job_throughput(50.0, 0.5, 1) == (100.0, 0.5)
