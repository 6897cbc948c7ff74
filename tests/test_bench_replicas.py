"""The multi-GPU form of the bench is replicas: each rank runs its own batch and
the only collective is the timing max. These tests run that logic as two gloo
processes on the CPU: the slowest rank's time wins, the job's throughput counts
every rank's tokens, and the ranks' batches are independent."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        slowest = bench.max_over_ranks(ms, w, torch.device("cpu"))
        cfg = W.config("tiny_sliding_decode")
        inp = W.generate(cfg, seed=bench.rank_seed(cfg["seed"], r))
        out[rank] = (w, r, local, slowest, bench.job_throughput(cfg["batch"] * cfg["q_len"], w, slowest),
                     inp["qkv"][:4].copy())
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_is_the_slowest_and_throughput_counts_both():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    for rank in range(world):
        w, r, local, slowest, tput, _ = res[rank]
        assert (w, r, local) == (world, rank, rank)
        assert slowest == 15.0
        assert tput == pytest.approx(2 * 2 / 15e-3)
    assert not np.array_equal(res[0][5], res[1][5])  # independent batches per replica


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(64, 1, 16.0e-3) == pytest.approx(64 / 16e-6)
    assert bench.rank_seed(1002, 0) == 1002 and bench.rank_seed(1002, 1) != 1002
