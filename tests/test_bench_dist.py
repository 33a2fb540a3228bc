"""The N > 1 bench path on CPU: two gloo ranks, each an independent replica,
reduce only their timing and unit counts (max of times, sum of units); the
replicas draw different inputs (seed = rank)."""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import make_e2e_inputs, step_config


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        # rank r: (r + 1) ms for 10 (r + 1) committed tokens
        ms, units, value = bench.job_throughput(rank + 1.0, 10 * (rank + 1))
        out[rank] = (ms, units, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time_and_total_units():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == (2.0, 30.0, pytest.approx(30.0 / 2e-3))


def test_single_process_needs_no_group():
    assert bench.job_throughput(4.0, 8) == (4.0, 8.0, 2000.0)


def test_replicas_draw_different_inputs():
    a, b = step_config("tiny", seed=0), step_config("tiny", seed=1)
    assert not np.array_equal(a["q"], b["q"]) and not np.array_equal(a["hidden"], b["hidden"])
    e0, e1 = make_e2e_inputs(seed=0, layers=1, d=64, H=2, dh=32, ffn=64, V=64, prompt_len=8, resp_len=16,
                             blk=8, vic=4), make_e2e_inputs(seed=1, layers=1, d=64, H=2, dh=32, ffn=64, V=64,
                                                            prompt_len=8, resp_len=16, blk=8, vic=4)
    assert not np.array_equal(e0["prompt"], e1["prompt"])


def test_one_thread_oracle_sample_runs():
    """The single-thread oracle baseline runs in a fresh interpreter with the
    BLAS / OpenMP pools at one thread; the bench swallows its failure, so
    this is where a broken sample shows."""
    r = bench.time_oracle_one_thread("tiny", False, 0.5)
    assert r is not None and r["steps"] >= 1 and r["secs"] > 0 and r["commits"] >= r["steps"]
