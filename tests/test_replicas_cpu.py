"""The multi-GPU path is replicas only: every rank runs its own streams with its own
caches and no data-path collective; the one collective reduces the timings to the
slowest rank's.  These tests run that host logic as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from autoregressive_codebook_tts_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank 0 is slower on the first timing, rank 1 on the second
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25], world)
        # each rank's own replica inputs (seeded by rank)
        rows, _, _, _ = W.qkv(2, 16, 8, 128, seed=rank)
        q.put((rank, got, float(rows.double().sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_keep_their_own_inputs():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, got, _ in res:
        assert got == [2.0, 5.0, 0.25], rank
    assert res[0][2] != res[1][2]  # replicas draw different streams


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]


def test_whole_job_throughput_counts_every_replica():
    # 2 replicas x 1e9 bytes x 10 steps in 5 s (slowest rank) = 4 GB/s
    assert bench.whole_job_gbs(2, 1e9, 10, 5.0) == pytest.approx(4.0)
    assert bench.whole_job_gbs(1, 1e9, 10, 5.0) == pytest.approx(2.0)
