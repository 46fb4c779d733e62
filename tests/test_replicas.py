"""The multi-GPU path of bench.py is replicas only (every rank runs its own
seeded batch, no data-path collective); its only cross-rank steps are the
barriers and the max-over-ranks timing reduction.  Those run here on CPU as
two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_setup()
        assert (w, r) == (world, rank)
        dist.barrier()
        # rank r's timed region took 10 + r ms, its e2e 40 - r ms
        total, e2e = bench.max_over_ranks(dist, [10.0 + rank, 40.0 - rank], "cpu")
        out[rank] = (total, e2e, bench.job_rate(1e12, 5, world, total))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_on_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        total, e2e, rate = out[rank]
        assert total == 11.0 and e2e == 40.0  # the slowest rank's times, on every rank
        assert rate == pytest.approx(1e12 * 5 * world / 11e-3)


def test_one_process_needs_no_group():
    assert bench.max_over_ranks(None, [3, 4.5], "cpu") == [3.0, 4.5]
    assert bench.job_rate(2.0, 10, 1, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_0_only():
    class Args:
        workload, steps, warmup = "fwd_b1_h1_n256_d64", 1, 3
    assert bench.bench_reference(Args, 2, 1) is None
    line = bench.bench_reference(Args, 2, 0)
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
