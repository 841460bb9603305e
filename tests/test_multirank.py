"""Host logic of the multi-rank benchmark path, on CPU with world-size-2 gloo ranks.

Every rank runs its own batch of the workload (no collective on the data path);
the job's time is the slowest rank's and its throughput counts every rank's work.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from exact_head_attention_gb300 import workloads


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(times[rank], dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world, port = 2, _free_port()
    times = [1.25, 3.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(2.0, None, "cpu") == 2.0


def test_job_throughput_counts_every_rank():
    w = workloads.WORKLOADS[workloads.HEADLINE]
    f, b = bench.step_flops(w)
    assert f == pytest.approx(4 * 12 * 8192 * 8192 * 128 / 2)
    assert b == pytest.approx(2.5 * f)
    one = bench.job_throughput(f + b, 1, 0.72)
    assert bench.job_throughput(f + b, 8, 0.72) == pytest.approx(8 * one)


def test_ranks_draw_different_batches():
    w = workloads.custom(1, 1, 16, 16, 64)
    a, b = workloads.make_inputs(w, seed_offset=0), workloads.make_inputs(w, seed_offset=1)
    assert not (a["q"] == b["q"]).all()
