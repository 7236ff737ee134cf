"""The N > 1 host logic of bench.py on CPU with gloo (world size 2).

Rows are independent, so each rank runs its own batch with no data-path
collective; the only cross-rank steps are the barrier and the max over ranks
of the timed region, and rank 0 alone prints.  These run here as two gloo
processes on 127.0.0.1.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = [12.5, 20.0][rank]
        m = bench.max_over_ranks(local_ms, world, "cpu")
        out[rank] = m
        # whole-job throughput: all ranks' rows over the slowest rank's time
        out[world + rank] = bench.whole_job_throughput(512, 10, world, m)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Array("d", 2 * world)
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert list(out[:world]) == [20.0, 20.0]
    assert out[world] == pytest.approx(2 * 512 * 10 / 0.020)
    assert out[world] == out[world + 1]


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.whole_job_throughput(512, 200, 1, 100.0) == pytest.approx(512 * 200 / 0.1)


def test_reference_arm_non_zero_rank_exits_without_work(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "1000"])
    assert bench.run_reference(args) == 0
