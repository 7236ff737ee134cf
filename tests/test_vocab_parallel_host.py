"""The vocabulary-parallel data plane on CPU (gloo, world sizes 2 and 4).

The only exchange of the vocabulary-parallel path is an all-gather of the
ranks' quarter states; these checks need no GPU: every rank receives every
rank's states, in rank order, byte for byte (NaN payloads and -inf included),
and rank r owns the contiguous vocabulary shard r.
"""

import os

import pytest
import torch
import torch.multiprocessing as mp

from invariant_token_logprobs_gb300 import lp
from invariant_token_logprobs_gb300 import vocab_parallel as vp

import _vocab_parallel_workers as workers


@pytest.mark.parametrize("world", [2, 4])
def test_gather_in_rank_order_byte_exact(world, tmp_path):
    mp.spawn(workers.host_gather, args=(world, str(tmp_path / "rendezvous"), str(tmp_path)), nprocs=world,
             join=True)
    T, nq = 5, 4 // world
    for rank in range(world):
        res = torch.load(os.path.join(tmp_path, f"rank{rank}.pt"))
        got = res["got"]
        assert len(got) == world
        for src in range(world):
            expect = torch.arange(T * nq * 8, dtype=torch.int32).view(T, nq, 8) + (src << 20)
            expect[0, 0, 0] = 0x7FC00000 + src
            expect[1, 0, 4] = -8388608
            assert got[src].shape == (T, nq, 8)
            assert torch.equal(got[src], expect), (rank, src)
        idx, n, b, e = res["shard"]
        assert (idx, n) == (rank, world)
        assert (b, e) == lp.vocab_shard_range(151936, rank, world)


def test_single_process_is_its_own_group():
    part = torch.zeros((3, 4, 8))
    got = vp.gather_partials(part)
    assert len(got) == 1 and got[0] is part
    assert vp.shard_of_rank(151936) == (0, 1, 0, 151936)


@pytest.mark.parametrize("world", [2, 4])
def test_fused_backward_gathers_partials_in_rank_order(world, tmp_path):
    """Each rank asks for its own shard, every rank's merge receives the partial
    grad_H of every rank in rank order, and each rank keeps its own grad_W rows."""
    mp.spawn(workers.host_fused_backward, args=(world, str(tmp_path / "rendezvous"), str(tmp_path)),
             nprocs=world, join=True)
    T, d, V = 3, 8, 4096
    for rank in range(world):
        res = torch.load(os.path.join(tmp_path, f"rank{rank}.pt"))
        b, e = lp.vocab_shard_range(V, rank, world)
        assert res["calls"]["shard"] == (rank, world, e - b, V)
        merged = res["calls"]["merged"]
        assert len(merged) == world
        for src in range(world):
            expect = torch.full((T, d), float(src + 1)) + torch.arange(T * d).view(T, d)
            assert torch.equal(merged[src], expect), (rank, src)
        assert torch.equal(res["gH"], torch.stack(merged).sum(0))
        assert torch.equal(res["gW"], torch.full((e - b, d), float(-rank)))
