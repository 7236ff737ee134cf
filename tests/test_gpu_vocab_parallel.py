"""Vocabulary-parallel logprobs across processes: bit-identical to one GPU.

World sizes 2 and 4, every rank a separate process on cuda:0, gloo with
host-staged all-gather (the kernels of different ranks never wait on one
another: each rank's partials kernel finishes before its states are
exchanged on the host).  Fused path at the Qwen3-Next head shape
(T=16384, d=2048, V=151936, 1/2 or 1/4 of W per rank); logits path on the
peaked 1024 x 151936 logits at temperature 0.7.  Every rank's merged logp and
entropy must equal the unsharded single-process call bit for bit (the
prior-art report's tp4_equals_tp1).
"""

import os

import pytest
import torch
import torch.multiprocessing as mp

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import bits

import _vocab_parallel_workers as workers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def references():
    lp.load()
    x = synth.fused_inputs("fused_qwen3_next", device=DEV)
    fused = lp.linear_logprob(x.H, x.W, x.y)
    del x
    z = synth.logits_inputs("logits_peaked", device=DEV)
    logits = lp.logprob_from_logits(z.z, z.y, temperature=0.7)
    del z
    torch.cuda.synchronize()
    return {"fused": [t.cpu() for t in fused], "logits": [t.cpu() for t in logits]}


@pytest.mark.parametrize("path", ["fused", "logits"])
@pytest.mark.parametrize("world", [2, 4])
def test_vocab_parallel_equals_single_gpu(world, path, references, tmp_path):
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=workers.gpu_vocab_parallel,
                         args=(r, world, str(tmp_path / "rendezvous"), str(tmp_path), path))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    ref_lp, ref_ent = references[path]
    for r in range(world):
        got = torch.load(os.path.join(tmp_path, f"rank{r}.pt"))
        assert torch.equal(bits(got["logp"]), bits(ref_lp)), (world, path, r)
        assert torch.equal(bits(got["ent"]), bits(ref_ent)), (world, path, r)
