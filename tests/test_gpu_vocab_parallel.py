"""Vocabulary-parallel logprobs across processes: bit-identical to one GPU.

World sizes 2 and 4, every rank a separate process on cuda:0, gloo with
host-staged all-gather (the kernels of different ranks never wait on one
another: each rank's partials kernel finishes before its states are
exchanged on the host).  Fused path at the Qwen3-Next head shape
(T=16384, d=2048, V=151936, 1/2 or 1/4 of W per rank); logits path on the
peaked 1024 x 151936 logits at temperature 0.7, forward only and forward with
log Z plus each rank's columns of dL/dz.  Every rank's merged logp, entropy
(and log Z) must equal the unsharded single-process call bit for bit (the
prior-art report's tp4_equals_tp1), and each rank's gradient columns the same
columns of the single-process gradient.
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
    # training on the logits path: forward with log Z and the full dL/dz, whose
    # column shards every rank must reproduce
    T, V = z.z.shape
    gl, ge = workers.upstream(T)
    t_lp, t_ent, t_lse = lp.logprob_from_logits_lse(z.z, z.y, 0.7)
    grad = lp.logprob_from_logits_backward(z.z, z.y, gl, ge, 0.7, saved_lse=t_lse,
                                           saved_entropy=t_ent)
    shas = {}
    for n in (2, 4):
        for r in range(n):
            b, e = lp.vocab_shard_range(V, r, n)
            shas[(n, r)] = workers.sha256_of(grad[:, b:e])
    del z, grad
    torch.cuda.synchronize()
    return {"fused": [t.cpu() for t in fused], "logits": [t.cpu() for t in logits],
            "logits_train": [t.cpu() for t in (t_lp, t_ent, t_lse)], "grad_sha": shas}


@pytest.mark.parametrize("path", ["fused", "logits", "logits_train"])
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
    ref_lp, ref_ent = references[path][:2]
    for r in range(world):
        got = torch.load(os.path.join(tmp_path, f"rank{r}.pt"))
        assert torch.equal(bits(got["logp"]), bits(ref_lp)), (world, path, r)
        assert torch.equal(bits(got["ent"]), bits(ref_ent)), (world, path, r)
        if path == "logits_train":
            assert torch.equal(bits(got["lse"]), bits(references[path][2])), (world, r)
            assert got["grad_sha"] == references["grad_sha"][(world, r)], (world, r)
