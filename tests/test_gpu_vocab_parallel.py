"""Vocabulary-parallel logprobs across processes: bit-identical to one GPU.

World sizes 2 and 4, every rank a separate process on cuda:0, gloo with
host-staged all-gather (the kernels of different ranks never wait on one
another: each rank's partials kernel finishes before its states are
exchanged on the host).  Fused path at the Qwen3-Next head shape
(T=16384, d=2048, V=151936, 1/2 or 1/4 of W per rank); logits path on the
peaked 1024 x 151936 logits at temperature 0.7, forward only and forward with
log Z plus each rank's columns of dL/dz.  Fused training at the Qwen3-8B head
(T=512, d=4096, V=151936, temperature 0.9): forward with log Z, then each
rank's grad_W rows and partial grad_H, all-gathered and merged.  Every rank's
merged logp, entropy (and log Z) must equal the unsharded single-process call
bit for bit (the prior-art report's tp4_equals_tp1), each rank's gradient
columns (or grad_W rows) the same part of the single-process gradient, and
every rank's grad_H the single-process grad_H; the same training step through
the vocabulary-parallel autograd binding must give every rank the
single-process autograd gradients (bf16) of H and of its rows of W.
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
    # fused training: forward with log Z and the single-GPU backward
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    T, V = x.H.shape[0], x.W.shape[0]
    gl, ge = workers.upstream(T)
    f_lp, f_ent, f_lse = lp.linear_logprob_lse(x.H, x.W, x.y, 0.9)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, 0.9, saved_lse=f_lse,
                                        saved_entropy=f_ent)
    w_shas = {}
    for n in (2, 4):
        for r in range(n):
            b, e = lp.vocab_shard_range(V, r, n)
            w_shas[(n, r)] = workers.sha256_of(gW[b:e])
    h_sha = workers.sha256_of(gH)
    del gH, gW
    # the same through the single-GPU autograd binding (bf16 gradients)
    from invariant_token_logprobs_gb300 import autograd as ag
    H = x.H.clone().requires_grad_(True)
    Wg = x.W.clone().requires_grad_(True)
    a_lp, a_ent = ag.linear_logprob(H, Wg, x.y, 0.9)
    ((a_lp * gl).sum() + (a_ent * ge).sum()).backward()
    aw_shas = {}
    for n in (2, 4):
        for r in range(n):
            b, e = lp.vocab_shard_range(V, r, n)
            aw_shas[(n, r)] = workers.sha256_of(Wg.grad[b:e])
    ah_sha = workers.sha256_of(H.grad)
    a_out = [a_lp.detach().cpu(), a_ent.detach().cpu()]
    del x, H, Wg, a_lp, a_ent
    torch.cuda.synchronize()
    return {"fused": [t.cpu() for t in fused], "logits": [t.cpu() for t in logits],
            "logits_train": [t.cpu() for t in (t_lp, t_ent, t_lse)], "grad_sha": shas,
            "fused_train": [t.cpu() for t in (f_lp, f_ent, f_lse)], "grad_w_sha": w_shas,
            "grad_h_sha": h_sha, "fused_autograd": a_out, "ag_w_sha": aw_shas, "ag_h_sha": ah_sha}


@pytest.mark.parametrize("path", ["fused", "logits", "logits_train", "fused_train",
                                  "fused_autograd"])
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
        if path == "fused_train":
            assert torch.equal(bits(got["lse"]), bits(references[path][2])), (world, r)
            assert got["grad_h_sha"] == references["grad_h_sha"], (world, r)
            assert got["grad_w_sha"] == references["grad_w_sha"][(world, r)], (world, r)
        if path == "fused_autograd":
            assert got["grad_h_sha"] == references["ag_h_sha"], (world, r)
            assert got["grad_w_sha"] == references["ag_w_sha"][(world, r)], (world, r)
