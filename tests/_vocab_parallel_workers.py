"""Rank processes of the vocabulary-parallel tests (spawned by
tests/test_vocab_parallel_host.py and tests/test_gpu_vocab_parallel.py)."""

from __future__ import annotations

import os

import torch
import torch.distributed as dist


def upstream(T: int):
    """The upstream gradients of the logits-path training test (same on every rank)."""
    g = torch.Generator(device="cuda:0")
    g.manual_seed(21)
    return (torch.randn(T, generator=g, device="cuda:0"),
            torch.randn(T, generator=g, device="cuda:0"))


def sha256_of(t: torch.Tensor) -> str:
    import hashlib
    t = t.contiguous()
    if t.dtype == torch.bfloat16:  # numpy has no bfloat16: hash the same bytes as int16
        t = t.view(torch.int16)
    return hashlib.sha256(t.cpu().numpy().tobytes()).hexdigest()


def _init(rank: int, world: int, init_file: str) -> None:
    # a file rendezvous: no TCP port to pick or to collide on
    dist.init_process_group("gloo", init_method=f"file://{init_file}", rank=rank,
                            world_size=world)


def host_gather(rank: int, world: int, init_file: str, out_dir: str) -> None:
    """Each rank contributes a [T, 4 / world, 8] state tensor whose bytes name
    the rank (with -inf and NaN payloads among them); the gathered tensors are
    saved for the parent to check."""
    from invariant_token_logprobs_gb300 import vocab_parallel as vp
    _init(rank, world, init_file)
    try:
        T, nq = 5, 4 // world
        bits = torch.arange(T * nq * 8, dtype=torch.int32).view(T, nq, 8) + (rank << 20)
        bits[0, 0, 0] = 0x7FC00000 + rank  # NaN with a payload
        bits[1, 0, 4] = -8388608            # -inf (0xff800000)
        part = bits.view(torch.float32)
        got = vp.gather_partials(part)
        shard = vp.shard_of_rank(151936)
        torch.save({"got": [g.view(torch.int32).clone() for g in got], "shard": shard},
                   os.path.join(out_dir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


def gpu_vocab_parallel(rank: int, world: int, init_file: str, out_dir: str, path: str) -> None:
    """Every rank on cuda:0: its shard's partial states, an all-gather over
    gloo (host-staged), the fixed merge.  Saves logp and entropy."""
    from invariant_token_logprobs_gb300 import lp, synth
    from invariant_token_logprobs_gb300 import vocab_parallel as vp
    _init(rank, world, init_file)
    try:
        torch.cuda.set_device(0)
        lp.load(build_if_needed=False)
        if path == "fused":
            x = synth.fused_inputs("fused_qwen3_next", device="cuda:0")
            V = x.W.shape[0]
            _, n, b, e = vp.shard_of_rank(V)
            w_shard = x.W[b:e]
            del x.W
            logp, ent = vp.vocab_parallel_linear_logprob(x.H, w_shard, x.y, V)
        elif path == "logits":
            x = synth.logits_inputs("logits_peaked", device="cuda:0")
            V = x.z.shape[1]
            _, n, b, e = vp.shard_of_rank(V)
            logp, ent = vp.vocab_parallel_logprob_from_logits(x.z[:, b:e], x.y, V,
                                                              temperature=0.7)
        elif path == "fused_train":
            # forward with log Z over the shards, then this rank's backward: its grad_W
            # rows, its partial grad_H, the all-gather and the merge of the partials
            x = synth.fused_inputs("fused_qwen3_8b", device="cuda:0")
            T, V = x.H.shape[0], x.W.shape[0]
            _, n, b, e = vp.shard_of_rank(V)
            w_shard = x.W[b:e].contiguous()
            del x.W
            gl, ge = upstream(T)
            logp, ent, lse = vp.vocab_parallel_linear_logprob_lse(x.H, w_shard, x.y, V,
                                                                  temperature=0.9)
            gH, gW = vp.vocab_parallel_linear_logprob_backward(x.H, w_shard, x.y, V, lse, ent,
                                                               gl, ge, temperature=0.9)
            torch.cuda.synchronize()
            torch.save({"logp": logp.cpu(), "ent": ent.cpu(), "lse": lse.cpu(),
                        "grad_h_sha": sha256_of(gH), "grad_w_sha": sha256_of(gW)},
                       os.path.join(out_dir, f"rank{rank}.pt"))
            return
        elif path == "fused_autograd":
            # the same through torch.autograd: a loss on logp and entropy, .backward()
            from invariant_token_logprobs_gb300 import autograd as ag
            x = synth.fused_inputs("fused_qwen3_8b", device="cuda:0")
            T, V = x.H.shape[0], x.W.shape[0]
            _, n, b, e = vp.shard_of_rank(V)
            w_shard = x.W[b:e].contiguous().requires_grad_(True)
            del x.W
            H = x.H.clone().requires_grad_(True)
            gl, ge = upstream(T)
            logp, ent = ag.vocab_parallel_linear_logprob(H, w_shard, x.y, V, temperature=0.9)
            ((logp * gl).sum() + (ent * ge).sum()).backward()
            torch.cuda.synchronize()
            torch.save({"logp": logp.detach().cpu(), "ent": ent.detach().cpu(),
                        "grad_h_sha": sha256_of(H.grad), "grad_w_sha": sha256_of(w_shard.grad)},
                       os.path.join(out_dir, f"rank{rank}.pt"))
            return
        else:  # logits_train: forward with log Z, then this rank's columns of dL/dz
            x = synth.logits_inputs("logits_peaked", device="cuda:0")
            T, V = x.z.shape
            _, n, b, e = vp.shard_of_rank(V)
            gl, ge = upstream(T)
            logp, ent, lse = vp.vocab_parallel_logprob_from_logits_lse(x.z[:, b:e], x.y, V,
                                                                       temperature=0.7)
            grad = vp.vocab_parallel_logprob_from_logits_backward(x.z[:, b:e], x.y, V, lse, ent,
                                                                  gl, ge, temperature=0.7)
            torch.cuda.synchronize()
            torch.save({"logp": logp.cpu(), "ent": ent.cpu(), "lse": lse.cpu(),
                        "grad_sha": sha256_of(grad)}, os.path.join(out_dir, f"rank{rank}.pt"))
            return
        torch.cuda.synchronize()
        torch.save({"logp": logp.cpu(), "ent": ent.cpu()}, os.path.join(out_dir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


def host_fused_backward(rank: int, world: int, init_file: str, out_dir: str) -> None:
    """The fused backward's orchestration on CPU: the library's compute calls are
    replaced by fakes that record their arguments, so what is checked is the
    shard each rank asks for, the rank order of the gathered partial grad_H and
    what the merge receives."""
    from invariant_token_logprobs_gb300 import lp
    from invariant_token_logprobs_gb300 import vocab_parallel as vp
    _init(rank, world, init_file)
    try:
        calls = {}
        T, d, V = 3, 8, 4096

        def fake_partials_backward(H, W_shard, y, vocab_total, shard_index, n_shards, lse, ent,
                                   gl, ge, **kw):
            calls["shard"] = (shard_index, n_shards, W_shard.shape[0], vocab_total)
            part = torch.full((T, d), float(shard_index + 1)) + torch.arange(T * d).view(T, d)
            return part, torch.full((W_shard.shape[0], d), float(-shard_index))

        def fake_merge(parts, stream=None):
            calls["merged"] = [p.clone() for p in parts]
            return torch.stack(parts).sum(0)

        lp.linear_logprob_partials_backward = fake_partials_backward
        lp.merge_grad_h_partials = fake_merge
        _, n, b, e = vp.shard_of_rank(V)
        H = torch.zeros((T, d))
        gH, gW = vp.vocab_parallel_linear_logprob_backward(
            H, torch.zeros((e - b, d)), torch.zeros(T, dtype=torch.int64), V,
            torch.zeros(T), torch.zeros(T), torch.zeros(T), None)
        torch.save({"calls": calls, "gH": gH, "gW": gW}, os.path.join(out_dir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()
