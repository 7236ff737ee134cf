"""Small parity cases of every entry point, shared by the checked-build test:
run once with the normal library (in the test process) and once with the
checked library (in a child process); every output must have the same bits."""

from __future__ import annotations

import torch

DEV = "cuda:0"


def run_cases(lp, synth) -> dict:
    out = {}

    def keep(name, *ts):
        for i, t in enumerate(ts):
            if t is not None:
                out[f"{name}.{i}"] = t.detach().contiguous().view(torch.uint8).cpu()

    # logits path: ragged vocabularies, an unaligned row stride, temperature, shards
    for T, V in [(37, 1001), (64, 8192), (4, 3), (9, 4096 + 13)]:
        x = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=100 + V)
        keep(f"logits{T}x{V}", *lp.logprob_from_logits(x.z, x.y))
        keep(f"logits{T}x{V}.t07", *lp.logprob_from_logits(x.z, x.y, temperature=0.7))
        for n in (2, 4):
            parts = []
            for i in range(n):
                b, e = lp.vocab_shard_range(V, i, n)
                parts.append(lp.logprob_partials_from_logits(x.z[:, b:e], x.y, V, i, n))
            keep(f"logits{T}x{V}.merge{n}", *lp.merge_partials(parts))
    x = synth.logits_inputs("logits_peaked", device=DEV, T=16, V=20000, seed=7)
    wide = torch.empty((16, 20001), device=DEV)
    wide[:, :20000] = x.z
    keep("logits.unaligned", *lp.logprob_from_logits(wide[:, :20000], x.y))
    # logits-path backward: with log Z, aligned and unaligned rows, temperature
    g = torch.Generator(device=DEV)
    g.manual_seed(16)
    gl = torch.randn(16, generator=g, device=DEV)
    ge = torch.randn(16, generator=g, device=DEV)
    keep("logits.lse", *lp.logprob_from_logits_lse(x.z, x.y, 0.7))
    keep("logits.bwd", lp.logprob_from_logits_backward(x.z, x.y, gl, ge))
    keep("logits.bwd.unaligned", lp.logprob_from_logits_backward(wide[:, :20000], x.y, gl, None,
                                                                 temperature=0.7))
    # vocabulary-parallel training: merge with log Z, each shard's gradient columns
    for n in (2, 4):
        parts = []
        for i in range(n):
            b, e = lp.vocab_shard_range(20000, i, n)
            parts.append(lp.logprob_partials_from_logits(x.z[:, b:e], x.y, 20000, i, n))
        m = [torch.empty(16, device=DEV) for _ in range(3)]
        lp.lp_merge_partials_lse(parts, 16, m[0], m[1], m[2])
        keep(f"logits.merge_lse{n}", *m)
        for i in range(n):
            b, e = lp.vocab_shard_range(20000, i, n)
            gs = torch.empty((16, e - b), device=DEV)
            lp.lp_logprob_partials_from_logits_backward(x.z[:, b:e], x.y, 20000, i, n, 1.0, m[2],
                                                        m[1], gl, ge, gs)
            keep(f"logits.bwd.shard{n}.{i}", gs)

    # fused path: tiny, fewer than 16 rows, ragged V, temperature, shards, lse, no-alloc
    for T, d, V in [(64, 256, 8192), (5, 256, 3001), (300, 512, 20003)]:
        f = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T + d)
        keep(f"fused{T}", *lp.linear_logprob(f.H, f.W, f.y))
        keep(f"fused{T}.t07", *lp.linear_logprob(f.H, f.W, f.y, temperature=0.7))
        keep(f"fused{T}.lse", *lp.linear_logprob_lse(f.H, f.W, f.y))
        for n in (2, 4):
            parts = []
            for i in range(n):
                b, e = lp.vocab_shard_range(V, i, n)
                parts.append(lp.linear_logprob_partials(f.H, f.W[b:e], f.y, V, i, n))
            keep(f"fused{T}.merge{n}", *lp.merge_partials(parts))
        logp = torch.empty(T, device=DEV)
        ent = torch.empty(T, device=DEV)
        lp.lp_linear_logprob_noalloc(f.H, f.W, f.y, logp, ent)
        keep(f"fused{T}.noalloc", logp, ent)

    # backward: fp32 and bf16 grad_W, the padded small batch, saved statistics
    for T, d, V in [(64, 256, 8192), (5, 64, 3001)]:
        f = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T + 3)
        g = torch.Generator(device=DEV)
        g.manual_seed(T)
        gl = torch.randn(T, generator=g, device=DEV)
        ge = torch.randn(T, generator=g, device=DEV)
        keep(f"bwd{T}", *lp.linear_logprob_backward(f.H, f.W, f.y, gl, ge))
        keep(f"bwd{T}.bf16", *lp.linear_logprob_backward(f.H, f.W, f.y, gl, ge,
                                                         grad_W_dtype=torch.bfloat16))
        _, ent, lse = lp.linear_logprob_lse(f.H, f.W, f.y, temperature=0.8)
        keep(f"bwd{T}.saved", *lp.linear_logprob_backward(f.H, f.W, f.y, gl, None, temperature=0.8,
                                                          saved_lse=lse, saved_entropy=ent))
    # vocabulary-parallel backward: every shard's partial grad_H and grad_W rows, the
    # merge (V % 64 == 0: quarter-ordered grad_H), and the padded small batch
    for T, d, V in [(64, 256, 8192), (5, 64, 4096 + 64), (300, 128, 20480)]:
        f = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T + 5)
        g = torch.Generator(device=DEV)
        g.manual_seed(T + 1)
        gl = torch.randn(T, generator=g, device=DEV)
        ge = torch.randn(T, generator=g, device=DEV)
        _, ent, lse = lp.linear_logprob_lse(f.H, f.W, f.y)
        for n in (1, 2, 4):
            parts = []
            for i in range(n):
                b, e = lp.vocab_shard_range(V, i, n)
                ph, pw = lp.linear_logprob_partials_backward(f.H, f.W[b:e], f.y, V, i, n, lse, ent,
                                                             gl, ge)
                keep(f"bwd{T}.shard{n}.{i}", ph, pw)
                parts.append(ph)
            keep(f"bwd{T}.shard{n}.merged", lp.merge_grad_h_partials(parts))
        # grad_W added into a main gradient
        main = torch.ones((V, d), device=DEV)
        keep(f"bwd{T}.acc", *lp.linear_logprob_backward(f.H, f.W, f.y, gl, ge, saved_lse=lse,
                                                        saved_entropy=ent, accumulate_into=main))
    torch.cuda.synchronize()
    return out
