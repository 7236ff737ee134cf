"""torch.autograd bindings of the fused path and of the logits path.

    logp, entropy = linear_logprob(H, W, y, temperature=1.0)
    logp, entropy = logprob_from_logits(z, y, temperature=1.0)
    logp, entropy = vocab_parallel_linear_logprob(H, W_shard, y, V, group)
    logp, entropy = vocab_parallel_logprob_from_logits(z_shard, y, V, group)

returns the selected-token log-probabilities and entropies of z = H W^T / tau
(lp_linear_logprob_lse) and back-propagates into H and W through
lp_linear_logprob_backward with the forward's log Z and entropy kept, so the
backward does not recompute them.  This is argument marshalling only: every
step runs in liblp's kernels, on the current stream.

The vocabulary-parallel forms run on every rank of a torch.distributed group
(1, 2 or 4 ranks, rank r holding shard r of W's rows or of the logits'
columns, see vocab_parallel.shard_of_rank): the forward all-gathers the
shards' quarter states and every rank gets the single-GPU logp and entropy;
the backward gives every rank the single-GPU grad_H (the shards' partial
grad_H all-gathered and merged in a fixed order) and its own rows of grad_W,
or its own columns of dL/dz, with the single-GPU bits.

Gradients come back in the inputs' dtypes: grad_H is the float32 result
rounded to H's dtype; grad_W is asked of the library in bfloat16 when W is
bfloat16 (the float32 result rounded to nearest even, the same bits as
rounding it afterwards) and in float32 otherwise.  An output the loss does not
use contributes nothing (its upstream gradient is passed as absent).
"""

from __future__ import annotations

import torch

from . import lp
from . import vocab_parallel as vp


class _LinearLogprob(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, y, temperature):
        logp, entropy, lse = lp.linear_logprob_lse(H, W, y, temperature)
        ctx.save_for_backward(H, W, y, lse, entropy)
        ctx.temperature = float(temperature)
        ctx.set_materialize_grads(False)
        return logp, entropy

    @staticmethod
    def backward(ctx, g_logp, g_entropy):
        H, W, y, lse, entropy = ctx.saved_tensors
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if (not need_h and not need_w) or (g_logp is None and g_entropy is None):
            return None, None, None, None
        gl = None if g_logp is None else g_logp.float().contiguous()
        ge = None if g_entropy is None else g_entropy.float().contiguous()
        w_dtype = torch.bfloat16 if W.dtype == torch.bfloat16 else torch.float32
        grad_h, grad_w = lp.linear_logprob_backward(
            H, W, y, gl, ge, temperature=ctx.temperature, with_grad_W=need_w,
            saved_lse=lse, saved_entropy=entropy, grad_W_dtype=w_dtype)
        grad_h = grad_h.to(H.dtype) if need_h else None
        grad_w = grad_w.to(W.dtype) if need_w else None
        return grad_h, grad_w, None, None


def linear_logprob(H: torch.Tensor, W: torch.Tensor, y: torch.Tensor,
                   temperature: float = 1.0):
    """(logp [T], entropy [T]) float32 of the fused path, differentiable in H and W
    (bf16 H [T, d] and W [V, d], int64 targets y [T])."""
    return _LinearLogprob.apply(H, W, y, temperature)


class _LogprobFromLogits(torch.autograd.Function):
    @staticmethod
    def forward(ctx, z, y, temperature):
        logp, entropy, lse = lp.logprob_from_logits_lse(z, y, temperature)
        ctx.save_for_backward(z, y, lse, entropy)
        ctx.temperature = float(temperature)
        ctx.set_materialize_grads(False)
        return logp, entropy

    @staticmethod
    def backward(ctx, g_logp, g_entropy):
        z, y, lse, entropy = ctx.saved_tensors
        if not ctx.needs_input_grad[0] or (g_logp is None and g_entropy is None):
            return None, None, None
        gl = None if g_logp is None else g_logp.float().contiguous()
        ge = None if g_entropy is None else g_entropy.float().contiguous()
        grad = lp.logprob_from_logits_backward(z, y, gl, ge, ctx.temperature, saved_lse=lse,
                                               saved_entropy=entropy)
        return grad, None, None


def logprob_from_logits(z: torch.Tensor, y: torch.Tensor, temperature: float = 1.0):
    """(logp [T], entropy [T]) float32 of the logits path, differentiable in the
    float32 logits z [T, V] (rows contiguous; int64 targets y [T]); the backward
    is lp_logprob_from_logits_backward with the forward's log Z and entropy."""
    return _LogprobFromLogits.apply(z, y, temperature)


class _VocabParallelLinearLogprob(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W_shard, y, vocab_total, group, temperature):
        logp, entropy, lse = vp.vocab_parallel_linear_logprob_lse(H, W_shard, y, vocab_total,
                                                                  group, temperature)
        ctx.save_for_backward(H, W_shard, y, lse, entropy)
        ctx.vocab_total = int(vocab_total)
        ctx.group = group
        ctx.temperature = float(temperature)
        ctx.set_materialize_grads(False)
        return logp, entropy

    @staticmethod
    def backward(ctx, g_logp, g_entropy):
        H, W_shard, y, lse, entropy = ctx.saved_tensors
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        # every rank runs the exchange of the partial grad_H, so the ranks' calls
        # stay matched whatever their own inputs need
        gl = None if g_logp is None else g_logp.float().contiguous()
        ge = None if g_entropy is None else g_entropy.float().contiguous()
        if gl is None and ge is None:
            gl = torch.zeros(H.shape[0], dtype=torch.float32, device=H.device)
        w_dtype = torch.bfloat16 if W_shard.dtype == torch.bfloat16 else torch.float32
        grad_h, grad_w = vp.vocab_parallel_linear_logprob_backward(
            H, W_shard, y, ctx.vocab_total, lse, entropy, gl, ge, ctx.group, ctx.temperature,
            with_grad_W=need_w, grad_W_dtype=w_dtype)
        grad_h = grad_h.to(H.dtype) if need_h else None
        grad_w = grad_w.to(W_shard.dtype) if need_w else None
        return grad_h, grad_w, None, None, None, None


def vocab_parallel_linear_logprob(H: torch.Tensor, W_shard: torch.Tensor, y: torch.Tensor,
                                  vocab_total: int, group=None, temperature: float = 1.0):
    """(logp [T], entropy [T]) of the fused path with W split by rows across the
    ranks of `group`, differentiable in H (every rank gets the whole,
    single-GPU grad_H) and in W_shard (its rows of grad_W); V % 64 == 0 for
    more than one rank."""
    return _VocabParallelLinearLogprob.apply(H, W_shard, y, vocab_total, group, temperature)


class _VocabParallelLogprobFromLogits(torch.autograd.Function):
    @staticmethod
    def forward(ctx, z_shard, y, vocab_total, group, temperature):
        logp, entropy, lse = vp.vocab_parallel_logprob_from_logits_lse(z_shard, y, vocab_total,
                                                                       group, temperature)
        ctx.save_for_backward(z_shard, y, lse, entropy)
        ctx.vocab_total = int(vocab_total)
        ctx.group = group
        ctx.temperature = float(temperature)
        ctx.set_materialize_grads(False)
        return logp, entropy

    @staticmethod
    def backward(ctx, g_logp, g_entropy):
        z_shard, y, lse, entropy = ctx.saved_tensors
        if not ctx.needs_input_grad[0] or (g_logp is None and g_entropy is None):
            return None, None, None, None, None
        gl = None if g_logp is None else g_logp.float().contiguous()
        ge = None if g_entropy is None else g_entropy.float().contiguous()
        grad = vp.vocab_parallel_logprob_from_logits_backward(
            z_shard, y, ctx.vocab_total, lse, entropy, gl, ge, ctx.group, ctx.temperature)
        return grad, None, None, None, None


def vocab_parallel_logprob_from_logits(z_shard: torch.Tensor, y: torch.Tensor, vocab_total: int,
                                       group=None, temperature: float = 1.0):
    """(logp [T], entropy [T]) from fp32 logits split by columns across the ranks
    of `group`, differentiable in z_shard (its columns of dL/dz; no exchange in
    the backward)."""
    return _VocabParallelLogprobFromLogits.apply(z_shard, y, vocab_total, group, temperature)
