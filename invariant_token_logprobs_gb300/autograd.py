"""torch.autograd bindings of the fused path and of the logits path.

    logp, entropy = linear_logprob(H, W, y, temperature=1.0)
    logp, entropy = logprob_from_logits(z, y, temperature=1.0)

returns the selected-token log-probabilities and entropies of z = H W^T / tau
(lp_linear_logprob_lse) and back-propagates into H and W through
lp_linear_logprob_backward with the forward's log Z and entropy kept, so the
backward does not recompute them.  This is argument marshalling only: every
step runs in liblp's kernels, on the current stream.

Gradients come back in the inputs' dtypes: grad_H is the float32 result
rounded to H's dtype; grad_W is asked of the library in bfloat16 when W is
bfloat16 (the float32 result rounded to nearest even, the same bits as
rounding it afterwards) and in float32 otherwise.  An output the loss does not
use contributes nothing (its upstream gradient is passed as absent).
"""

from __future__ import annotations

import torch

from . import lp


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
