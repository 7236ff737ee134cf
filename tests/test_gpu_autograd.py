"""The torch.autograd binding of the fused path against direct calls of the
library: forward bits, and gradients equal to lp_linear_logprob_backward's
(rounded to the inputs' bf16) for a loss on both outputs and on logp alone."""

import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from invariant_token_logprobs_gb300.autograd import linear_logprob, logprob_from_logits
from _gpu_helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _b16(t):
    return t.contiguous().view(torch.int16).cpu()


@pytest.mark.parametrize("T,tau", [(64, 1.0), (300, 0.7)])
def test_autograd_matches_direct_calls(T, tau):
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=256, V=20000, seed=11)
    g = torch.Generator(device=DEV).manual_seed(3)
    a = torch.randn(T, generator=g, device=DEV)
    b = torch.randn(T, generator=g, device=DEV)
    H = x.H.clone().requires_grad_(True)
    W = x.W.clone().requires_grad_(True)
    logp, ent = linear_logprob(H, W, x.y, tau)
    ref_lp, ref_ent, _ = lp.linear_logprob_lse(x.H, x.W, x.y, tau)
    assert torch.equal(bits(logp.detach()), bits(ref_lp))
    assert torch.equal(bits(ent.detach()), bits(ref_ent))
    ((logp * a).sum() + (ent * b).sum()).backward()
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, a, b, temperature=tau,
                                        grad_W_dtype=torch.bfloat16)
    assert H.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert torch.equal(_b16(H.grad), _b16(gH.to(torch.bfloat16)))
    assert torch.equal(_b16(W.grad), _b16(gW))


def test_autograd_logp_only_and_frozen_weight():
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV, T=48, d=256, V=8192, seed=12)
    a = torch.randn(48, generator=torch.Generator(device=DEV).manual_seed(4), device=DEV)
    H = x.H.clone().requires_grad_(True)
    logp, _ = linear_logprob(H, x.W, x.y)
    (logp * a).sum().backward()
    gH, _ = lp.linear_logprob_backward(x.H, x.W, x.y, a, None, with_grad_W=False)
    assert torch.equal(_b16(H.grad), _b16(gH.to(torch.bfloat16)))


def test_logits_autograd_matches_direct_calls():
    lp.load()
    z = synth.logits_inputs("logits_peaked", device=DEV, T=32, V=9001, seed=15)
    g = torch.Generator(device=DEV).manual_seed(5)
    a = torch.randn(32, generator=g, device=DEV)
    b = torch.randn(32, generator=g, device=DEV)
    zz = z.z.clone().requires_grad_(True)
    logp, ent = logprob_from_logits(zz, z.y, 0.7)
    ((logp * a).sum() + (ent * b).sum()).backward()
    ref = lp.logprob_from_logits_backward(z.z, z.y, a, b, temperature=0.7)
    assert torch.equal(bits(zz.grad), bits(ref))


def test_vocab_parallel_autograd_single_rank_matches_direct_calls():
    """Without a process group (one rank, the whole vocabulary) the
    vocabulary-parallel bindings give the single-GPU bindings' bits."""
    from invariant_token_logprobs_gb300.autograd import (vocab_parallel_linear_logprob,
                                                         vocab_parallel_logprob_from_logits)
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV, T=40, d=128, V=8192, seed=21)
    g = torch.Generator(device=DEV).manual_seed(6)
    a = torch.randn(40, generator=g, device=DEV)
    b = torch.randn(40, generator=g, device=DEV)
    outs = []
    for fn in (lambda H, W: linear_logprob(H, W, x.y, 0.8),
               lambda H, W: vocab_parallel_linear_logprob(H, W, x.y, 8192, None, 0.8)):
        H = x.H.clone().requires_grad_(True)
        W = x.W.clone().requires_grad_(True)
        logp, ent = fn(H, W)
        ((logp * a).sum() + (ent * b).sum()).backward()
        outs.append((logp.detach(), ent.detach(), H.grad, W.grad))
    for u, v in zip(*outs):
        assert torch.equal(u.contiguous().view(torch.int16 if u.dtype == torch.bfloat16 else torch.int32),
                           v.contiguous().view(torch.int16 if v.dtype == torch.bfloat16 else torch.int32))
    z = synth.logits_inputs("logits_peaked", device=DEV, T=24, V=5000, seed=22)
    grads = []
    for fn in (lambda zz: logprob_from_logits(zz, z.y, 0.7),
               lambda zz: vocab_parallel_logprob_from_logits(zz, z.y, 5000, None, 0.7)):
        zz = z.z.clone().requires_grad_(True)
        logp, ent = fn(zz)
        ((logp * a[:24]).sum() + (ent * b[:24]).sum()).backward()
        grads.append(zz.grad)
    assert torch.equal(bits(grads[0]), bits(grads[1]))
