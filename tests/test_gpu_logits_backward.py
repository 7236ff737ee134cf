"""The logits-path backward (lp_logprob_from_logits_backward) on a GB300 against
the fp64 oracle's dL/dz, through the C ABI.

Bound per element, from the arithmetic: the kernel forms log p = z/tau - log Z
in float32 from the forward's float32 log Z (within ~2e-6 of the true value at
|log p| < 32, its own rounding included) and p with the hardware 2^x (relative
error < 2^-22), so p and log p + entropy carry a relative / absolute error of
at most ~4e-6; with a factor of 2.5 on that,
    |G - G_ref| <= 1e-5 * p * (|g_logp| + |g_ent| (|log p| + |entropy| + 1))
                   + 1e-6 * |G_ref| + 1e-30.
Bitwise checks: a row's gradient does not depend on the batch or the row
stride; log-probabilities and entropies of the forward with log Z are the bits
of the plain logits-path call.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lp.load()


def _tau32(tau):
    return float(np.float32(tau))


def _upstream(T, seed, with_logp=True, with_ent=True):
    g = torch.Generator(device=DEV).manual_seed(seed)
    gl = torch.randn(T, generator=g, device=DEV) if with_logp else None
    ge = torch.randn(T, generator=g, device=DEV) if with_ent else None
    return gl, ge


def _check_rows(z, y, gl, ge, tau, grad, rows):
    zc = z[rows].double().cpu().numpy()
    yc = y[rows].cpu().numpy()
    glc = np.zeros(len(yc)) if gl is None else gl[rows].double().cpu().numpy()
    gec = None if ge is None else ge[rows].double().cpu().numpy()
    ref = oracle.selected_logprob_grad_logits(zc, yc, glc, gec, _tau32(tau))
    # p, log p and the entropy of the same rows, for the bound
    zs = zc / _tau32(tau)
    log_z = oracle.logsumexp_rows(zs)
    log_p = zs - log_z[:, None]
    p = np.exp(log_p)
    with np.errstate(invalid="ignore"):
        ent = -np.where(p > 0.0, p * log_p, 0.0).sum(axis=1)
    ge_abs = np.zeros(len(yc)) if gec is None else np.abs(gec)
    with np.errstate(invalid="ignore"):
        scale = np.abs(glc)[:, None] + ge_abs[:, None] * (np.abs(log_p) + np.abs(ent)[:, None] + 1.0)
        bound = 1e-5 * np.where(p > 0.0, p * scale, 0.0) + 1e-6 * np.abs(ref) + 1e-30
    got = grad[rows].double().cpu().numpy()
    excess = np.abs(got - ref) - bound
    assert np.all(excess <= 0.0), float(np.max(excess))


@pytest.mark.parametrize("T,V,tau", [(7, 1000, 1.0), (33, 4099, 0.7), (64, 8192 + 37, 1.6)])
def test_small_shapes_against_oracle(T, V, tau):
    z = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=5)
    gl, ge = _upstream(T, 6)
    grad = lp.logprob_from_logits_backward(z.z, z.y, gl, ge, temperature=tau)
    torch.cuda.synchronize()
    _check_rows(z.z, z.y, gl, ge, tau, grad, slice(None))


@pytest.mark.parametrize("with_logp,with_ent", [(True, False), (False, True)])
def test_one_upstream_gradient(with_logp, with_ent):
    z = synth.logits_inputs("logits_peaked", device=DEV, T=16, V=3001, seed=7)
    gl, ge = _upstream(16, 8, with_logp, with_ent)
    grad = lp.logprob_from_logits_backward(z.z, z.y, gl, ge)
    torch.cuda.synchronize()
    _check_rows(z.z, z.y, gl, ge, 1.0, grad, slice(None))


def test_bad_targets_and_minus_infinity():
    z = synth.logits_inputs("logits_peaked", device=DEV, T=6, V=513, seed=9)
    y = z.y.clone()
    y[1] = -1
    y[2] = 513
    zz = z.z.clone()
    zz[3, ::7] = -math.inf
    gl, ge = _upstream(6, 10)
    grad = lp.logprob_from_logits_backward(zz, y, gl, ge)
    torch.cuda.synchronize()
    assert torch.all(grad[3, ::7] == 0)
    assert torch.isfinite(grad).all()
    _check_rows(zz, y, gl, ge, 1.0, grad, slice(None))


def test_row_stride_and_batch_do_not_change_bits():
    z = synth.logits_inputs("logits_peaked", device=DEV, T=40, V=5003, seed=11)
    gl, ge = _upstream(40, 12)
    full = lp.logprob_from_logits_backward(z.z, z.y, gl, ge)
    # unaligned row strides for the logits and for the gradient
    wide = torch.zeros(40, 5003 + 2, device=DEV)  # rows 4 bytes past 16-byte alignment
    wide[:, :5003] = z.z
    zs = wide[:, :5003]
    _, ent, lse = lp.logprob_from_logits_lse(zs, z.y)
    gbuf = torch.zeros(40, 5003 + 3, device=DEV)  # rows 8 bytes past alignment
    lp.lp_logprob_from_logits_backward(zs, z.y, 1.0, lse, ent, gl, ge, gbuf[:, :5003])
    assert torch.equal(bits(gbuf[:, :5003].contiguous()), bits(full))
    # a slice of rows alone
    sub = slice(9, 23)
    part = lp.logprob_from_logits_backward(z.z[sub].contiguous(), z.y[sub].contiguous(),
                                           gl[sub].contiguous(), ge[sub].contiguous())
    assert torch.equal(bits(part), bits(full[sub].contiguous()))


def test_forward_with_lse_matches_plain_call():
    z = synth.logits_inputs("logits_peaked", device=DEV, T=64, V=20000, seed=13)
    for tau in (1.0, 0.7):
        logp, ent, lse = lp.logprob_from_logits_lse(z.z, z.y, tau)
        ref_lp, ref_ent = lp.logprob_from_logits(z.z, z.y, temperature=tau)
        assert torch.equal(bits(logp), bits(ref_lp)) and torch.equal(bits(ent), bits(ref_ent))
        ref_lse = oracle.logsumexp_rows(z.z.double().cpu().numpy() / _tau32(tau))
        assert np.max(np.abs(lse.double().cpu().numpy() - ref_lse)) <= 4e-6


def test_full_size_peaked_sampled_rows():
    z = synth.logits_inputs("logits_peaked", device=DEV)
    T = z.z.shape[0]
    gl, ge = _upstream(T, 14)
    logp, ent, lse = lp.logprob_from_logits_lse(z.z, z.y)
    grad = lp.logprob_from_logits_backward(z.z, z.y, gl, ge, saved_lse=lse, saved_entropy=ent)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 257, 511, 512, 777, 1022, 1023])
    _check_rows(z.z, z.y, gl, ge, 1.0, grad, rows)
