"""Backward of the fused path on a GB300: grad_H and grad_W against the fp64
oracle, determinism, and row invariance of grad_H.

Tolerance (from the arithmetic): the kernel forms G = dL/dz in fp32 and rounds
it to bf16 before two tensor-core products with fp32 accumulation.  bf16 keeps
8 significant bits, so its round-to-nearest error is at most 2^-8 relative
(the unit roundoff of an 8-bit significand); a product term G[t,v] X[.,k] then
carries at most 2^-8 |G X| of error.  The products add at most about
n 2^-24 sum |terms| for n terms summed in one fp32 chain: grad_H = G W sums
V terms in 19 fixed ranges (n = V/19 + 19), or, when V % 64 == 0, in 7 ranges
per quarter added in order and then as (Q0 + Q1) + (Q2 + Q3) (n = V/28 + 9,
below V/19 + 19); grad_W = G^T H sums T terms (n = T).  So the tests allow (2^-8 + n 2^-24) sum |G X| + 1e-6 per element,
the sums taken in fp64 from the oracle's G.  These are absolute-sum bounds:
they hold also where the terms cancel (the entropy-only gradient, whose rows
of G sum to zero).  A bf16 grad_W must be the fp32 grad_W of the same call
rounded to nearest even, bit for bit.
"""

import numpy as np
import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import bits

from oracle import logprob as olp

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lp.load()


def _upstream(T, seed, with_logp=True, with_ent=True):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    gl = torch.randn(T, generator=g, device=DEV) if with_logp else None
    ge = torch.randn(T, generator=g, device=DEV) * 0.5 if with_ent else None
    return gl, ge


def _np(t):
    return None if t is None else t.double().cpu().numpy()


def _check_against_oracle(x, gl, ge, tau, gH, gW, rows=None, w_cols=97):
    h = x.H.float().cpu().numpy().astype(np.float64)
    w = x.W.float().cpu().numpy().astype(np.float64)
    y = x.y.cpu().numpy()
    T = h.shape[0]
    gl_np = np.zeros(T) if gl is None else _np(gl)
    ge_np = np.zeros(T) if ge is None else _np(ge)
    z = np.empty((T, w.shape[0]))
    for v0 in range(0, w.shape[0], 8192):
        z[:, v0:v0 + 8192] = olp.linear_logits(h, w[v0:v0 + 8192])
    G = olp.selected_logprob_grad_logits(z, y, gl_np, ge_np, temperature=tau)
    del z
    r = np.arange(T) if rows is None else np.asarray(rows)
    ref_h = G[r] @ w
    bound_h = (2.0 ** -8 + (w.shape[0] / 19 + 19) * 2.0 ** -24) * (np.abs(G[r]) @ np.abs(w)) + 1e-6
    got_h = gH[torch.as_tensor(r)].double().cpu().numpy()
    err_h = np.abs(got_h - ref_h)
    assert np.all(err_h <= bound_h), (float(err_h.max()), float((err_h / bound_h).max()))
    out = {"grad_H_max_err": float(err_h.max()), "grad_H_max_ratio": float((err_h / bound_h).max())}
    if gW is not None:
        spread = np.arange(0, w.shape[0], max(1, w.shape[0] // w_cols))
        targets = y[(y >= 0) & (y < w.shape[0])]
        vs = np.unique(np.concatenate([spread, targets if w_cols > 97 else targets[:16]]))
        ref_w = G[:, vs].T @ h
        bound_w = (2.0 ** -8 + T * 2.0 ** -24) * (np.abs(G[:, vs]).T @ np.abs(h)) + 1e-6
        got_w = gW[torch.as_tensor(vs)].double().cpu().numpy()
        err_w = np.abs(got_w - ref_w)
        assert np.all(err_w <= bound_w), (float(err_w.max()), float((err_w / bound_w).max()))
        out["grad_W_max_err"] = float(err_w.max())
        out["grad_W_max_ratio"] = float((err_w / bound_w).max())
        out["grad_W_columns"] = int(vs.size)
    return out


@pytest.mark.parametrize("T,d,V,tau", [(64, 256, 8192, 1.0), (37, 72, 1001, 0.7),
                                       (300, 128, 20003, 1.0), (1, 64, 512, 1.6),
                                       (600, 136, 5003, 1.0), (513, 64, 3000, 0.9),
                                       (9, 64, 3, 1.0), (20, 72, 1, 1.0)])
def test_backward_small_against_oracle(T, d, V, tau):
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T + V)
    gl, ge = _upstream(T, seed=T)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, temperature=tau)
    torch.cuda.synchronize()
    _check_against_oracle(x, gl, ge, tau, gH, gW)


@pytest.mark.parametrize("T", [5, 40])
def test_backward_hidden_size_not_a_multiple_of_8(T):
    """d = 60 with H and W rows at a stride of 64 (their padding holds ones,
    which must not be read); T = 5 goes through the padded small-batch path."""
    d, V = 60, 777
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=8)
    Hs = torch.ones((T, 64), dtype=x.H.dtype, device=DEV)
    Ws = torch.ones((V, 64), dtype=x.W.dtype, device=DEV)
    Hs[:, :d] = x.H
    Ws[:, :d] = x.W
    gl, ge = _upstream(T, seed=T + 1)
    gH, gW = lp.linear_logprob_backward(Hs[:, :d], Ws[:, :d], x.y, gl, ge, temperature=0.8)
    torch.cuda.synchronize()
    _check_against_oracle(x, gl, ge, 0.8, gH, gW)


def test_backward_one_upstream_and_bad_targets():
    x = synth.fused_inputs("fused_tiny", device=DEV, T=40, d=128, V=5000, seed=12)
    x.y[3] = -1
    x.y[7] = 5000
    gl, ge = _upstream(40, seed=5)
    for a, b in ((gl, None), (None, ge)):
        gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, a, b)
        torch.cuda.synchronize()
        _check_against_oracle(x, a, b, 1.0, gH, gW)
    gH, none = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, with_grad_W=False)
    assert none is None and torch.isfinite(gH).all()


def test_backward_qwen3_8b_head_all_rows():
    """The headline shape: every row of grad_H, and 1024 spread columns of
    grad_W plus every target column."""
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    gl, ge = _upstream(512, seed=2)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
    torch.cuda.synchronize()
    out = _check_against_oracle(x, gl, ge, 1.0, gH, gW, w_cols=1024)
    print(f"qwen3-8b head backward: {out}")


def test_backward_qwen3_8b_head_entropy_only():
    """Entropy gradient alone: every row of G sums to zero (heavy cancellation
    in both products); the absolute-sum bound must still hold."""
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    _, ge = _upstream(512, seed=3, with_logp=False)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, None, ge)
    torch.cuda.synchronize()
    out = _check_against_oracle(x, None, ge, 1.0, gH, gW, w_cols=1024)
    print(f"qwen3-8b head backward, entropy only: {out}")


@pytest.mark.parametrize("T,d,V", [(300, 128, 20003), (5, 64, 3001), (512, 4096, 151936)])
def test_backward_bf16_grad_W_is_rounded_fp32(T, d, V):
    """grad_W in bf16 holds the fp32 results of the same products rounded to
    nearest even; grad_H is unchanged."""
    spec = "fused_qwen3_8b" if d == 4096 else "fused_tiny"
    x = synth.fused_inputs(spec, device=DEV, T=T, d=d, V=V, seed=T + 1)
    gl, ge = _upstream(T, seed=11)
    h32, w32 = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
    h16, w16 = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, grad_W_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert w16.dtype == torch.bfloat16
    assert torch.equal(bits(h16.reshape(-1)), bits(h32.reshape(-1)))
    assert torch.equal(w16.view(torch.int16), w32.to(torch.bfloat16).view(torch.int16))


def test_backward_with_saved_forward_statistics():
    """Entropy and log-sum-exp kept from the forward give the same bits as the
    backward's own recomputation."""
    x = synth.fused_inputs("fused_tiny", device=DEV, T=200, d=256, V=30000, seed=14)
    gl, ge = _upstream(200, seed=3)
    for tau in (1.0, 0.7):
        logp, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y, temperature=tau)
        ref_lp, ref_ent = lp.linear_logprob(x.H, x.W, x.y, temperature=tau)
        assert torch.equal(bits(logp), bits(ref_lp)) and torch.equal(bits(ent), bits(ref_ent))
        z = olp.linear_logits(x.H.float().cpu().numpy(), x.W.float().cpu().numpy()) / tau
        lse_ref = olp.logsumexp_rows(z)
        assert float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref))) <= 1e-4
        a = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, temperature=tau)
        b = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, temperature=tau, saved_lse=lse,
                                       saved_entropy=ent)
        assert torch.equal(bits(a[0].reshape(-1)), bits(b[0].reshape(-1)))
        assert torch.equal(bits(a[1].reshape(-1)), bits(b[1].reshape(-1)))


def test_backward_grid_size_invariant():
    """The backward's results do not depend on the persistent grid size."""
    x = synth.fused_inputs("fused_tiny", device=DEV, T=300, d=256, V=30000, seed=6)
    gl, ge = _upstream(300, seed=4)
    ref_h, ref_w = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
    try:
        for limit in (2, 16, 50):
            lp.lp_set_persistent_grid_limit(limit)
            h, w = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
            torch.cuda.synchronize()
            assert torch.equal(bits(h.reshape(-1)), bits(ref_h.reshape(-1))), limit
            assert torch.equal(bits(w.reshape(-1)), bits(ref_w.reshape(-1))), limit
    finally:
        lp.lp_set_persistent_grid_limit(0)


def test_backward_deterministic_and_row_invariant():
    x = synth.fused_inputs("fused_tiny", device=DEV, T=300, d=256, V=30000, seed=4)
    gl, ge = _upstream(300, seed=9)
    ref_h, ref_w = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
    for _ in range(3):
        h, w = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
        assert torch.equal(bits(h.reshape(-1)), bits(ref_h.reshape(-1)))
        assert torch.equal(bits(w.reshape(-1)), bits(ref_w.reshape(-1)))
    # rows of grad_H depend only on their own inputs
    sub = slice(100, 140)
    h_sub, _ = lp.linear_logprob_backward(x.H[sub].contiguous(), x.W, x.y[sub],
                                          gl[sub].contiguous(), ge[sub].contiguous(),
                                          with_grad_W=False)
    assert torch.equal(bits(h_sub.reshape(-1)), bits(ref_h[sub].reshape(-1)))
