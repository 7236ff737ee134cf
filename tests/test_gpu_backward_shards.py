"""Vocabulary-parallel backward of the fused path on one GB300: every shard's
partial grad_H and grad_W rows through lp_linear_logprob_partials_backward,
merged with lp_merge_grad_h_partials, against the single-GPU backward.

The bar is bit-identity, the tp4_equals_tp1 property of the RL-Kernel logprob
prior-art report (report.json, candidates.*.tp4_equals_tp1) carried to the
gradients: with 1, 2 or 4 shards of whole vocabulary quarters the merged
grad_H and the concatenated grad_W rows must be the bits of
lp_linear_logprob_backward on the same inputs and saved statistics.  That
holds by construction when V % 64 == 0 (grad_H is summed per quarter, then as
(Q0 + Q1) + (Q2 + Q3); a shard's partial is one subtree) and needs the tensor
cores to give an element the same bits wherever it sits in a tile (a shard's
grad_W rows are at other tile offsets than on one GPU).  Each shard's partial
is also checked against the fp64 oracle on its own columns, with the bound of
the single-GPU backward tests (a partial sums fewer terms).
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


def _upstream(T, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn(T, generator=g, device=DEV), torch.randn(T, generator=g, device=DEV) * 0.5


def _sharded(x, V, n, gl, ge, lse, ent, tau=1.0, dtype=torch.float32):
    parts, rows = [], []
    for i in range(n):
        b, e = lp.vocab_shard_range(V, i, n)
        ph, pw = lp.linear_logprob_partials_backward(x.H, x.W[b:e], x.y, V, i, n, lse, ent, gl,
                                                     ge, temperature=tau, grad_W_dtype=dtype)
        parts.append(ph)
        rows.append(pw)
    return parts, lp.merge_grad_h_partials(parts), torch.cat(rows)


@pytest.mark.parametrize("T,d,V,tau,dtype", [
    (64, 256, 8192, 1.0, torch.float32),
    (300, 512, 20480, 0.7, torch.float32),   # ragged row blocks, temperature
    (5, 64, 4096 + 64, 1.0, torch.bfloat16),  # the padded small batch, bf16 grad_W
    (129, 128, 64 * 1187, 1.0, torch.float32),  # quarters of 18992: not a multiple of 64
    (1100, 256, 40960, 0.8, torch.float32),  # five row blocks (ragged), the wide gradient ring
])
def test_shards_equal_single_gpu(T, d, V, tau, dtype):
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T + d)
    gl, ge = _upstream(T, T)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y, tau)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, tau, saved_lse=lse,
                                        saved_entropy=ent, grad_W_dtype=dtype)
    for n in (1, 2, 4):
        _, mH, mW = _sharded(x, V, n, gl, ge, lse, ent, tau, dtype)
        torch.cuda.synchronize()
        assert torch.equal(bits(mH), bits(gH)), (n, "grad_H")
        assert torch.equal(bits(mW), bits(gW)), (n, "grad_W")


def test_shard_partials_against_oracle():
    """Each shard's partial grad_H = G[:, shard] W_shard and its grad_W rows,
    against the fp64 oracle's G restricted to the shard's columns."""
    T, d, V = 96, 192, 8192 + 64
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=31)
    gl, ge = _upstream(T, 32)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    h = x.H.float().cpu().numpy().astype(np.float64)
    w = x.W.float().cpu().numpy().astype(np.float64)
    y = x.y.cpu().numpy()
    G = olp.selected_logprob_grad_logits(olp.linear_logits(h, w), y, gl.double().cpu().numpy(),
                                         ge.double().cpu().numpy())
    for n in (2, 4):
        parts, _, rows = _sharded(x, V, n, gl, ge, lse, ent)
        torch.cuda.synchronize()
        for i in range(n):
            b, e = lp.vocab_shard_range(V, i, n)
            ref = G[:, b:e] @ w[b:e]
            bound = (2.0 ** -8 + ((e - b) / 7 + 9) * 2.0 ** -24) * (np.abs(G[:, b:e]) @ np.abs(w[b:e])) + 1e-6
            err = np.abs(parts[i].double().cpu().numpy() - ref)
            assert np.all(err <= bound), (n, i, float((err / bound).max()))
        ref_w = G.T @ h
        bound_w = (2.0 ** -8 + T * 2.0 ** -24) * (np.abs(G).T @ np.abs(h)) + 1e-6
        err_w = np.abs(rows.double().cpu().numpy() - ref_w)
        assert np.all(err_w <= bound_w), (n, float((err_w / bound_w).max()))


def test_headline_shape_shards_equal_single_gpu():
    """T = 512, d = 4096, V = 151936 (the fused_qwen3_8b head), 2 and 4 shards."""
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    V = x.W.shape[0]
    gl, ge = _upstream(512, 7)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, saved_lse=lse, saved_entropy=ent)
    for n in (2, 4):
        _, mH, mW = _sharded(x, V, n, gl, ge, lse, ent)
        torch.cuda.synchronize()
        assert torch.equal(bits(mH), bits(gH)), n
        assert torch.equal(bits(mW), bits(gW)), n
        del mH, mW


def test_one_shard_is_the_single_gpu_call_for_any_vocabulary():
    """n_shards = 1 is the plain backward, also when V % 64 != 0 (whose grad_H is
    summed over 19 ranges of the whole vocabulary); more shards are refused there."""
    T, d, V = 40, 128, 5003
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=9)
    gl, ge = _upstream(T, 10)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, saved_lse=lse, saved_entropy=ent)
    pH, pW = lp.linear_logprob_partials_backward(x.H, x.W, x.y, V, 0, 1, lse, ent, gl, ge)
    torch.cuda.synchronize()
    assert torch.equal(bits(pH), bits(gH)) and torch.equal(bits(pW), bits(gW))
    b, e = lp.vocab_shard_range(V, 0, 2)
    with pytest.raises(lp.LpError):
        lp.linear_logprob_partials_backward(x.H, x.W[b:e], x.y, V, 0, 2, lse, ent, gl, ge)


def test_merge_in_place_and_without_grad_W():
    T, d, V = 64, 256, 8192
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=12)
    gl, ge = _upstream(T, 13)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    parts, merged, _ = _sharded(x, V, 4, gl, ge, lse, ent)
    no_w = []
    for i in range(4):
        b, e = lp.vocab_shard_range(V, i, 4)
        ph, pw = lp.linear_logprob_partials_backward(x.H, x.W[b:e], x.y, V, i, 4, lse, ent, gl,
                                                     ge, with_grad_W=False)
        assert pw is None
        no_w.append(ph)
    for a, c in zip(parts, no_w):
        assert torch.equal(bits(a), bits(c))
    lp.lp_merge_grad_h_partials(no_w, no_w[0])  # the output is partial 0
    torch.cuda.synchronize()
    assert torch.equal(bits(no_w[0]), bits(merged))


@pytest.mark.parametrize("T,V", [(20, 64), (33, 192), (17, 320), (3, 128)])
def test_tiny_quarters(T, V):
    """Quarters of 16 to 80 columns (one to five 16-deep MMA steps, at most two K
    blocks), shards of a few W rows: 1, 2 and 4 shards against the single-GPU
    backward, and the single-GPU backward against the fp64 oracle."""
    d = 64
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T * V)
    gl, ge = _upstream(T, T + V)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, saved_lse=lse, saved_entropy=ent)
    for n in (1, 2, 4):
        _, mH, mW = _sharded(x, V, n, gl, ge, lse, ent)
        torch.cuda.synchronize()
        assert torch.equal(bits(mH), bits(gH)), n
        assert torch.equal(bits(mW), bits(gW)), n
    h = x.H.float().cpu().numpy().astype(np.float64)
    w = x.W.float().cpu().numpy().astype(np.float64)
    G = olp.selected_logprob_grad_logits(olp.linear_logits(h, w), x.y.cpu().numpy(),
                                         gl.double().cpu().numpy(), ge.double().cpu().numpy())
    bound_h = (2.0 ** -8 + (V / 7 + 9) * 2.0 ** -24) * (np.abs(G) @ np.abs(w)) + 1e-6
    assert np.all(np.abs(gH.double().cpu().numpy() - G @ w) <= bound_h)
    bound_w = (2.0 ** -8 + T * 2.0 ** -24) * (np.abs(G).T @ np.abs(h)) + 1e-6
    assert np.all(np.abs(gW.double().cpu().numpy() - G.T @ h) <= bound_w)
