"""Temperature-scaled logprobs (softmax(z / tau)) on a GB300, through the C ABI.

Oracle: the fp64 definition applied to z / tau.  The library never rounds a
scaled logit: maxima are taken over the raw logits, each difference z - m is
multiplied by 1/tau (on the logits path as a float pair, so the rounding of
1/tau does not bias every term alike) and the target enters as (t - M) / tau
in float64.  So the logits-given path keeps its unscaled bounds (2e-6 on logp,
1e-5 on entropy) at any tau, and the fused path its 1e-4.  Every invariance of
the unscaled path must hold at a fixed tau, and tau = 1 must give exactly the
unscaled bits.
"""

import numpy as np
import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import (FUSED_TOL, LOGITS_ENT_TOL, LOGITS_LOGP_TOL, bits, excess_over_rounding,
                          max_err, oracle_fused, oracle_logits)

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lp.load()


def _tau32(tau: float) -> float:
    """The temperature the library receives: the C ABI takes it as a float."""
    return float(np.float32(tau))


def _oracle_logits_t(z, y, tau, rows=None):
    zz = z if rows is None else z[rows]
    yy = y if rows is None else y[rows]
    return oracle.selected_logprob(zz.double().cpu().numpy(), yy.cpu().numpy(),
                                   temperature=_tau32(tau))


@pytest.mark.parametrize("tau", [0.7, 1.6])
@pytest.mark.parametrize("T,V", [(64, 8192), (37, 1001), (4, 3)])
def test_logits_temperature_all_rows(tau, T, V):
    x = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=200 + V)
    logp, ent = lp.logprob_from_logits(x.z, x.y, temperature=tau)
    r_lp, r_ent = _oracle_logits_t(x.z, x.y, tau)
    assert max_err(logp, r_lp) <= LOGITS_LOGP_TOL and max_err(ent, r_ent) <= LOGITS_ENT_TOL


@pytest.mark.parametrize("tau", [0.7, 1.6])
def test_logits_temperature_full_size_all_rows(tau):
    x = synth.logits_inputs("logits_peaked", device=DEV)
    logp, ent = lp.logprob_from_logits(x.z, x.y, temperature=tau)
    r_lp, r_ent = _oracle_logits_t(x.z, x.y, tau)
    e1, e2 = max_err(logp, r_lp), max_err(ent, r_ent)
    ex = excess_over_rounding(logp, r_lp)
    print(f"peaked tau={tau}: logp err {e1:.3e} (beyond output rounding {ex:.3e}), "
          f"entropy err {e2:.3e}")
    assert e1 <= LOGITS_LOGP_TOL and e2 <= LOGITS_ENT_TOL
    assert ex <= 1e-7


def test_temperature_one_is_bitwise_unscaled():
    x = synth.logits_inputs("logits_peaked", device=DEV, T=96, V=20000, seed=9)
    a = lp.logprob_from_logits(x.z, x.y)
    b = lp.logprob_from_logits(x.z, x.y, temperature=1.0)
    assert torch.equal(bits(a[0]), bits(b[0])) and torch.equal(bits(a[1]), bits(b[1]))
    f = synth.fused_inputs("fused_tiny", device=DEV)
    c = lp.linear_logprob(f.H, f.W, f.y)
    d = lp.linear_logprob(f.H, f.W, f.y, temperature=1.0)
    assert torch.equal(bits(c[0]), bits(d[0])) and torch.equal(bits(c[1]), bits(d[1]))


def test_logits_temperature_shards_and_offsets_bitwise():
    V = 151936
    x = synth.logits_inputs("logits_peaked", device=DEV, T=48, V=V, seed=31)
    ref = lp.logprob_from_logits(x.z, x.y, temperature=0.7)
    for n in (2, 4):
        parts = []
        for i in range(n):
            b, e = lp.vocab_shard_range(V, i, n)
            parts.append(lp.logprob_partials_from_logits(x.z[:, b:e], x.y, V, i, n, temperature=0.7))
        m = lp.merge_partials(parts)
        assert torch.equal(bits(m[0]), bits(ref[0])) and torch.equal(bits(m[1]), bits(ref[1]))
    idx = torch.tensor([47, 3, 20], device=DEV)
    sub = lp.logprob_from_logits(x.z[idx].contiguous(), x.y[idx], temperature=0.7)
    assert torch.equal(bits(sub[0]), bits(ref[0][idx])) and torch.equal(bits(sub[1]), bits(ref[1][idx]))


@pytest.mark.parametrize("tau", [0.7, 1.6])
def test_fused_temperature_all_rows(tau):
    x = synth.fused_inputs("fused_tiny", device=DEV)
    logp, ent = lp.linear_logprob(x.H, x.W, x.y, temperature=tau)
    r = oracle.linear_selected_logprob(x.H.float().cpu().numpy(), x.W.float().cpu().numpy(),
                                       x.y.cpu().numpy(), temperature=_tau32(tau))
    assert max_err(logp, r[0]) <= FUSED_TOL and max_err(ent, r[1]) <= FUSED_TOL


def test_fused_temperature_qwen3_8b_sampled_rows_and_shards():
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    V = x.W.shape[0]
    logp, ent = lp.linear_logprob(x.H, x.W, x.y, temperature=0.7)
    rows = torch.tensor([0, 129, 255, 256, 511])
    w_host = x.W.float().cpu().numpy()
    r = oracle.linear_selected_logprob(x.H[rows].float().cpu().numpy(), w_host,
                                       x.y[rows].cpu().numpy(), temperature=_tau32(0.7))
    e1, e2 = max_err(logp[rows], r[0]), max_err(ent[rows], r[1])
    print(f"qwen3-8b head tau=0.7: logp err {e1:.3e}, entropy err {e2:.3e}")
    assert e1 <= FUSED_TOL and e2 <= FUSED_TOL
    parts = []
    for i in range(4):
        b, e = lp.vocab_shard_range(V, i, 4)
        parts.append(lp.linear_logprob_partials(x.H, x.W[b:e], x.y, V, i, 4, temperature=0.7))
    m = lp.merge_partials(parts)
    assert torch.equal(bits(m[0]), bits(logp)) and torch.equal(bits(m[1]), bits(ent))
    sub = lp.linear_logprob(x.H[100:300].contiguous(), x.W, x.y[100:300], temperature=0.7)
    assert torch.equal(bits(sub[0]), bits(logp[100:300])) and torch.equal(bits(sub[1]), bits(ent[100:300]))
