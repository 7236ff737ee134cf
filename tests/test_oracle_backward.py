"""Pins for the fp64 oracle of the backward pass (CPU only).

The gradients are pinned to the derivative's definition: central finite
differences of the forward oracle's loss L = sum g_logp logp + g_ent entropy,
in float64 on tiny shapes (step 1e-5, expected agreement ~1e-8).  Closed
forms: the rows of dL/dz sum to zero (probabilities sum to one), and identical
W rows give dL/dH = 0.  Planted mistakes (sign of the entropy term, missing
one-hot, transposed dW, missing temperature factor) must each fail a pin.
"""

import types

import numpy as np
import pytest

from oracle import logprob as olp


def _loss(h, w, y, gl, ge, tau):
    lp, ent = olp.linear_selected_logprob(h, w, y, temperature=tau)
    return float(np.sum(gl * lp) + np.sum(ge * ent))


def _setup(seed=0, T=3, d=5, V=7):
    rng = np.random.default_rng(seed)
    h = rng.normal(0, 1, size=(T, d))
    w = rng.normal(0, 0.7, size=(V, d))
    y = rng.integers(0, V, size=T)
    gl = rng.normal(0, 1, size=T)
    ge = rng.normal(0, 1, size=T)
    return h, w, y, gl, ge


def pin_finite_differences(bwd):
    for tau in (1.0, 0.7):
        h, w, y, gl, ge = _setup(seed=int(tau * 10))
        dh, dw = bwd(h, w, y, gl, ge, tau)
        eps = 1e-5
        for arr, grad in ((h, dh), (w, dw)):
            num = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                old = arr[idx]
                arr[idx] = old + eps
                lp_ = _loss(h, w, y, gl, ge, tau)
                arr[idx] = old - eps
                lm_ = _loss(h, w, y, gl, ge, tau)
                arr[idx] = old
                num[idx] = (lp_ - lm_) / (2 * eps)
            assert np.max(np.abs(num - grad)) < 1e-7, (tau, np.max(np.abs(num - grad)))


def pin_closed_forms(bwd):
    h, w, y, gl, ge = _setup(seed=3, T=4, d=6, V=9)
    g = olp.selected_logprob_grad_logits(olp.linear_logits(h, w), y, gl, ge)
    assert np.max(np.abs(g.sum(axis=1))) < 1e-12
    w_same = np.repeat(w[:1], 9, axis=0)
    dh, dw = bwd(h, w_same, y, gl, ge, 1.0)
    assert np.max(np.abs(dh)) < 1e-12


PINS = [pin_finite_differences, pin_closed_forms]


def _oracle_bwd(h, w, y, gl, ge, tau):
    return olp.linear_selected_logprob_backward(h, w, y, gl, ge, temperature=tau)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_backward_pin(pin):
    pin(_oracle_bwd)


def _mutant(kind):
    def bwd(h, w, y, gl, ge, tau):
        g = olp.selected_logprob_grad_logits(olp.linear_logits(h, w), y, gl,
                                             -ge if kind == "ent_sign" else ge, tau)
        if kind == "no_onehot":
            g = g.copy()
            g[np.arange(len(y)), y] -= gl / tau
        if kind == "no_tau":
            g = g * tau
        dh = g @ np.asarray(w, dtype=np.float64)
        dw = g.T @ np.asarray(h, dtype=np.float64)
        if kind == "dw_from_dh":
            dw = (g @ np.asarray(w, dtype=np.float64)).sum() * np.ones_like(dw)
        return dh, dw
    return bwd


@pytest.mark.parametrize("kind", ["ent_sign", "no_onehot", "no_tau", "dw_from_dh"])
def test_backward_pins_catch_planted_mistakes(kind):
    caught = False
    for pin in PINS:
        try:
            pin(_mutant(kind))
        except AssertionError:
            caught = True
    assert caught, kind


def test_grad_logits_matches_finite_differences_of_logits_path():
    rng = np.random.default_rng(8)
    z = rng.normal(0, 2, size=(3, 11))
    y = np.array([2, 10, 0])
    gl = rng.normal(0, 1, size=3)
    ge = rng.normal(0, 1, size=3)
    g = olp.selected_logprob_grad_logits(z, y, gl, ge)
    eps = 1e-6
    for idx in np.ndindex(z.shape):
        zp = z.copy(); zp[idx] += eps
        zm = z.copy(); zm[idx] -= eps
        a = olp.selected_logprob(zp, y); b = olp.selected_logprob(zm, y)
        num = (np.sum(gl * (a[0] - b[0])) + np.sum(ge * (a[1] - b[1]))) / (2 * eps)
        assert abs(num - g[idx]) < 1e-7
