"""Pins for the fp64 oracle: closed forms, worked examples, brute force,
invariants and planted mistakes.  CPU only.

The oracle must be pinned to something other than itself before the CUDA
path is checked against it.  Each ``pin_*`` below takes an implementation (the oracle, or a
copy with a planted mistake) and raises AssertionError when it disagrees with
mathematics fixed independently of the oracle's own formula:

* closed forms for uniform rows, one dominant logit and k equal peaks (the
  structure of the peaked-logits workload), evaluated with mpmath at 50 digits;
* hand-derived worked examples (``tests/golden/worked_examples.json``);
* brute force with mpmath on tiny rows, with no max-shift at all;
* exact rational dot products for the LM-head projection;
* invariants: normalisation, shift invariance, bounds, -inf/NaN rules.

``test_pins_catch_planted_mistakes`` plants plausible mistakes in copies of the
oracle (dropped shift, wrong sign, wrong index, transposed operand, dropped
term, wrong axis, wrong log base) and checks that at least one pin fails for
each.
"""

from __future__ import annotations

import json
import math
import os
import types
from fractions import Fraction

import mpmath
import numpy as np
import pytest

import oracle
from oracle import logprob as olp

mpmath.mp.dps = 50
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _impl_from_module():
    return types.SimpleNamespace(
        selected_logprob=olp.selected_logprob,
        linear_logits=olp.linear_logits,
        linear_selected_logprob=olp.linear_selected_logprob,
    )


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def _close(a, b, tol, what):
    a = float(a)
    b = float(b)
    if math.isinf(b):
        assert a == b, f"{what}: {a} != {b}"
        return
    assert abs(a - b) <= tol * max(1.0, abs(b)), f"{what}: {a!r} vs {b!r}"


def pin_uniform(impl):
    """All logits equal: logp = -ln V, entropy = ln V, for any common value."""
    for V in (1, 2, 7, 8192, 151936):
        cs = np.array([0.0, -3.5, 1000.0, -1000.0])
        z = np.repeat(cs[:, None], V, axis=1)
        y = np.array([0, V - 1, V // 2, V // 3])
        logp, ent = impl.selected_logprob(z, y)
        lnv = mpmath.log(V)
        for i in range(len(cs)):
            _close(logp[i], -lnv, 1e-13, f"uniform logp V={V} c={cs[i]}")
            _close(ent[i], lnv, 1e-13, f"uniform entropy V={V} c={cs[i]}")


def _dominant_expect(V, delta, k=1):
    """k columns at delta, V-k at 0: Z' = k e^delta + V - k."""
    V = mpmath.mpf(V)
    k = mpmath.mpf(k)
    d = mpmath.mpf(delta)
    zp = k * mpmath.e ** d + V - k
    logp_peak = d - mpmath.log(zp)
    logp_other = -mpmath.log(zp)
    ent = mpmath.log(zp) - k * d * mpmath.e ** d / zp
    return logp_peak, logp_other, ent


def pin_dominant(impl):
    """One logit raised by delta over V-1 equal ones."""
    for V in (2, 10, 8192):
        for delta in (0.5, 5.0, 40.0):
            for c in (0.0, -2.0, 300.0):
                z = np.full((2, V), c)
                yp = V // 3
                z[:, yp] += delta
                y = np.array([yp, (yp + 1) % V])
                logp, ent = impl.selected_logprob(z, y)
                lp_peak, lp_other, e = _dominant_expect(V, delta)
                _close(logp[0], lp_peak, 1e-12, f"dominant logp V={V} d={delta}")
                _close(logp[1], lp_other, 1e-12, f"dominant other V={V} d={delta}")
                _close(ent[0], e, 1e-11, f"dominant entropy V={V} d={delta}")
                _close(ent[1], e, 1e-11, f"dominant entropy V={V} d={delta}")


def pin_k_peaks(impl):
    """k distinct columns raised by delta (the peaked-logits structure)."""
    V, k, delta = 151936, 8, 12.0
    rng = np.random.default_rng(11)
    z = np.zeros((2, V))
    cols = rng.choice(V, size=k, replace=False)
    z[:, cols] += delta
    other = int(np.setdiff1d(np.arange(V), cols)[5])
    y = np.array([int(cols[3]), other])
    logp, ent = impl.selected_logprob(z, y)
    lp_peak, lp_other, e = _dominant_expect(V, delta, k)
    _close(logp[0], lp_peak, 1e-12, "k-peak logp peak")
    _close(logp[1], lp_other, 1e-12, "k-peak logp other")
    _close(ent[0], e, 1e-11, "k-peak entropy")


def pin_worked_examples(impl):
    """Hand-derived rows z = ln(w) + shift (tests/golden/worked_examples.json)."""
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        w = [Fraction(x) for x in case["weights"]]
        V = len(w)
        total = sum(w)
        with np.errstate(divide="ignore"):
            z = np.log(np.array(case["weights"], dtype=np.float64)) + case["shift"]
        z = np.repeat(z[None, :], V, axis=0)
        y = np.arange(V)
        logp, ent = impl.selected_logprob(z, y)
        exp_ent = mpmath.mpf(0)
        for wv in w:
            if wv > 0:
                p = mpmath.mpf(wv.numerator) / wv.denominator / (mpmath.mpf(total.numerator) / total.denominator)
                exp_ent -= p * mpmath.log(p)
        for v in range(V):
            if w[v] == 0:
                assert logp[v] == -np.inf, f"{case['name']}: masked target"
            else:
                p = mpmath.mpf(w[v].numerator) / w[v].denominator / (mpmath.mpf(total.numerator) / total.denominator)
                # abs error of fp64 logits at |shift| ~ 700 is ~1e-13
                _close(logp[v], mpmath.log(p), 1e-12, f"{case['name']} logp[{v}]")
            _close(ent[v], exp_ent, 1e-12, f"{case['name']} entropy")


def pin_brute_force(impl):
    """mpmath at 50 digits on tiny rows, straight from the definition with no
    max-shift: Z = sum exp(z), logp = z_y - ln Z, H = -sum p ln p."""
    rng = np.random.default_rng(5)
    for V in (1, 3, 17, 64):
        z = rng.uniform(-20, 20, size=(4, V))
        y = rng.integers(0, V, size=4)
        logp, ent = impl.selected_logprob(z, y)
        for t in range(4):
            zs = [mpmath.mpf(float(x)) for x in z[t]]
            Z = mpmath.fsum(mpmath.e ** x for x in zs)
            lp = zs[int(y[t])] - mpmath.log(Z)
            H = -mpmath.fsum((mpmath.e ** x / Z) * (x - mpmath.log(Z)) for x in zs)
            _close(logp[t], lp, 1e-13, f"brute logp V={V}")
            _close(ent[t], H, 1e-12, f"brute entropy V={V}")


def pin_normalisation(impl):
    """sum_y exp(logp[y]) = 1 over all targets of one row (rows replicated)."""
    rng = np.random.default_rng(7)
    for V in (5, 100, 1000):
        row = rng.normal(0, 3, size=V)
        z = np.repeat(row[None, :], V, axis=0)
        logp, ent = impl.selected_logprob(z, np.arange(V))
        total = math.fsum(np.exp(logp))
        assert abs(total - 1.0) < 1e-12, f"normalisation V={V}: {total}"
        assert np.all(ent == ent[0]), "entropy must not depend on the target"
        # entropy is the expectation of -logp under p
        _close(ent[0], -math.fsum(np.exp(logp) * logp), 1e-12, f"entropy as E[-logp] V={V}")


def pin_shift_and_bounds(impl):
    rng = np.random.default_rng(9)
    V = 333
    z = rng.normal(0, 2, size=(6, V))
    y = rng.integers(0, V, size=6)
    lp0, e0 = impl.selected_logprob(z, y)
    for c in (-50.0, 17.0, 400.0):
        lp1, e1 = impl.selected_logprob(z + c, y)
        assert np.allclose(lp0, lp1, rtol=0, atol=1e-12 * (1 + abs(c))), "shift invariance logp"
        assert np.allclose(e0, e1, rtol=0, atol=1e-12 * (1 + abs(c))), "shift invariance entropy"
    assert np.all(lp0 <= 0.0)
    assert np.all(e0 >= 0.0) and np.all(e0 <= math.log(V) + 1e-12)
    # reversing the vocabulary order changes nothing
    lp2, e2 = impl.selected_logprob(z[:, ::-1], V - 1 - y)
    assert np.allclose(lp0, lp2, rtol=0, atol=1e-13) and np.allclose(e0, e2, rtol=0, atol=1e-13)


def pin_specials(impl):
    """-inf entries act as removed columns; all -inf, NaN logits and targets
    outside [0, V) give NaN logp; entropy survives a bad target."""
    rng = np.random.default_rng(13)
    V = 40
    base = rng.normal(0, 1, size=V)
    masked = base.copy()
    drop = np.array([0, 7, 39])
    masked[drop] = -np.inf
    keep = np.setdiff1d(np.arange(V), drop)
    y_full = np.array([3, 20, 38])
    y_kept = np.searchsorted(keep, y_full)
    lp_m, e_m = impl.selected_logprob(np.repeat(masked[None], 3, 0), y_full)
    lp_k, e_k = impl.selected_logprob(np.repeat(base[keep][None], 3, 0), y_kept)
    assert np.allclose(lp_m, lp_k, rtol=0, atol=1e-14) and np.allclose(e_m, e_k, rtol=0, atol=1e-14)
    lp, e = impl.selected_logprob(np.repeat(masked[None], 1, 0), np.array([7]))
    assert lp[0] == -np.inf
    lp, e = impl.selected_logprob(np.full((1, V), -np.inf), np.array([2]))
    assert np.isnan(lp[0]) and np.isnan(e[0])
    bad = base.copy()
    bad[5] = np.nan
    lp, e = impl.selected_logprob(bad[None], np.array([1]))
    assert np.isnan(lp[0]) and np.isnan(e[0])
    lp, e = impl.selected_logprob(np.repeat(base[None], 3, 0), np.array([-1, V, V + 100]))
    assert np.all(np.isnan(lp)) and np.all(np.isfinite(e))


def _bf16_exact(rng, shape, scale_bits):
    """Values a bf16 holds exactly: small signed integers times 2^-scale_bits."""
    return rng.integers(-127, 128, size=shape).astype(np.float64) * 2.0 ** -scale_bits


def pin_linear_exact(impl):
    """z = H W^T against exact rational dot products, non-square shapes."""
    rng = np.random.default_rng(17)
    T, d, V = 3, 16, 5
    h = _bf16_exact(rng, (T, d), 6)
    w = _bf16_exact(rng, (V, d), 9)
    z = impl.linear_logits(h, w)
    assert z.shape == (T, V)
    for t in range(T):
        for v in range(V):
            exact = sum(Fraction(float(h[t, k])) * Fraction(float(w[v, k])) for k in range(d))
            assert Fraction(float(z[t, v])) == exact, f"z[{t},{v}]"
    # the fused form is the logits form applied to those logits
    y = np.array([0, 4, 2])
    lp, e = impl.linear_selected_logprob(h, w, y, vocab_block=2)
    for t in range(T):
        zs = [mpmath.mpf(sum(Fraction(float(h[t, k])) * Fraction(float(w[v, k])) for k in range(d)).numerator)
              / sum(Fraction(float(h[t, k])) * Fraction(float(w[v, k])) for k in range(d)).denominator
              for v in range(V)]
        Z = mpmath.fsum(mpmath.e ** x for x in zs)
        _close(lp[t], zs[int(y[t])] - mpmath.log(Z), 1e-13, "fused logp")
        H = -mpmath.fsum((mpmath.e ** x / Z) * (x - mpmath.log(Z)) for x in zs)
        _close(e[t], H, 1e-12, "fused entropy")


def pin_linear_uniform_weights(impl):
    """Identical W rows give uniform logits: logp = -ln V, entropy = ln V."""
    rng = np.random.default_rng(19)
    T, d, V = 4, 32, 8192
    h = _bf16_exact(rng, (T, d), 4)
    w = np.repeat(_bf16_exact(rng, (1, d), 8), V, axis=0)
    lp, e = impl.linear_selected_logprob(h, w, rng.integers(0, V, size=T))
    for t in range(T):
        _close(lp[t], -mpmath.log(V), 1e-12, "linear uniform logp")
        _close(e[t], mpmath.log(V), 1e-12, "linear uniform entropy")


def pin_temperature(impl):
    """Temperature tau divides every logit: one dominant logit raised by delta
    gives logp = -ln(1 + (V-1) e^(-delta/tau)); a uniform row is unchanged;
    brute force at 50 digits on z / tau."""
    V = 1000
    for tau in (0.7, 1.6):
        for delta in (3.0, 9.0):
            z = np.zeros((2, V))
            z[:, 17] += delta
            lp, ent = impl.selected_logprob(z, np.array([17, 18]), temperature=tau)
            lp_peak, lp_other, e = _dominant_expect(V, delta / tau)
            _close(lp[0], lp_peak, 1e-12, f"temperature logp tau={tau}")
            _close(lp[1], lp_other, 1e-12, f"temperature other tau={tau}")
            _close(ent[0], e, 1e-11, f"temperature entropy tau={tau}")
        lp, ent = impl.selected_logprob(np.full((1, V), 4.0), np.array([3]), temperature=tau)
        _close(lp[0], -mpmath.log(V), 1e-13, "temperature uniform")
    rng = np.random.default_rng(23)
    z = rng.uniform(-10, 10, size=(3, 37))
    y = rng.integers(0, 37, size=3)
    lp, ent = impl.selected_logprob(z, y, temperature=0.7)
    for t in range(3):
        zs = [mpmath.mpf(float(x)) / mpmath.mpf("0.7") for x in z[t]]
        Z = mpmath.fsum(mpmath.e ** x for x in zs)
        _close(lp[t], zs[int(y[t])] - mpmath.log(Z), 1e-12, "temperature brute logp")
        H = -mpmath.fsum((mpmath.e ** x / Z) * (x - mpmath.log(Z)) for x in zs)
        _close(ent[t], H, 1e-11, "temperature brute entropy")
    h = _bf16_exact(rng, (2, 8), 5)
    w = _bf16_exact(rng, (40, 8), 5)
    yy = np.array([3, 39])
    a = impl.linear_selected_logprob(h, w, yy, temperature=0.7)
    b = impl.selected_logprob(impl.linear_logits(h, w), yy, temperature=0.7)
    assert np.allclose(a[0], b[0], rtol=0, atol=1e-13) and np.allclose(a[1], b[1], rtol=0, atol=1e-13)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(ValueError):
            impl.selected_logprob(z, y, temperature=bad)


PINS = [
    pin_uniform,
    pin_dominant,
    pin_k_peaks,
    pin_worked_examples,
    pin_brute_force,
    pin_normalisation,
    pin_shift_and_bounds,
    pin_specials,
    pin_linear_exact,
    pin_linear_uniform_weights,
    pin_temperature,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(_impl_from_module())


def test_package_exports():
    assert oracle.selected_logprob is olp.selected_logprob
    assert oracle.linear_selected_logprob is olp.linear_selected_logprob


def test_report_pairwise_difference_is_one_ulp_at_uniform_logp():
    """The report's pairwise candidate difference, 9.5367431640625e-07, is one
    fp32 ulp (2^-20) in [8, 16): the binade of the uniform-row logp -ln V for
    the 151936-entry vocabulary, as the oracle computes it."""
    with open(os.path.join(GOLDEN, "prior_art_report.json")) as f:
        rep = json.load(f)
    diff = rep["pairwise_max_abs_vs"]["rl_kernel_ws2~vllm_gather"]
    assert diff == 2.0 ** -20
    logp, _ = olp.selected_logprob(np.zeros((1, 151936)), np.array([0]))
    f32 = np.float32(logp[0])
    assert float(np.spacing(np.abs(f32))) == diff
    # the reported fp32-vs-fp64 errors are below one such ulp
    assert all(v < diff for v in rep["max_abs_vs_fp64"].values())


# ----------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# ----------------------------------------------------------------------------

def _sel_variant(*, shift=True, sign=1.0, tgt_off=0, ent_sign=1.0, ent_log=np.log,
                 drop_last=False, max_axis=1, ent_weight=True, temp_mul=False):
    def sel(z, y, temperature=1.0):
        t = float(temperature)
        if not (np.isfinite(t) and t > 0.0):
            raise ValueError("temperature")
        z = np.asarray(z, dtype=np.float64)
        z = z * t if temp_mul else z / t
        y = np.asarray(y, dtype=np.int64)
        T, V = z.shape
        zz = z[:, :-1] if (drop_last and V > 1) else z
        with np.errstate(all="ignore"):
            if shift:
                m = zz.max(axis=max_axis, keepdims=True)
                if max_axis == 0:
                    m = np.broadcast_to(m, zz.shape)[:, :1]
            else:
                m = np.zeros((T, 1))
            log_z = m[:, 0] + np.log(np.exp(zz - m).sum(axis=1))
            valid = (y >= 0) & (y < V)
            ys = np.clip(np.where(valid, y, 0) + tgt_off, 0, V - 1)
            logp = np.where(valid, sign * (z[np.arange(T), ys] - log_z), np.nan)
            p = np.exp(z - log_z[:, None])
            lp = ent_log(p) if ent_log is not np.log else z - log_z[:, None]
            w = p if ent_weight else np.ones_like(p)
            terms = np.where(p > 0, w * lp, 0.0)
            terms = np.where(np.isnan(lp), np.nan, terms)
            ent = -ent_sign * terms.sum(axis=1)
        return logp, ent
    return sel


def _linear_variant(kind):
    def lin(h, w):
        h = np.asarray(h, dtype=np.float64)
        w = np.asarray(w, dtype=np.float64)
        if kind == "transposed":
            return h @ w
        if kind == "drop_k":
            return h[:, :-1] @ w[:, :-1].T
        if kind == "swap_operands":
            return (w @ h.T)
        raise AssertionError(kind)
    return lin


def _mutant(sel=None, lin=None):
    s = sel or olp.selected_logprob
    lz = lin or olp.linear_logits

    def fused(h, w, y, vocab_block=8192, temperature=1.0):
        return s(lz(h, w), y, temperature)

    return types.SimpleNamespace(selected_logprob=s, linear_logits=lz, linear_selected_logprob=fused)


MUTANTS = {
    "no_max_shift": _mutant(_sel_variant(shift=False)),
    "logp_sign_flipped": _mutant(_sel_variant(sign=-1.0)),
    "target_index_off_by_one": _mutant(_sel_variant(tgt_off=1)),
    "entropy_sign_flipped": _mutant(_sel_variant(ent_sign=-1.0)),
    "entropy_log2": _mutant(_sel_variant(ent_log=np.log2)),
    "entropy_unweighted": _mutant(_sel_variant(ent_weight=False)),
    "last_vocab_column_dropped": _mutant(_sel_variant(drop_last=True)),
    "max_over_wrong_axis": _mutant(_sel_variant(max_axis=0)),
    "projection_transposed": _mutant(lin=_linear_variant("transposed")),
    "projection_drops_last_k": _mutant(lin=_linear_variant("drop_k")),
    "projection_operands_swapped": _mutant(lin=_linear_variant("swap_operands")),
    "temperature_multiplies": _mutant(_sel_variant(temp_mul=True)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    impl = MUTANTS[name]
    caught = []
    for pin in PINS:
        try:
            pin(impl)
        except Exception:  # AssertionError, or the mistake breaks a shape
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{name}' passed every pin"
