"""Plain, slow, fp64 CPU oracle for selected-token log-probabilities.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
this module.  The CUDA library never links, imports or calls it and the two
share no code: no kernels, helpers, tables or constants.

What it computes is the plain definition the sources rest on.  The RL-Kernel
logprob prior-art report (report.json, kind ``qwen3_next_logprob_prior_art``)
scores every candidate against one shared fp64 reference computed from the same
logits (each candidate's ``"reference": "shared_logits_fp64"`` and its
``max_abs_vs_fp64`` field).  For every row t of a logits matrix z and its
selected token y_t:

    logZ[t]    = log sum_v exp(z[t, v])
    logp[t]    = z[t, y_t] - logZ[t]
    entropy[t] = -sum_v p[t, v] * log p[t, v],   p[t, v] = exp(z[t, v] - logZ[t])

with 0 * log 0 taken as 0 (natural logarithm: nats).  The fused form
("linear_logp", recorded as ``rlkernel.linear_logp.bitwise.v1`` in the backend
readbacks of the RL-Kernel H100 PCP evidence record, h100-pcp.json, section
``validation``) first forms the logits as the LM-head projection z = H W^T and
then applies the same definition.

Readings where the sources are silent (each is listed with its reason in the
design notes of this repository):

* entropy is the Shannon entropy of softmax(z[t, :]) in nats;
* by default no temperature is applied (tau = 1); with a temperature tau > 0
  every logit is divided by tau first (the rollout engine samples at
  temperature 0.7: RL-Kernel H100 PCP evidence record, h100-pcp.json, section
  ``scope``), i.e. the definition above applied to z / tau;
* a target outside [0, V) has no defined log-probability: logp is NaN, the
  entropy is still reported;
* a logit of -inf contributes nothing; a row whose logits are all -inf has no
  distribution and gives NaN; NaN and +inf logits give NaN.

Everything is evaluated in float64 with numpy: ``max`` for the shift that keeps
``exp`` finite (the value of logZ does not depend on which maximum is used),
``exp``, ``log``, pairwise ``sum`` and one library matrix product.  No blocking,
fusion or reordering beyond that.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "logsumexp_rows",
    "selected_logprob",
    "linear_logits",
    "linear_selected_logprob",
    "selected_logprob_grad_logits",
    "linear_selected_logprob_backward",
]


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """logZ[t] = log sum_v exp(z[t, v]) in float64.

    The log-partition function under the selected-token log-probability of the
    logprob prior-art report (report.json, fp64 shared-logits reference).  The
    row maximum M is subtracted before ``exp`` only so that the sum stays finite;
    logZ = M + log sum_v exp(z - M) holds for any finite M.
    """
    z = np.asarray(z, dtype=np.float64)
    if z.ndim != 2:
        raise ValueError("z must be 2-D [T, V]")
    with np.errstate(invalid="ignore", over="ignore"):
        m = z.max(axis=1, keepdims=True)
        # A row of all -inf has no finite maximum; the shift is then NaN and so
        # is logZ, which is the documented result for such a row.
        shifted = z - m
        s = np.exp(shifted).sum(axis=1)
        with np.errstate(divide="ignore"):
            return m[:, 0] + np.log(s)


def _scaled(z: np.ndarray, temperature: float) -> np.ndarray:
    t = float(temperature)
    if not (np.isfinite(t) and t > 0.0):
        raise ValueError("temperature must be finite and > 0")
    return z if t == 1.0 else z / t


def selected_logprob(z: np.ndarray, y: np.ndarray,
                     temperature: float = 1.0) -> tuple[np.ndarray, np.ndarray]:
    """(logp[T], entropy[T]) in float64 for logits z [T, V] and targets y [T].

    logp[t] = z[t, y_t] - logZ[t]: the selected-token log-probability every
    candidate of the logprob prior-art report (report.json, ``candidates``)
    computes from shared logits.  entropy[t] = -sum_v p log p with
    p = exp(z - logZ): the per-row entropy the trainer logs as
    ``train/entropy_loss`` (H100 PCP evidence record, h100-pcp.json, section
    ``comparison``).

    A target outside [0, V) gives logp = NaN.  With ``temperature`` tau the
    logits are z / tau (the rollout's sampling temperature, h100-pcp.json,
    section ``scope``).
    """
    z = _scaled(np.asarray(z, dtype=np.float64), temperature)
    y = np.asarray(y, dtype=np.int64)
    if z.ndim != 2 or y.shape != (z.shape[0],):
        raise ValueError("expected z [T, V] and y [T]")
    t_rows, v = z.shape
    log_z = logsumexp_rows(z)

    valid = (y >= 0) & (y < v)
    y_safe = np.where(valid, y, 0)
    z_sel = z[np.arange(t_rows), y_safe]
    with np.errstate(invalid="ignore"):
        logp = np.where(valid, z_sel - log_z, np.nan)

        log_p = z - log_z[:, None]  # log p[t, v]
        p = np.exp(log_p)
        # 0 * log 0 := 0: an entry with p == 0 (a -inf logit) adds nothing.
        terms = np.where(p > 0.0, p * log_p, 0.0)
        # A row without a distribution (logZ NaN) stays NaN.
        terms = np.where(np.isnan(log_p), np.nan, terms)
        entropy = -terms.sum(axis=1)
    return logp, entropy


def linear_logits(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """z = H W^T in float64: the LM-head projection in front of linear_logp.

    ``h`` is [T, d] and ``w`` is [V, d], both holding the exact values of the
    bf16 inputs (any float dtype; bf16 values widen exactly).  Each product of
    two bf16 values is exact in float64 and the sum over d <= 4096 terms is
    exact to about 1e-16 relative, so this is the exact logit for all purposes
    of a 1e-4 tolerance.  One library matrix product is the whole step.
    """
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if h.ndim != 2 or w.ndim != 2 or h.shape[1] != w.shape[1]:
        raise ValueError("expected h [T, d] and w [V, d] with the same d")
    return h @ w.T


def linear_selected_logprob(
    h: np.ndarray, w: np.ndarray, y: np.ndarray, vocab_block: int = 8192,
    temperature: float = 1.0,
) -> tuple[np.ndarray, np.ndarray]:
    """(logp[T], entropy[T]) of softmax(H W^T) in float64.

    The fused linear_logp operator (``rlkernel.linear_logp.bitwise.v1`` in the
    H100 PCP evidence record, h100-pcp.json, section ``validation``): form the
    logits with :func:`linear_logits`, then apply :func:`selected_logprob`.
    ``vocab_block`` only bounds the float64 copy of W that is alive at once; the
    full [T, V] float64 logits are formed before any reduction.  With
    ``temperature`` tau the logits are H W^T / tau.
    """
    h = np.asarray(h)
    w = np.asarray(w)
    t_rows = h.shape[0]
    v = w.shape[0]
    z = np.empty((t_rows, v), dtype=np.float64)
    for v0 in range(0, v, vocab_block):
        v1 = min(v, v0 + vocab_block)
        z[:, v0:v1] = linear_logits(h, w[v0:v1])
    return selected_logprob(z, y, temperature)


def selected_logprob_grad_logits(z: np.ndarray, y: np.ndarray, g_logp: np.ndarray,
                                 g_ent: np.ndarray | None = None,
                                 temperature: float = 1.0) -> np.ndarray:
    """dL/dz [T, V] in float64 for L = sum_t g_logp[t] logp[t] + g_ent[t] entropy[t].

    The training side of the same operator (the trainer back-propagates through
    the log-probabilities it computes: h100-pcp.json, section ``comparison``,
    ``train/grad_norm``).  With p = softmax(z / tau):

        d logp[t]    / d z[t, v] = (delta(v, y_t) - p[t, v]) / tau
        d entropy[t] / d z[t, v] = -p[t, v] (log p[t, v] + entropy[t]) / tau

    (the second from entropy = -sum_u p_u log p_u and
    d p_u / d z_v = p_u (delta_uv - p_v) / tau).  A row whose target is outside
    [0, V) has no logp, so its logp term contributes no gradient; 0 log 0 is
    taken as 0.
    """
    z = _scaled(np.asarray(z, dtype=np.float64), temperature)
    y = np.asarray(y, dtype=np.int64)
    t_rows, v = z.shape
    g_logp = np.asarray(g_logp, dtype=np.float64).reshape(t_rows)
    g_ent = (np.zeros(t_rows) if g_ent is None
             else np.asarray(g_ent, dtype=np.float64).reshape(t_rows))
    log_z = logsumexp_rows(z)
    log_p = z - log_z[:, None]
    p = np.exp(log_p)
    with np.errstate(invalid="ignore"):
        ent = -np.where(p > 0.0, p * log_p, 0.0).sum(axis=1)
        valid = (y >= 0) & (y < v)
        g_logp = np.where(valid, g_logp, 0.0)
        grad = -g_logp[:, None] * p
        rows = np.arange(t_rows)[valid]
        grad[rows, y[valid]] += g_logp[valid]
        ent_term = np.where(p > 0.0, p * (log_p + ent[:, None]), 0.0)
        grad -= g_ent[:, None] * ent_term
    return grad / float(temperature)


def linear_selected_logprob_backward(
    h: np.ndarray, w: np.ndarray, y: np.ndarray, g_logp: np.ndarray,
    g_ent: np.ndarray | None = None, temperature: float = 1.0,
) -> tuple[np.ndarray, np.ndarray]:
    """(dL/dH [T, d], dL/dW [V, d]) in float64 for the fused operator.

    z = H W^T, so with G = dL/dz from :func:`selected_logprob_grad_logits`:
    dL/dH = G W and dL/dW = G^T H (two library matrix products).
    """
    h64 = np.asarray(h, dtype=np.float64)
    w64 = np.asarray(w, dtype=np.float64)
    g = selected_logprob_grad_logits(linear_logits(h64, w64), y, g_logp, g_ent, temperature)
    return g @ w64, g.T @ h64
