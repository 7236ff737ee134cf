"""Shared helpers of the GPU parity tests: oracle evaluation on host copies of
the exact tensors the CUDA path consumed, and error reports."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances (absolute), written into the tests' assertions:
LOGITS_LOGP_TOL = 2e-6      # logits-given path, logp
LOGITS_ENT_TOL = 1e-5       # logits-given path, entropy
FUSED_TOL = 1e-4            # fused bf16 path, logp and entropy


def oracle_logits(z: torch.Tensor, y: torch.Tensor, rows=None):
    zz = z if rows is None else z[rows]
    yy = y if rows is None else y[rows]
    return oracle.selected_logprob(zz.double().cpu().numpy(), yy.cpu().numpy())


def oracle_fused(H: torch.Tensor, W: torch.Tensor, y: torch.Tensor, rows=None, w_host=None):
    hh = H if rows is None else H[rows]
    yy = y if rows is None else y[rows]
    w = w_host if w_host is not None else W.float().cpu().numpy()
    return oracle.linear_selected_logprob(hh.float().cpu().numpy(), w, yy.cpu().numpy())


def max_err(gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu.double().cpu().numpy()
    both_nan = np.isnan(g) & np.isnan(ref)
    same_inf = np.isinf(g) & np.isinf(ref) & (np.sign(g) == np.sign(ref))
    with np.errstate(invalid="ignore"):  # inf - inf where both are the same infinity
        diff = np.where(both_nan | same_inf, 0.0, np.abs(g - ref))
    diff = np.where(np.isnan(diff), np.inf, diff)
    return float(diff.max()) if diff.size else 0.0


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int32).cpu()


def excess_over_rounding(gpu: torch.Tensor, ref: np.ndarray) -> float:
    """Largest |gpu - ref| beyond half an ulp of the float32 nearest ref, over
    the finite entries: what an output that is ref correctly rounded to float32
    would show as 0."""
    g = gpu.double().cpu().numpy()
    ok = np.isfinite(ref) & np.isfinite(g)
    r = ref[ok]
    half_ulp = np.spacing(np.abs(r).astype(np.float32)).astype(np.float64) / 2
    ex = np.abs(g[ok] - r) - half_ulp
    return float(max(ex.max(), 0.0)) if ex.size else 0.0
