"""Seeded synthetic workloads for selected-token log-probabilities.

This module only draws inputs: it holds none of the method's arithmetic.  Both
sides of a parity check (the CUDA library and the fp64 oracle) consume exactly
the tensors it returns.  Numbers come from ``torch.Generator`` seeded per
workload on the device the tensors are made on, so a workload is reproducible
on one device and torch build; nothing here is meant to match across devices.

Workloads (the shapes and value distributions the sources' workloads have):

* ``fused_tiny``: T=64, d=256, V=8192; H ~ N(0,1), W ~ N(0, 0.05^2), bf16;
  targets uniform in [0, V); seed 0.
* ``logits_peaked``: fp32 logits [1024, 151936] ~ N(0, 3^2); per row 8 distinct
  columns (uniform) raised by +12 after sampling; each target comes with
  probability 1/4 from the row's 8 raised columns (uniform among them), else
  uniform in [0, V); seed 1.
* ``fused_qwen3_8b``: T=512, d=4096, V=151936; H ~ N(0,1) then divided per row
  by sqrt(mean(h^2) + 1e-6) (RMS normalisation without gain, in float64), then
  rounded to bf16; W ~ N(0, 0.02^2) bf16; targets uniform; seed 2.
* ``batch_sweep``: d=4096, V=151936 with the distributions of
  ``fused_qwen3_8b``; 128 probe rows placed at random offsets among random
  filler rows in batches of T in {1, 7, 128, 512, 2048, 4096}; seed 3.
* ``fused_qwen3_next``: T=16384, d=2048, V=151936; H ~ N(0,1), W ~ N(0, 0.03^2)
  bf16; targets uniform; seed 4.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

__all__ = [
    "FusedInputs",
    "LogitsInputs",
    "WORKLOADS",
    "fused_inputs",
    "logits_inputs",
    "batch_sweep",
    "make_generator",
]


@dataclass(frozen=True)
class FusedSpec:
    name: str
    T: int
    d: int
    V: int
    h_std: float
    w_std: float
    rms_norm: bool
    seed: int


@dataclass(frozen=True)
class LogitsSpec:
    name: str
    T: int
    V: int
    std: float
    n_peaks: int
    peak_raise: float
    peak_target_frac: float
    seed: int


WORKLOADS = {
    "fused_tiny": FusedSpec("fused_tiny", 64, 256, 8192, 1.0, 0.05, False, 0),
    "logits_peaked": LogitsSpec("logits_peaked", 1024, 151936, 3.0, 8, 12.0, 0.25, 1),
    "fused_qwen3_8b": FusedSpec("fused_qwen3_8b", 512, 4096, 151936, 1.0, 0.02, True, 2),
    "batch_sweep": FusedSpec("batch_sweep", 128, 4096, 151936, 1.0, 0.02, True, 3),
    "fused_qwen3_next": FusedSpec("fused_qwen3_next", 16384, 2048, 151936, 1.0, 0.03, False, 4),
}

BATCH_SWEEP_SIZES = (1, 7, 128, 512, 2048, 4096)


@dataclass
class FusedInputs:
    H: torch.Tensor  # [T, d] bf16
    W: torch.Tensor  # [V, d] bf16
    y: torch.Tensor  # [T] int64


@dataclass
class LogitsInputs:
    z: torch.Tensor  # [T, V] fp32
    y: torch.Tensor  # [T] int64


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def _hidden(T, d, std, rms_norm, g, device) -> torch.Tensor:
    h = _normal((T, d), std, g, device)
    if rms_norm:
        h64 = h.double()
        h64 = h64 / torch.sqrt(h64.square().mean(dim=1, keepdim=True) + 1e-6)
        h = h64.float()
    return h.to(torch.bfloat16)


def fused_inputs(spec: FusedSpec | str, device="cpu", T: int | None = None,
                 d: int | None = None, V: int | None = None,
                 seed: int | None = None) -> FusedInputs:
    """H, W, y for a fused workload; T, d, V, seed may be overridden (smaller
    parity cases keep the distributions of the named workload)."""
    if isinstance(spec, str):
        spec = WORKLOADS[spec]
    T = spec.T if T is None else T
    d = spec.d if d is None else d
    V = spec.V if V is None else V
    seed = spec.seed if seed is None else seed
    g = make_generator(seed, device)
    W = _normal((V, d), spec.w_std, g, device).to(torch.bfloat16)
    H = _hidden(T, d, spec.h_std, spec.rms_norm, g, device)
    y = torch.randint(0, V, (T,), generator=g, device=device, dtype=torch.int64)
    return FusedInputs(H=H, W=W, y=y)


def logits_inputs(spec: LogitsSpec | str = "logits_peaked", device="cpu",
                  T: int | None = None, V: int | None = None,
                  seed: int | None = None) -> LogitsInputs:
    """Peaked fp32 logits and targets (see the module docstring)."""
    if isinstance(spec, str):
        spec = WORKLOADS[spec]
    T = spec.T if T is None else T
    V = spec.V if V is None else V
    seed = spec.seed if seed is None else seed
    g = make_generator(seed, device)
    z = _normal((T, V), spec.std, g, device)
    k = min(spec.n_peaks, V)
    if k > 0:
        # k distinct columns per row: the k largest of V uniform keys.
        keys = torch.rand((T, V), generator=g, device=device)
        peaks = keys.topk(k, dim=1).indices
        del keys
        z.scatter_add_(1, peaks, torch.full(peaks.shape, spec.peak_raise,
                                            device=device, dtype=torch.float32))
    else:
        peaks = torch.zeros((T, 1), dtype=torch.int64, device=device)
    uniform_y = torch.randint(0, V, (T,), generator=g, device=device, dtype=torch.int64)
    pick = torch.randint(0, max(k, 1), (T, 1), generator=g, device=device, dtype=torch.int64)
    from_peak = torch.rand((T,), generator=g, device=device) < spec.peak_target_frac
    peak_y = peaks.gather(1, pick)[:, 0]
    y = torch.where(from_peak & (k > 0), peak_y, uniform_y)
    return LogitsInputs(z=z, y=y)


@dataclass
class SweepBatch:
    T: int
    H: torch.Tensor          # [T, d] bf16
    y: torch.Tensor          # [T] int64
    probe_slots: torch.Tensor  # [n] row index inside this batch
    probe_ids: torch.Tensor    # [n] which probe row sits there


def batch_sweep(device="cpu", sizes=BATCH_SWEEP_SIZES, n_probe: int = 128,
                d: int | None = None, V: int | None = None, seed: int | None = None):
    """The batch-invariance sweep: W, the probe rows and, per batch size, the
    list of batches that together hold every probe row at a random offset.

    Batches smaller than the probe set are repeated until every probe row has
    appeared once; rows of a batch not taken by a probe are fresh filler rows
    from the same distribution.  Returns (W, probe_H, probe_y, {T: [SweepBatch]}).
    """
    spec = WORKLOADS["batch_sweep"]
    d = spec.d if d is None else d
    V = spec.V if V is None else V
    seed = spec.seed if seed is None else seed
    g = make_generator(seed, device)
    W = _normal((V, d), spec.w_std, g, device).to(torch.bfloat16)
    probe_H = _hidden(n_probe, d, spec.h_std, spec.rms_norm, g, device)
    probe_y = torch.randint(0, V, (n_probe,), generator=g, device=device, dtype=torch.int64)
    gc = make_generator(seed + 1000, "cpu")  # placement decisions on the host
    out = {}
    for T in sizes:
        batches = []
        order = torch.randperm(n_probe, generator=gc)
        per = min(T, n_probe)
        for b0 in range(0, n_probe, per):
            ids = order[b0:b0 + per]
            slots = torch.randperm(T, generator=gc)[: len(ids)]
            H = _hidden(T, d, spec.h_std, spec.rms_norm, g, device)
            y = torch.randint(0, V, (T,), generator=g, device=device, dtype=torch.int64)
            H[slots.to(device)] = probe_H[ids.to(device)]
            y[slots.to(device)] = probe_y[ids.to(device)]
            batches.append(SweepBatch(T=T, H=H, y=y, probe_slots=slots, probe_ids=ids))
        out[T] = batches
    return W, probe_H, probe_y, out
