"""lp_linear_logprob_noalloc: the fused call for callers that cannot allocate
device memory (a host runtime that owns all device memory and forbids
cudaMalloc in plug-ins, or a latency-critical path that must not risk a
synchronising allocation).  It uses the library's fixed device scratch instead
of a workspace.

Checked through the C ABI against lp_linear_logprob on the same inputs, on two
calls in a row (different shapes, so the second call reuses scratch the first
one left behind), within the fused-path tolerance (and, since both run the same
kernels, bit for bit).  The file is named so that pytest collects it last.
"""

import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import FUSED_TOL, bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _compare(x):
    T = x.H.shape[0]
    ref_lp, ref_ent = lp.linear_logprob(x.H, x.W, x.y)
    logp = torch.full((T,), float("nan"), device=DEV)
    ent = torch.full((T,), float("nan"), device=DEV)
    lp.lp_linear_logprob_noalloc(x.H, x.W, x.y, logp, ent)
    torch.cuda.synchronize()
    assert float((logp - ref_lp).abs().max()) <= FUSED_TOL
    assert float((ent - ref_ent).abs().max()) <= FUSED_TOL
    assert torch.equal(bits(logp), bits(ref_lp)) and torch.equal(bits(ent), bits(ref_ent))


def test_noalloc_matches_workspace_call_twice_in_a_row():
    lp.load()
    a = synth.fused_inputs("fused_tiny", device=DEV)
    b = synth.fused_inputs("fused_tiny", device=DEV, T=300, d=512, V=20000 + 3, seed=11)
    c = synth.fused_inputs("fused_tiny", device=DEV, T=5, d=256, V=3001, seed=12)
    _compare(a)
    _compare(b)
    _compare(c)  # fewer than 16 rows: the 16-row copy of H lives in the scratch too
    _compare(a)


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = lp.load()
    A = 1 << 20  # never dereferenced: the size check comes first
    V, d = 151936, 4096
    assert lp.lp_linear_logprob_workspace_size(3518, d, V) <= 32 << 20
    assert lp.lp_linear_logprob_workspace_size(3519, d, V) > 32 << 20
    st = lib.lp_linear_logprob_noalloc(A, d, A, d, A, 3519, d, V, A, A, None)
    assert st == 4  # LP_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_follows_the_current_context():
    """The scratch array's device address belongs to one CUDA context: a call in
    another context (a second context on the device, or the primary context
    re-created after a reset) must look it up again, never reuse a stale one.
    Run in a child process that drives the device through the driver API only."""
    import os
    import subprocess
    import sys
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_noalloc_context_child.py")
    res = subprocess.run([sys.executable, child], capture_output=True, text=True, timeout=300)
    print(res.stdout)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip().endswith("ok")


def test_noalloc_timeout_shows_as_nan_then_recovers():
    """A no-alloc call whose bounded device-side wait gives up has no workspace
    for lp_get_device_error to read: its logp and entropy are NaN instead.  The
    next call on the same context is exact again."""
    import math
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV)
    T = x.H.shape[0]
    ref_lp, ref_ent = lp.linear_logprob(x.H, x.W, x.y)
    logp = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    lp.lp_set_fault_injection(1)
    try:
        lp.lp_linear_logprob_noalloc(x.H, x.W, x.y, logp, ent)
        torch.cuda.synchronize()
    finally:
        lp.lp_set_fault_injection(0)
    assert all(math.isnan(v) for v in logp.tolist())
    assert all(math.isnan(v) for v in ent.tolist())
    lp.lp_linear_logprob_noalloc(x.H, x.W, x.y, logp, ent)
    torch.cuda.synchronize()
    assert torch.equal(bits(logp), bits(ref_lp)) and torch.equal(bits(ent), bits(ref_ent))
