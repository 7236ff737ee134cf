"""The bounded device-side waits of the fused kernel, exercised without a GPU
fault.

With fault injection on, the first CTA pair announces one TMA load it never
issues; its pipeline waits give up after their time bound (about a second),
set the workspace error word, drain and free tensor memory, and the kernel
returns.  The call's outputs are NaN, lp_get_device_error reports
LP_ERR_TIMEOUT, and the next call on the same context gives correct results.
"""

import math

import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_withheld_load_times_out_cleanly():
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV)
    T, d = x.H.shape
    V = x.W.shape[0]
    ref = lp.linear_logprob(x.H, x.W, x.y)
    ws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
    logp = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    lp.lp_set_fault_injection(1)
    try:
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
        torch.cuda.synchronize()
    finally:
        lp.lp_set_fault_injection(0)
    word = lp.lp_get_device_error(ws)
    assert word != 0
    st = lp.load().lp_get_device_error(ws.data_ptr(), ws.numel(), None, None)
    assert lp.STATUS[st] == "LP_ERR_TIMEOUT"
    assert all(math.isnan(v) for v in logp.tolist())
    # the context is still usable and the next call is exact
    lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
    torch.cuda.synchronize()
    assert lp.lp_get_device_error(ws) == 0
    assert torch.equal(bits(logp), bits(ref[0])) and torch.equal(bits(ent), bits(ref[1]))
