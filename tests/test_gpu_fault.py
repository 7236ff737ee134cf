"""The bounded device-side waits of the fused kernel, exercised without a GPU
fault.

With fault injection on, the first CTA pair announces one TMA load it never
issues; its pipeline waits give up after their time bound (about a second),
set the workspace error word, drain and free tensor memory, and the kernel
returns.  The call's outputs are NaN, lp_get_device_error reports
LP_ERR_TIMEOUT, and the next call on the same context gives correct results.
The same holds for the grad_W product of the backward (its last CTA fills
grad_W with NaN).
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


def _bits16(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_backward_withheld_load_poisons_grad_W(dtype):
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV)
    T, d = x.H.shape
    V = x.W.shape[0]
    g = torch.Generator().manual_seed(5)
    gl = torch.randn(T, generator=g).to(DEV)
    ge = torch.randn(T, generator=g).to(DEV)
    ref_h, ref_w = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, grad_W_dtype=dtype)
    ws = torch.empty(lp.lp_linear_logprob_backward_workspace_size(T, d, V), dtype=torch.uint8,
                     device=DEV)
    lp.lp_set_fault_injection(2)
    try:
        gh, gw = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, workspace=ws,
                                            grad_W_dtype=dtype)
        torch.cuda.synchronize()
    finally:
        lp.lp_set_fault_injection(0)
    assert lp.lp_get_device_error(ws) != 0
    assert torch.isnan(gw.float()).all()
    # grad_H comes from the kernels before the product that gave up
    assert torch.equal(bits(gh), bits(ref_h))
    # the context is still usable and the next call is exact
    gh, gw = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, workspace=ws, grad_W_dtype=dtype)
    torch.cuda.synchronize()
    assert lp.lp_get_device_error(ws) == 0
    assert torch.equal(bits(gh), bits(ref_h)) and torch.equal(_bits16(gw), _bits16(ref_w))


def test_backward_withheld_load_poisons_an_accumulated_grad_W():
    """Accumulating into a main gradient when a wait of the grad_W product gives
    up: the main gradient is NaN afterwards (documented), grad_H is exact, and
    the next accumulating call adds exactly."""
    lp.load()
    x = synth.fused_inputs("fused_tiny", device=DEV)
    T, d = x.H.shape
    V = x.W.shape[0]
    g = torch.Generator().manual_seed(6)
    gl = torch.randn(T, generator=g).to(DEV)
    ge = torch.randn(T, generator=g).to(DEV)
    ref_h, ref_w = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
    ws = torch.empty(lp.lp_linear_logprob_backward_workspace_size(T, d, V), dtype=torch.uint8,
                     device=DEV)
    main = torch.ones((V, d), device=DEV)
    lp.lp_set_fault_injection(2)
    try:
        gh, _ = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, workspace=ws,
                                           accumulate_into=main)
        torch.cuda.synchronize()
    finally:
        lp.lp_set_fault_injection(0)
    assert lp.lp_get_device_error(ws) != 0
    assert torch.isnan(main).all()
    assert torch.equal(bits(gh), bits(ref_h))
    main.fill_(1.0)
    lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, workspace=ws, accumulate_into=main)
    torch.cuda.synchronize()
    assert lp.lp_get_device_error(ws) == 0
    assert torch.equal(bits(main), bits(1.0 + ref_w))
