"""grad_W accumulated into a float32 main gradient (LP_GRAD_W_FLOAT32_ACCUMULATE)
on a GB300: the result must be the float32 sum, rounded to nearest, of the main
gradient and the grad_W the same call writes on its own, bit for bit (one add
per element by the TMA unit's reduction, every element the target of one box),
and grad_H must not change.  Main gradients are N(0, 1), so neither addend nor
sum is subnormal."""

import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lp.load()


def _upstream(T, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn(T, generator=g, device=DEV), torch.randn(T, generator=g, device=DEV) * 0.5


def _main_grad(V, d, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn((V, d), generator=g, device=DEV)


@pytest.mark.parametrize("T,d,V", [(64, 256, 8192), (5, 64, 4160), (300, 512, 20003),
                                   (512, 4096, 151936)])
def test_accumulate_is_the_float32_sum(T, d, V):
    spec = "fused_qwen3_8b" if V == 151936 else "fused_tiny"
    x = synth.fused_inputs(spec, device=DEV, T=T, d=d, V=V, seed=T + d)
    gl, ge = _upstream(T, T)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    gH, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, saved_lse=lse, saved_entropy=ent)
    main = _main_grad(V, d, 3)
    expect = main + gW
    del gW
    aH, acc = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, saved_lse=lse, saved_entropy=ent,
                                         accumulate_into=main)
    torch.cuda.synchronize()
    assert acc is main
    assert torch.equal(bits(aH), bits(gH))
    assert torch.equal(bits(main), bits(expect))


def test_two_micro_batches():
    """Two backward calls accumulated into one main gradient: ((main + g1) + g2)."""
    T, d, V = 96, 128, 8192
    main = _main_grad(V, d, 4)
    expect = main.clone()
    for k in range(2):
        x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=40 + k)
        gl, ge = _upstream(T, 50 + k)
        _, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge)
        expect = expect + gW
        lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, accumulate_into=main)
    torch.cuda.synchronize()
    assert torch.equal(bits(main), bits(expect))


def test_shards_accumulate_their_rows():
    T, d, V = 64, 128, 16384
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=60)
    gl, ge = _upstream(T, 61)
    _, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    _, gW = lp.linear_logprob_backward(x.H, x.W, x.y, gl, ge, saved_lse=lse, saved_entropy=ent)
    main = _main_grad(V, d, 5)
    expect = main + gW
    for i in range(4):
        b, e = lp.vocab_shard_range(V, i, 4)
        ws = torch.empty(lp.lp_linear_logprob_partials_backward_workspace_size(T, d, V, 4),
                         dtype=torch.uint8, device=DEV)
        part = torch.empty((T, d), device=DEV)
        lp.lp_linear_logprob_partials_backward(x.H, x.W[b:e], x.y, V, i, 4, 1.0, lse, ent, gl, ge,
                                               part, main[b:e], ws, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(bits(main), bits(expect))
    # the convenience form, two shards, on top
    expect = expect + gW
    for i in range(2):
        b, e = lp.vocab_shard_range(V, i, 2)
        _, rows = lp.linear_logprob_partials_backward(x.H, x.W[b:e], x.y, V, i, 2, lse, ent, gl,
                                                      ge, accumulate_into=main[b:e])
        assert rows.data_ptr() == main[b:e].data_ptr()
    torch.cuda.synchronize()
    assert torch.equal(bits(main), bits(expect))


def test_accumulate_needs_float32():
    x = synth.fused_inputs("fused_tiny", device=DEV, T=16, d=64, V=4096, seed=70)
    with pytest.raises(TypeError):
        lp.linear_logprob_backward(x.H, x.W, x.y, torch.ones(16, device=DEV),
                                   accumulate_into=torch.zeros((4096, 64), dtype=torch.bfloat16,
                                                               device=DEV))
