"""Parity and invariance of the fused LM-head + logprob path on a GB300, through
the C ABI.

Oracle: fp64 CPU logits H W^T from the same bf16 values, then the fp64
definition.  Tolerance 1e-4 absolute on logp and entropy.  Bitwise checks:
1/2/4 vocabulary shards merged on one GPU, persistent grid size, CUDA-graph
replay versus eager, repeats, and (in test_gpu_batch_sweep.py) batch size and
row offset.
"""

import math

import numpy as np
import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import FUSED_TOL, bits, max_err, oracle_fused

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lp.load()
    yield
    lp.lp_set_persistent_grid_limit(0)


def _check_all_rows(x, tol=FUSED_TOL):
    logp, ent = lp.linear_logprob(x.H, x.W, x.y)
    torch.cuda.synchronize()
    ref_lp, ref_ent = oracle_fused(x.H, x.W, x.y)
    e_lp, e_ent = max_err(logp, ref_lp), max_err(ent, ref_ent)
    assert e_lp <= tol and e_ent <= tol, (e_lp, e_ent)
    return logp, ent


def test_tiny_workload_all_rows():
    x = synth.fused_inputs("fused_tiny", device=DEV)
    _check_all_rows(x)


@pytest.mark.parametrize("T,d,V", [
    (1, 64, 512),          # one row, one K block
    (7, 72, 1001),         # K tail (72 = 64 + 8), ragged quarters
    (129, 256, 8192 + 37), # two row blocks, ragged vocabulary
    (300, 136, 3),         # V < 4: empty quarters
    (33, 8, 1),            # V == 1: logp == 0
    (256, 512, 4 * 256 * 2 + 4),
])
def test_ragged_shapes_all_rows(T, d, V):
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=T + d + V)
    _check_all_rows(x)


@pytest.mark.parametrize("T", [5, 40])
def test_hidden_size_not_a_multiple_of_8(T):
    """d = 60 with rows padded to a stride of 64 (the boundary requires
    16-byte row strides, not d % 8 == 0); T = 5 goes through the 16-row copy
    of H, T = 40 reads H in place."""
    d, V = 60, 777
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=3)
    Hs = torch.zeros((T, 64), dtype=x.H.dtype, device=DEV)
    Ws = torch.zeros((V, 64), dtype=x.W.dtype, device=DEV)
    Hs[:, :d] = x.H
    Ws[:, :d] = x.W
    Hs[:, d:] = 1.0  # the row padding must never be read as data
    Ws[:, d:] = 1.0
    logp, ent = lp.linear_logprob(Hs[:, :d], Ws[:, :d], x.y)
    torch.cuda.synchronize()
    ref_lp, ref_ent = oracle_fused(x.H, x.W, x.y)
    e_lp, e_ent = max_err(logp, ref_lp), max_err(ent, ref_ent)
    assert e_lp <= FUSED_TOL and e_ent <= FUSED_TOL, (e_lp, e_ent)


def test_qwen3_8b_head_full_size_all_rows():
    """The headline shape, every row against the oracle (3.2e11 fp64
    multiply-adds on the host, a few seconds)."""
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    logp, ent = lp.linear_logprob(x.H, x.W, x.y)
    ref_lp, ref_ent = oracle_fused(x.H, x.W, x.y)
    e_lp, e_ent = max_err(logp, ref_lp), max_err(ent, ref_ent)
    print(f"qwen3-8b head, all 512 rows: logp err {e_lp:.3e}, entropy err {e_ent:.3e}")
    assert e_lp <= FUSED_TOL and e_ent <= FUSED_TOL


def test_wide_hidden_large_vocabulary_sampled_rows():
    """The largest shapes of the tests: d = 8192 (128 K blocks per tile) and
    V = 262147 (256 tiles per quarter, ragged quarters), sampled rows; plus
    2-shard bitwise equality at that size."""
    T, d, V = 96, 8192, 262147
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV, T=T, d=d, V=V, seed=11)
    logp, ent = lp.linear_logprob(x.H, x.W, x.y)
    rows = torch.tensor([0, 37, 64, 95])
    ref_lp, ref_ent = oracle_fused(x.H, x.W, x.y, rows)
    e_lp, e_ent = max_err(logp[rows], ref_lp), max_err(ent[rows], ref_ent)
    print(f"d=8192, V=262147: logp err {e_lp:.3e}, entropy err {e_ent:.3e}")
    assert e_lp <= FUSED_TOL and e_ent <= FUSED_TOL
    parts = []
    for i in range(2):
        b, e = lp.vocab_shard_range(V, i, 2)
        parts.append(lp.linear_logprob_partials(x.H, x.W[b:e], x.y, V, i, 2))
    m_lp, m_ent = lp.merge_partials(parts)
    assert torch.equal(bits(m_lp), bits(logp)) and torch.equal(bits(m_ent), bits(ent))


def test_qwen3_next_head_shards_bitwise_and_sampled_parity():
    x = synth.fused_inputs("fused_qwen3_next", device=DEV)
    V = x.W.shape[0]
    ref_lp, ref_ent = lp.linear_logprob(x.H, x.W, x.y)
    for n in (1, 2, 4):
        parts = []
        for i in range(n):
            b, e = lp.vocab_shard_range(V, i, n)
            parts.append(lp.linear_logprob_partials(x.H, x.W[b:e], x.y, V, i, n))
        m_lp, m_ent = lp.merge_partials(parts)
        assert torch.equal(bits(m_lp), bits(ref_lp)), f"{n} shards logp"
        assert torch.equal(bits(m_ent), bits(ref_ent)), f"{n} shards entropy"
    rows = torch.tensor([0, 5, 127, 128, 4095, 8191, 8192, 12345, 16383])
    o_lp, o_ent = oracle_fused(x.H, x.W, x.y, rows)
    e_lp, e_ent = max_err(ref_lp[rows], o_lp), max_err(ref_ent[rows], o_ent)
    print(f"qwen3-next head: logp err {e_lp:.3e}, entropy err {e_ent:.3e}")
    assert e_lp <= FUSED_TOL and e_ent <= FUSED_TOL


@pytest.mark.parametrize("V", [8192 + 37, 3])
def test_small_shards_bitwise(V):
    x = synth.fused_inputs("fused_tiny", device=DEV, T=150, d=128, V=V, seed=9)
    ref_lp, ref_ent = lp.linear_logprob(x.H, x.W, x.y)
    for n in (2, 4):
        parts = []
        for i in range(n):
            b, e = lp.vocab_shard_range(V, i, n)
            if e == b:  # an empty shard of a tiny vocabulary: pass one dummy row
                w = torch.zeros((1, 128), dtype=torch.bfloat16, device=DEV)
            else:
                w = x.W[b:e]
            parts.append(lp.linear_logprob_partials(x.H, w, x.y, V, i, n))
        m_lp, m_ent = lp.merge_partials(parts)
        assert torch.equal(bits(m_lp), bits(ref_lp)) and torch.equal(bits(m_ent), bits(ref_ent))


def test_grid_size_invariance_and_repeats():
    x = synth.fused_inputs("fused_tiny", device=DEV, T=300, d=256, V=20000, seed=5)
    ref = lp.linear_logprob(x.H, x.W, x.y)
    for limit in (1, 3, 16, 77, 0):
        lp.lp_set_persistent_grid_limit(limit)
        out = lp.linear_logprob(x.H, x.W, x.y)
        assert torch.equal(bits(out[0]), bits(ref[0])) and torch.equal(bits(out[1]), bits(ref[1])), limit
    lp.lp_set_persistent_grid_limit(0)
    seen = set()
    for _ in range(10):
        o = lp.linear_logprob(x.H, x.W, x.y)
        seen.add((bits(o[0]).numpy().tobytes(), bits(o[1]).numpy().tobytes()))
    assert len(seen) == 1


@pytest.mark.parametrize("d", [512, 320])
def test_ring_choice_keeps_bits(d):
    """Batches of one 256-row block run the kernel with 64-deep K stages, larger
    ones with 128-deep stages (d = 320: the last stage half past the end of
    the rows, read as zeros); a row's bits must not notice."""
    x = synth.fused_inputs("fused_tiny", device=DEV, T=257, d=d, V=20000, seed=6)
    full = lp.linear_logprob(x.H, x.W, x.y)
    for sl in (slice(0, 256), slice(1, 257), slice(100, 101)):
        part = lp.linear_logprob(x.H[sl].contiguous(), x.W, x.y[sl].contiguous())
        assert torch.equal(bits(part[0]), bits(full[0][sl])), sl
        assert torch.equal(bits(part[1]), bits(full[1][sl])), sl


def test_cuda_graph_replay_matches_eager():
    x = synth.fused_inputs("fused_tiny", device=DEV, T=200, d=256, V=30000, seed=6)
    T, d = x.H.shape
    V = x.W.shape[0]
    ws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
    logp = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    eager = lp.linear_logprob(x.H, x.W, x.y)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws, stream=s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
    logp.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bits(logp), bits(eager[0])) and torch.equal(bits(ent), bits(eager[1]))
    assert lp.lp_get_device_error(ws) == 0


def test_bad_targets_and_closed_forms():
    T, d, V = 8, 64, 4096
    g = torch.Generator(device=DEV)
    g.manual_seed(1)
    H = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
    # identical W rows: uniform logits, logp = -ln V, entropy = ln V
    W = torch.randn((1, d), generator=g, device=DEV).mul(0.05).to(torch.bfloat16).expand(V, d).contiguous()
    y = torch.tensor([0, 1, V - 1, -1, V, 5, 6, 7], device=DEV)
    logp, ent = lp.linear_logprob(H, W, y)
    lpv, env = logp.double().cpu(), ent.double().cpu()
    for i in (0, 1, 2, 5, 6, 7):
        assert abs(lpv[i] + math.log(V)) <= 1e-5 and abs(env[i] - math.log(V)) <= 1e-5
    assert math.isnan(lpv[3]) and math.isnan(lpv[4])
    assert math.isfinite(env[3]) and math.isfinite(env[4])
    # one dominant logit: W row y aligned with H gives logp close to 0
    H2 = torch.zeros((2, d), device=DEV)
    H2[:, 0] = 8.0
    W2 = torch.zeros((V, d), device=DEV)
    W2[17, 0] = 8.0  # z[17] = 64, others 0
    y2 = torch.tensor([17, 18], device=DEV)
    lp2, ent2 = lp.linear_logprob(H2.to(torch.bfloat16), W2.to(torch.bfloat16), y2)
    exp_lp = -math.log1p((V - 1) * math.exp(-64.0))
    assert abs(float(lp2[0]) - exp_lp) <= 1e-6 and abs(float(lp2[1]) - (-64.0 + exp_lp)) <= 1e-4
    assert abs(float(ent2[0])) <= 1e-4


def test_empty_batch_and_device_error_word():
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device=DEV)
    H = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((0,), dtype=torch.int64, device=DEV)
    logp, ent = lp.linear_logprob(H, W, y)
    assert logp.numel() == 0
    x = synth.fused_inputs("fused_tiny", device=DEV)
    ws = torch.empty(lp.lp_linear_logprob_workspace_size(64, 256, 8192), dtype=torch.uint8, device=DEV)
    lp.linear_logprob(x.H, x.W, x.y, workspace=ws)
    assert lp.lp_get_device_error(ws) == 0


def test_one_distinct_result_over_sustained_load():
    """500 back-to-back calls at the headline shape (~0.2 s of load, long
    enough for the GPU to reach its power limit and lower its clocks) give one
    distinct result."""
    x = synth.fused_inputs("fused_qwen3_8b", device=DEV)
    T, d = x.H.shape
    V = x.W.shape[0]
    ws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
    ref_lp, ref_ent = lp.linear_logprob(x.H, x.W, x.y, workspace=ws)
    logp = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    mismatches = torch.zeros((), dtype=torch.int64, device=DEV)
    for _ in range(500):
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
        mismatches += (logp.view(torch.int32) != ref_lp.view(torch.int32)).sum()
        mismatches += (ent.view(torch.int32) != ref_ent.view(torch.int32)).sum()
    assert int(mismatches) == 0

