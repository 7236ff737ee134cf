"""CUDA-graph capture vs eager, byte for byte, at capture sizes 1..8.

The RL-Kernel H100 PCP evidence record (h100-pcp.json, section "validation",
"cudagraph") checks that the rollout engine captures graphs for batch sizes
1..8 and that eager and graph-replayed results have 0 byte mismatches
("eager_and_cuda_graph_byte_mismatches": 0).  Here each entry point is captured
once per size on static buffers; fresh inputs are copied into those buffers
before every replay, and the replayed outputs must equal an eager call on the
same inputs bit for bit.
"""

import pytest
import torch

from invariant_token_logprobs_gb300 import lp, synth
from _gpu_helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SIZES = range(1, 9)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lp.load()


def _capture(fn):
    """Warm up fn on a side stream, then capture it into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("tau", [None, 0.7])
def test_fused_graph_replay_bytes_equal_eager(tau):
    d, V = 1024, 151936
    W = synth.fused_inputs("fused_qwen3_8b", device=DEV, T=1, d=d, V=V).W
    for T in SIZES:
        H = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
        y = torch.empty((T,), dtype=torch.int64, device=DEV)
        logp = torch.empty(T, device=DEV)
        ent = torch.empty(T, device=DEV)
        ws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
        if tau is None:
            fn = lambda: lp.lp_linear_logprob(H, W, y, logp, ent, ws)
        else:
            fn = lambda: lp.lp_linear_logprob_temperature(H, W, y, tau, logp, ent, ws)
        first = synth.fused_inputs("fused_qwen3_8b", device=DEV, T=T, d=d, V=16, seed=90 + T)
        H.copy_(first.H)
        y.random_(0, V)
        g = _capture(fn)
        for trial in range(3):
            x = synth.fused_inputs("fused_qwen3_8b", device=DEV, T=T, d=d, V=16, seed=1000 * T + trial)
            H.copy_(x.H)
            y.copy_(torch.randint(0, V, (T,), device=DEV))
            g.replay()
            torch.cuda.synchronize()
            got = (bits(logp), bits(ent))
            ref = lp.linear_logprob(H.clone(), W, y.clone(), temperature=tau)
            assert torch.equal(got[0], bits(ref[0])), f"T={T} trial {trial} logp"
            assert torch.equal(got[1], bits(ref[1])), f"T={T} trial {trial} entropy"
        assert lp.lp_get_device_error(ws) == 0


@pytest.mark.parametrize("tau", [None, 0.7])
def test_logits_graph_replay_bytes_equal_eager(tau):
    V = 151936
    for T in SIZES:
        z = torch.empty((T, V), device=DEV)
        y = torch.empty((T,), dtype=torch.int64, device=DEV)
        logp = torch.empty(T, device=DEV)
        ent = torch.empty(T, device=DEV)
        if tau is None:
            fn = lambda: lp.lp_logprob_from_logits(z, y, logp, ent)
        else:
            fn = lambda: lp.lp_logprob_from_logits_temperature(z, y, tau, logp, ent)
        x0 = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=50 + T)
        z.copy_(x0.z)
        y.copy_(x0.y)
        g = _capture(fn)
        for trial in range(3):
            x = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=700 * T + trial)
            z.copy_(x.z)
            y.copy_(x.y)
            g.replay()
            torch.cuda.synchronize()
            ref = lp.logprob_from_logits(z.clone(), y.clone(), temperature=tau)
            assert torch.equal(bits(logp), bits(ref[0])), f"T={T} trial {trial} logp"
            assert torch.equal(bits(ent), bits(ref[1])), f"T={T} trial {trial} entropy"


def test_logits_backward_graph_replay_bytes_equal_eager():
    # forward with log Z and the backward captured together, as a trainer would
    V = 151936
    for T in SIZES:
        z = torch.empty((T, V), device=DEV)
        y = torch.empty((T,), dtype=torch.int64, device=DEV)
        gl = torch.empty(T, device=DEV)
        ge = torch.empty(T, device=DEV)
        logp = torch.empty(T, device=DEV)
        ent = torch.empty(T, device=DEV)
        lse = torch.empty(T, device=DEV)
        grad = torch.empty((T, V), device=DEV)

        def fn():
            lp.lp_logprob_from_logits_lse(z, y, 0.7, logp, ent, lse)
            lp.lp_logprob_from_logits_backward(z, y, 0.7, lse, ent, gl, ge, grad)

        x0 = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=60 + T)
        z.copy_(x0.z)
        y.copy_(x0.y)
        gl.normal_()
        ge.normal_()
        g = _capture(fn)
        for trial in range(2):
            x = synth.logits_inputs("logits_peaked", device=DEV, T=T, V=V, seed=900 * T + trial)
            z.copy_(x.z)
            y.copy_(x.y)
            gl.normal_()
            ge.normal_()
            g.replay()
            torch.cuda.synchronize()
            ref = lp.logprob_from_logits_backward(z.clone(), y.clone(), gl.clone(), ge.clone(),
                                                  temperature=0.7)
            assert torch.equal(bits(grad), bits(ref)), f"T={T} trial {trial}"


def test_sharded_merge_graph_replay_bytes_equal_eager():
    """The 4-shard fused path (partials of each shard, then the fixed merge)
    captured as one graph equals the eager unsharded call."""
    d, V, T = 512, 151936, 8
    x = synth.fused_inputs("fused_qwen3_next", device=DEV, T=T, d=d, V=V, seed=3)
    ranges = [lp.vocab_shard_range(V, i, 4) for i in range(4)]
    parts = [torch.empty((T, 1, lp.STATE_FLOATS), device=DEV) for _ in range(4)]
    wss = [torch.empty(lp.lp_linear_logprob_partials_workspace_size(T, d, V, 4), dtype=torch.uint8,
                       device=DEV) for _ in range(4)]
    logp = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)

    def fn():
        for i, (b, e) in enumerate(ranges):
            lp.lp_linear_logprob_partials(x.H, x.W[b:e], x.y, V, i, 4, parts[i], wss[i])
        lp.lp_merge_partials(parts, T, logp, ent)

    g = _capture(fn)
    logp.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = lp.linear_logprob(x.H, x.W, x.y)
    assert torch.equal(bits(logp), bits(ref[0])) and torch.equal(bits(ent), bits(ref[1]))


@pytest.mark.parametrize("saved", [False, True])
def test_backward_graph_replay_bytes_equal_eager(saved):
    """The backward (with and without the forward's saved statistics) captured
    once on static buffers; replays on fresh rows equal eager calls."""
    T, d, V = 40, 256, 20000
    W = synth.fused_inputs("fused_tiny", device=DEV, T=1, d=d, V=V, seed=3).W
    H = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    y = torch.empty(T, dtype=torch.int64, device=DEV)
    gl = torch.empty(T, device=DEV)
    ge = torch.empty(T, device=DEV)
    lse = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    logp = torch.empty(T, device=DEV)
    fws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
    ws = torch.empty(lp.lp_linear_logprob_backward_workspace_size(T, d, V), dtype=torch.uint8,
                     device=DEV)
    gH = torch.empty((T, d), device=DEV)
    gW = torch.empty((V, d), device=DEV)

    def fill(seed):
        x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=seed)
        H.copy_(x.H)
        y.copy_(x.y)
        g = torch.Generator(device=DEV)
        g.manual_seed(seed)
        gl.copy_(torch.randn(T, generator=g, device=DEV))
        ge.copy_(torch.randn(T, generator=g, device=DEV))
        if saved:
            lp.lp_linear_logprob_lse(H, W, y, 1.0, logp, ent, lse, fws)

    def call():
        lp.lp_linear_logprob_backward(H, W, y, 1.0, lse if saved else None,
                                      ent if saved else None, gl, ge, gH, gW, ws)

    fill(100)
    graph = _capture(call)
    for seed in (101, 102):
        fill(seed)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got_h, got_w = gH.clone(), gW.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(bits(got_h.reshape(-1)), bits(gH.reshape(-1)))
        assert torch.equal(bits(got_w.reshape(-1)), bits(gW.reshape(-1)))


def test_shard_backward_graph_replay_bytes_equal_eager():
    """Two shards' backward and the merge of their partial grad_H captured once
    on static buffers (V % 64 == 0: the quarter order); replays equal eager
    calls and the single-GPU backward."""
    T, d, V, n = 48, 128, 16384, 2
    W = synth.fused_inputs("fused_tiny", device=DEV, T=1, d=d, V=V, seed=5).W
    H = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    y = torch.empty(T, dtype=torch.int64, device=DEV)
    gl = torch.empty(T, device=DEV)
    ge = torch.empty(T, device=DEV)
    lse = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    logp = torch.empty(T, device=DEV)
    fws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
    wsz = lp.lp_linear_logprob_partials_backward_workspace_size(T, d, V, n)
    ws = [torch.empty(wsz, dtype=torch.uint8, device=DEV) for _ in range(n)]
    rng = [lp.vocab_shard_range(V, i, n) for i in range(n)]
    parts = [torch.empty((T, d), device=DEV) for _ in range(n)]
    rows = [torch.empty((e - b, d), device=DEV) for b, e in rng]
    gH = torch.empty((T, d), device=DEV)

    def fill(seed):
        x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=seed)
        H.copy_(x.H)
        y.copy_(x.y)
        g = torch.Generator(device=DEV)
        g.manual_seed(seed)
        gl.copy_(torch.randn(T, generator=g, device=DEV))
        ge.copy_(torch.randn(T, generator=g, device=DEV))
        lp.lp_linear_logprob_lse(H, W, y, 1.0, logp, ent, lse, fws)

    def call():
        for i, (b, e) in enumerate(rng):
            lp.lp_linear_logprob_partials_backward(H, W[b:e], y, V, i, n, 1.0, lse, ent, gl, ge,
                                                   parts[i], rows[i], ws[i])
        lp.lp_merge_grad_h_partials(parts, gH)

    fill(200)
    graph = _capture(call)
    for seed in (201, 202):
        fill(seed)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got_h, got_w = gH.clone(), torch.cat(rows)
        call()
        torch.cuda.synchronize()
        assert torch.equal(got_h.view(torch.int32), gH.view(torch.int32)), seed
        assert torch.equal(got_w.view(torch.int32), torch.cat(rows).view(torch.int32)), seed
        ref_h, ref_w = lp.linear_logprob_backward(H, W, y, gl, ge, saved_lse=lse,
                                                  saved_entropy=ent)
        torch.cuda.synchronize()
        assert torch.equal(ref_h.view(torch.int32), got_h.view(torch.int32)), seed
        assert torch.equal(ref_w.view(torch.int32), got_w.view(torch.int32)), seed


def test_accumulating_backward_graph_replay_bytes_equal_eager():
    """The backward adding grad_W into a main gradient, captured once: two
    replays add what two eager calls add, byte for byte."""
    T, d, V = 32, 128, 8192
    x = synth.fused_inputs("fused_tiny", device=DEV, T=T, d=d, V=V, seed=7)
    g = torch.Generator(device=DEV)
    g.manual_seed(8)
    gl = torch.randn(T, generator=g, device=DEV)
    ge = torch.randn(T, generator=g, device=DEV)
    lse = torch.empty(T, device=DEV)
    ent = torch.empty(T, device=DEV)
    logp = torch.empty(T, device=DEV)
    fws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=DEV)
    lp.lp_linear_logprob_lse(x.H, x.W, x.y, 1.0, logp, ent, lse, fws)
    ws = torch.empty(lp.lp_linear_logprob_backward_workspace_size(T, d, V), dtype=torch.uint8,
                     device=DEV)
    gH = torch.empty((T, d), device=DEV)
    main = torch.randn((V, d), generator=g, device=DEV)
    start = main.clone()

    def call():
        lp.lp_linear_logprob_backward_ex(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, main, ws,
                                         accumulate=True)

    graph = _capture(call)  # a warm-up call inside _capture may run eagerly: start again
    main.copy_(start)
    torch.cuda.synchronize()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    replayed = main.clone()
    main.copy_(start)
    call()
    call()
    torch.cuda.synchronize()
    assert torch.equal(bits(replayed.reshape(-1)), bits(main.reshape(-1)))
