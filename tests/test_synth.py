"""The seeded workload generator: shapes, dtypes, distributions, determinism."""

import torch

from invariant_token_logprobs_gb300 import synth


def test_fused_shapes_and_determinism():
    a = synth.fused_inputs("fused_tiny")
    b = synth.fused_inputs("fused_tiny")
    assert a.H.shape == (64, 256) and a.W.shape == (8192, 256) and a.y.shape == (64,)
    assert a.H.dtype == torch.bfloat16 and a.W.dtype == torch.bfloat16 and a.y.dtype == torch.int64
    assert torch.equal(a.H, b.H) and torch.equal(a.W, b.W) and torch.equal(a.y, b.y)
    assert int(a.y.min()) >= 0 and int(a.y.max()) < 8192
    assert abs(float(a.W.float().std()) - 0.05) < 0.002
    assert abs(float(a.H.float().std()) - 1.0) < 0.02


def test_rms_normalised_rows():
    x = synth.fused_inputs("fused_qwen3_8b", T=16, d=512, V=64)
    rms = x.H.double().square().mean(dim=1).sqrt()
    assert torch.allclose(rms, torch.ones_like(rms), atol=1e-2)
    assert abs(float(x.W.float().std()) - 0.02) < 0.002


def test_peaked_logits():
    x = synth.logits_inputs("logits_peaked", T=256, V=4096)
    z = x.z
    assert z.dtype == torch.float32 and z.shape == (256, 4096)
    # 8 raised columns per row: the top-8 sit near +12 above the rest
    top = z.topk(8, dim=1).values
    assert float(top.min()) > 12.0 - 4 * 3.0
    frac_peak = float((z.gather(1, x.y[:, None])[:, 0] > 12.0 - 3 * 3.0).float().mean())
    assert 0.15 < frac_peak < 0.40


def test_batch_sweep_covers_every_probe():
    W, ph, py, batches = synth.batch_sweep(sizes=(1, 7, 128), n_probe=16, d=64, V=96)
    for T, bl in batches.items():
        seen = torch.cat([b.probe_ids for b in bl]).sort().values
        assert torch.equal(seen, torch.arange(16))
        for b in bl:
            assert b.H.shape == (T, 64)
            assert torch.equal(b.H[b.probe_slots], ph[b.probe_ids])
            assert torch.equal(b.y[b.probe_slots], py[b.probe_ids])
