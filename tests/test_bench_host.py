"""Host-side logic of bench.py (no GPU): the clock-record window, the traffic
lookup in the committed ncu summaries, and the throughput arithmetic."""

import datetime as dt
import os
import sys

import pytest

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
import bench  # noqa: E402


def _write_samples(path, t0, samples):
    """samples: (seconds after t0, sm_mhz, power_cap_active)"""
    with open(path, "w") as f:
        for dt_s, mhz, cap in samples:
            ts = dt.datetime.fromtimestamp(t0 + dt_s).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            f.write(f"{ts}, 0, {mhz}, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, "
                    f"{'Active' if cap else 'Not Active'}\n")


def test_clock_window_follows_the_refresh_lag(tmp_path):
    t0 = 1.7e9
    # idle readings until 0.1 s into a 0.5 s timed region, then power-capped ones,
    # which nvidia-smi keeps showing for up to ~0.1 s after the region ends
    samples = [(x / 100.0, 2070, False) for x in range(-20, 10)]
    samples += [(x / 100.0, 1650, True) for x in range(10, 62)]
    samples += [(x / 100.0, 2070, False) for x in range(66, 90)]
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    _write_samples(s.path, t0, samples)
    out = s.summary(t0, t0 + 0.5)
    assert out["sm_mhz"] == 1650
    assert out["reasons"] == ["sw_power_cap"]
    assert out["sm_max_mhz"] == 2070
    assert out["samples"] > 0


def test_clock_window_short_region_uses_following_samples(tmp_path):
    t0 = 1.7e9
    samples = [(x / 100.0, 2070, False) for x in range(-20, 0)]
    samples += [(x / 100.0, 1700, True) for x in range(0, 15)]
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    _write_samples(s.path, t0, samples)
    out = s.summary(t0, t0 + 0.05)  # shorter than one refresh
    assert out["reasons"] == ["sw_power_cap"] and out["sm_mhz"] == 1700


def test_profile_traffic_needs_matching_sources(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    summary = tmp_path / "k.txt"
    good = bench.sha256_files([str(src)])
    summary.write_text(f"kernel: k\nsource_sha256: {good}\ndram_bytes_per_launch_full_size: 1.5e9\n")
    assert bench.profile_traffic(str(summary), [str(src)]) == pytest.approx(1.5e9)
    src.write_text("kernel v2\n")  # the kernel changed since the counters were taken
    assert bench.profile_traffic(str(summary), [str(src)]) is None
    assert bench.profile_traffic(str(tmp_path / "absent.txt"), [str(src)]) is None


def test_committed_summaries_parse():
    for summary, sources in ((bench.PROFILE_SUMMARY, bench.LINEAR_SOURCES),
                             (bench.LOGITS_PROFILE_SUMMARY, bench.LOGITS_SOURCES)):
        fields = {}
        with open(summary) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        assert len(fields["source_sha256"]) == 64
        assert float(fields["dram_bytes_per_launch_full_size"]) > 0


def test_whole_job_throughput():
    # 512 rows per rank, 10 steps, 2 ranks, slowest rank 5 ms -> 2048 rows/ms
    assert bench.whole_job_throughput(512, 10, 2, 5.0) == pytest.approx(2048e3)


def test_profile_traffic_per_call_field(tmp_path):
    src = tmp_path / "b.cu"
    src.write_text("backward v1\n")
    summary = tmp_path / "b.txt"
    h = bench.sha256_files([str(src)])
    summary.write_text(f"source_sha256: {h}\ndram_bytes_per_call_full_size: 5.73e9\n")
    assert bench.profile_traffic(str(summary), [str(src)], "dram_bytes_per_call_full_size") == \
        pytest.approx(5.73e9)
    # a field the summary does not hold reads as unknown
    assert bench.profile_traffic(str(summary), [str(src)]) is None


def test_tp_option_parses_and_defaults_to_replicas():
    assert bench.parse_args([]).tp == 0
    assert bench.parse_args(["--tp", "4", "--gpus", "4"]).tp == 4


def test_profile_hash_follows_code_not_comments(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// header\n__global__ void k(int* p) {\n  *p = 1;  /* one */\n}\n")
    h0 = bench.sha256_files([str(a)])
    a.write_text("// a new header line\n\n__global__ void k(int* p) {\n  *p = 1;  // one\n}\n")
    assert bench.sha256_files([str(a)]) == h0
    a.write_text("__global__ void k(int* p) {\n  *p = 2;\n}\n")
    assert bench.sha256_files([str(a)]) != h0
