#!/usr/bin/env python
"""Benchmark of batch-invariant selected-token log-probabilities on GB300.

One step = one call of the fused LM-head projection + logprob path
(lp_linear_logprob: the tensor-core kernel, then the fixed-order merge kernel)
on the Qwen3-8B head shape: T=512 rows, d=4096, V=151936, bf16 H and W,
int64 targets, fp32 logp and entropy out.  Inputs are seeded synthetic tensors
(random-init weights of that shape), resident in HBM before timing; W (1.245
GB) is larger than L2, so no flush is needed between steps.

Printed: one JSON line with the step throughput in selected-token logprobs/s,
the roofline of the dominant kernel (timed alone with CUDA events recorded by
the library around it), the fp64 CPU oracle timed on a sample on this host,
an end-to-end figure through the C ABI with host buffers, SM clocks sampled
during the timed region, and a secondary line item for the logits-given path
on the peaked 1024 x 151936 fp32 logits.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lp|reference]
                       [--tp N]
For N > 1 launch one process per GPU with torch.distributed.run; every rank
runs its own batch of rows (weak scaling, no collective on the data path) and
rank 0 prints the whole-job throughput over the slowest rank's time.
With --tp N (N = the number of ranks, 2 or 4) the ranks instead split the
vocabulary: each holds 1/N of W, computes its quarter states, all-gathers them
over NCCL and merges (vocab parallel, strong scaling: the same 512 rows per
step whatever N).
"""

from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "selected-token logprobs/sec at T=512,d=4096,V=151936 bf16; % of roofline"
WORKLOAD = "fused_qwen3_8b"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "lp_linear_kernel.fused_qwen3_8b.txt")
LOGITS_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "lp_logits_final_kernel.logits_peaked.txt")
# the sources that define the fused kernel and the logits kernel, hashed in
# this order
LINEAR_SOURCES = [os.path.join(ROOT, "invariant_token_logprobs_gb300", "csrc", f)
                  for f in ("lp_linear.cu", "lp_tcgen05.cuh", "lp_device.cuh")]
LOGITS_SOURCES = [os.path.join(ROOT, "invariant_token_logprobs_gb300", "csrc", f)
                  for f in ("lp_logits.cu", "lp_device.cuh")]
BACKWARD_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "backward.fused_qwen3_8b.txt")
BACKWARD_SOURCES = [os.path.join(ROOT, "invariant_token_logprobs_gb300", "csrc", f)
                    for f in ("lp_backward.cu", "lp_linear.cu", "lp_tcgen05.cuh", "lp_device.cuh")]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    # 1000 steps of the headline workload keep the GPU busy ~0.4 s, several
    # refreshes of nvidia-smi's clock readings (about every 100 ms)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["lp", "reference"], default="lp")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-logits", action="store_true", help="skip the logits-path line item")
    p.add_argument("--no-backward", action="store_true", help="skip the backward line item")
    p.add_argument("--no-sweep", action="store_true", help="skip the batch-size sweep item")
    p.add_argument("--no-tp", action="store_true",
                   help="skip the per-rank vocabulary-parallel latency item")
    p.add_argument("--tp", type=int, default=0,
                   help="vocabulary-parallel ranks, 1, 2 or 4 (must equal the number of "
                        "processes); 0: the default replica mode")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    return p.parse_args(argv)


# --------------------------------------------------------------------- helpers

def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(v: float, world: int, device) -> float:
    """The largest of one float per rank (every rank gets it); identity when
    world == 1.  `device` is where the collective's tensor lives (the GPU for
    NCCL, the CPU for gloo)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(rows_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Rows of all ranks per second of the slowest rank (weak scaling)."""
    return world * rows_per_rank * steps / (max_ms / 1e3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def code_text(src: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and empty lines:
    what a profile's numbers depend on (an edit of a comment leaves it as is)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def sha256_files(paths) -> str:
    """SHA-256 of the files' code (code_text) concatenated in the given order."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(code_text(f.read()).encode("utf-8"))
        h.update(b"\n")
    return h.hexdigest()


def profile_traffic(summary=PROFILE_SUMMARY, sources=LINEAR_SOURCES,
                    field="dram_bytes_per_launch_full_size"):
    """DRAM bytes per launch of a kernel (or per call, for `field`) from its
    committed ncu summary, or None when the summary is absent or was taken on
    different kernel sources."""
    if not os.path.exists(summary):
        return None
    fields = {}
    with open(summary) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_sha256") != sha256_files(sources):
        return None
    try:
        return float(fields[field])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 20):
        self.device_index = device_index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="lp_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            cmd = ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                   "--format=csv,noheader,nounits", "-lms", str(self.period_ms)]
            if shutil.which("stdbuf"):  # line-buffered, so no sample is lost when it stops
                cmd = ["stdbuf", "-oL"] + cmd
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0:  # wait for the first sample
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.3)  # readings lag the GPU by up to ~100 ms: take those after the end
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self, t_begin: float, t_end: float):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                    except ValueError:
                        continue
            os.unlink(self.path)
        # nvidia-smi refreshes these readings about every 100 ms, so a sample
        # shows the state up to ~100 ms earlier: the window runs to 150 ms past
        # the end of the timed region and starts 100 ms into it when it is long
        # enough (earlier samples still show the GPU before the load)
        lo = t_begin + 0.1 if t_end - t_begin > 0.3 else t_begin
        inside = [r for r in rows if lo <= r[0] <= t_end + 0.15]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside),
                "window": ("timed region, shifted by nvidia-smi's ~100 ms refresh"
                           if inside else "nearest samples (timed region shorter than sampling)")}


# ------------------------------------------------------------- CPU oracle legs

def oracle_sample_seconds(h_host, w_host, y_host, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.linear_selected_logprob(h_host[rows], w_host, y_host[rows])
    return time.perf_counter() - t0


def cpu_baseline(x, budget_s: float):
    """The fp64 oracle as it stands on the same workload, on this host's cores:
    all rows, repeated until about `budget_s` seconds of CPU work."""
    import numpy as np
    h = x.H.float().cpu().numpy()
    w = x.W.float().cpu().numpy()
    y = x.y.cpu().numpy()
    T = h.shape[0]
    rows = np.arange(T)
    done, sec = 0, 0.0
    while sec < budget_s:
        sec += oracle_sample_seconds(h, w, y, rows)
        done += T
    return {"value": done / sec, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"{done // T} pass(es) over all {T} rows of {WORKLOAD} (d=4096, full V=151936), "
                      f"fp64 numpy oracle, {sec:.1f} s"}


def run_reference(args):
    """--impl reference: the fp64 CPU oracle, timed per step on a bounded row sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch
    from invariant_token_logprobs_gb300 import synth
    import oracle

    torch.set_num_threads(host_cores())
    x = synth.fused_inputs(WORKLOAD, device="cpu")
    h = x.H.float().numpy()
    w64 = x.W.double().numpy()  # the oracle's own dtype, converted once outside the steps
    y = x.y.numpy()
    T = h.shape[0]
    # size each step so the whole run stays within about two minutes
    t0 = time.perf_counter()
    oracle.linear_selected_logprob(h[:4], w64, y[:4])
    per4 = time.perf_counter() - t0
    per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    rows_per_step = int(max(1, min(T, 4 * per_step_budget / max(per4, 1e-6))))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        r = rng.integers(0, T, rows_per_step)
        oracle.linear_selected_logprob(h[r], w64, y[r])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = rng.integers(0, T, rows_per_step)
        oracle.linear_selected_logprob(h[r], w64, y[r])
    sec = time.perf_counter() - t0
    value = rows_per_step * args.steps / sec
    sample = (f"{rows_per_step} random rows of {WORKLOAD} per step (d=4096, full V=151936), "
              f"fp64 numpy oracle, W pre-converted to fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T, "d": 4096, "V": 151936, "seed": 2,
                   "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": host_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- GPU arm

def run_lp(args):
    import torch
    import torch.distributed as dist
    from invariant_token_logprobs_gb300 import lp, synth

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = lp.load()
    peaks, peaks_kind = load_peaks()

    spec = synth.WORKLOADS[WORKLOAD]
    x = synth.fused_inputs(WORKLOAD, device=dev, seed=spec.seed + 1000 * rank)
    T, d = x.H.shape
    V = x.W.shape[0]
    ws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=dev)
    logp = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over(v: float) -> float:
        return max_over_ranks(v, world, dev)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(max(3, args.warmup)):
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
    K = args.steps
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    torch.cuda.nvtx.range_push("lp.bench.fused_timed")
    ev0.record(stream)
    for _ in range(K):
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
    ev1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_end = time.time()
    barrier()
    sampler.stop()
    clocks = sampler.summary(t_begin, t_end)
    err_word = lp.lp_get_device_error(ws)
    if err_word != 0:
        raise RuntimeError(f"device-side wait gave up (error word {err_word})")
    total_ms = max_over(ev0.elapsed_time(ev1))
    ms_per_step = total_ms / K
    value = whole_job_throughput(T, K, world, total_ms)

    # the dominant kernel alone: a second loop of the same length, in which the
    # library records an event pair around every tensor-core kernel launch
    k_start = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    k_stop = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for ev in k_start + k_stop:  # torch creates an event on its first record
        ev.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        lp.lp_set_kernel_timing_events(k_start[i], k_stop[i])
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
    torch.cuda.synchronize()
    lp.lp_set_kernel_timing_events(None, None)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(k_start, k_stop))
    kernel_ms = max_over(kernel_ms)

    # the repeat property of the pages' candidates (distinct results in 10
    # repeats): ten more calls on the same inputs, each output hashed
    torch.cuda.nvtx.range_push("lp.bench.repeats")
    hashes = []
    for _ in range(10):
        lp.lp_linear_logprob(x.H, x.W, x.y, logp, ent, ws)
        both = torch.cat([logp, ent]).cpu().view(torch.int32).numpy().tobytes()
        hashes.append(hashlib.sha256(both).hexdigest())
    torch.cuda.nvtx.range_pop()
    repeats = {"calls": 10, "distinct_results": len(set(hashes)),
               "outputs_sha256": hashes[0][:16],
               "note": "logp and entropy of the headline inputs, hashed after each call"}

    # the other two properties the pages grade, on the same inputs (one GPU):
    # 2 and 4 vocabulary shards merged against the unsharded call, and rows
    # computed in batches of 1 and 7 against the same rows of the T-row call
    torch.cuda.nvtx.range_push("lp.bench.properties")
    ref = torch.cat([logp, ent]).view(torch.int32)
    tp_equal = {}
    for n in (2, 4):
        parts = []
        for i in range(n):
            b, e = lp.vocab_shard_range(V, i, n)
            parts.append(lp.linear_logprob_partials(x.H, x.W[b:e], x.y, V, i, n))
        m_lp, m_ent = lp.merge_partials(parts)
        tp_equal[f"tp{n}_equals_tp1"] = bool(torch.equal(torch.cat([m_lp, m_ent]).view(torch.int32),
                                                         ref))
    batch_equal = True
    for r0, rows in ((0, 7), (T // 2, 1), (T - 7, 7)):
        s_lp, s_ent = lp.linear_logprob(x.H[r0:r0 + rows].contiguous(), x.W,
                                        x.y[r0:r0 + rows].contiguous())
        batch_equal &= bool(torch.equal(s_lp.view(torch.int32), logp[r0:r0 + rows].view(torch.int32))
                            and torch.equal(s_ent.view(torch.int32),
                                            ent[r0:r0 + rows].view(torch.int32)))
    torch.cuda.nvtx.range_pop()
    properties = dict(tp_equal, batch_bitwise=batch_equal,
                      distinct_results_in_repeats=repeats["distinct_results"],
                      note="checked on the headline inputs on one GPU after the timed loops: "
                           "shards' quarter states merged in the fixed order, and sub-batches "
                           "of 1 and 7 rows, bit for bit against the T-row call")

    flops = 2.0 * T * d * V
    w_bytes = 2.0 * V * d + 2.0 * T * d + 8.0 * T + 8.0 * T
    peak_tf = peaks["bf16_tflops"]
    achieved_tf = flops / (kernel_ms / 1e3) / 1e12
    roofline_us = max(flops / (peak_tf * 1e12), w_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e6
    roofline = {
        "bound": "tensor", "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s",
        "frac": achieved_tf / peak_tf, "traffic": profile_traffic(),
        "frac_vs_sustained": achieved_tf / peaks.get("bf16_tflops_sustained", peak_tf),
        "kernel": "lp_linear_kernel", "kernel_us": kernel_ms * 1e3,
        "timing": "kernel_us from a second loop of the same length with an event pair around "
                  "every tensor-core kernel; value and ms_per_step from the plain loop",
        "algorithmic_flops_per_launch": flops, "roofline_us": roofline_us,
        "peak_source": f"{peaks_kind} bf16 burst ({'MEASURED_PEAKS.json' if peaks_kind == 'measured' else 'fallback'})",
    }

    # end to end through the C ABI with host buffers: every step copies H and
    # the targets in from pinned host memory and logp and entropy out.
    # Pipelined (the headline): the copies run on a second stream, double
    # buffered, so step i+1's inputs arrive while step i computes.  Serial:
    # copy in, compute, copy out, one after the other on one stream.
    h_host = x.H.cpu().pin_memory()
    y_host = x.y.cpu().pin_memory()
    lp_host = [torch.empty(T, pin_memory=True) for _ in range(2)]
    ent_host = [torch.empty(T, pin_memory=True) for _ in range(2)]
    h_dev = [torch.empty_like(x.H) for _ in range(2)]
    y_dev = [torch.empty_like(x.y) for _ in range(2)]
    lp_dev = [torch.empty(T, device=dev) for _ in range(2)]
    ent_dev = [torch.empty(T, device=dev) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    K2 = K  # as many steps as the device-resident loop, so both run in the same power state

    def pipelined(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        copy_stream.wait_stream(stream)

        def copy_in(i):
            b = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(done[b])  # step i-2 has read buffer b
                h_dev[b].copy_(h_host, non_blocking=True)
                y_dev[b].copy_(y_host, non_blocking=True)
                in_ready[b].record(copy_stream)

        copy_in(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(in_ready[b])
            lp.lp_linear_logprob(h_dev[b], x.W, y_dev[b], lp_dev[b], ent_dev[b], ws)
            done[b].record(stream)
            if i + 1 < n:
                copy_in(i + 1)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(done[b])
                lp_host[b].copy_(lp_dev[b], non_blocking=True)
                ent_host[b].copy_(ent_dev[b], non_blocking=True)
        stream.wait_stream(copy_stream)

    def serial(n):
        for _ in range(n):
            h_dev[0].copy_(h_host, non_blocking=True)
            y_dev[0].copy_(y_host, non_blocking=True)
            lp.lp_linear_logprob(h_dev[0], x.W, y_dev[0], lp_dev[0], ent_dev[0], ws)
            lp_host[0].copy_(lp_dev[0], non_blocking=True)
            ent_host[0].copy_(ent_dev[0], non_blocking=True)

    def timed(fn, n):
        fn(3)
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(n)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over(e0.elapsed_time(e1))

    torch.cuda.nvtx.range_push("lp.bench.e2e")
    e2e_ms = timed(pipelined, K2)
    serial_ms = timed(serial, K2)
    torch.cuda.nvtx.range_pop()
    # the host copies (slot 1: the pipelined run, slot 0: the serial run) hold the
    # same bits as the device-resident run's outputs
    ref_lp = logp.cpu().view(torch.int32)
    ref_ent = ent.cpu().view(torch.int32)
    for slot in range(2 if K2 > 1 else 1):
        if not (torch.equal(lp_host[slot].view(torch.int32), ref_lp) and
                torch.equal(ent_host[slot].view(torch.int32), ref_ent)):
            raise RuntimeError("end-to-end outputs differ from the device-resident run")
    e2e = {"value": whole_job_throughput(T, K2, world, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": h_host.numel() * h_host.element_size() + y_host.numel() * 8,
           "d2h_bytes_per_step": 8 * T, "steps": K2,
           "serial_value": whole_job_throughput(T, K2, world, serial_ms),
           "note": "W (the LM-head weight) is resident model state; per step H and targets go in "
                   "from pinned host memory and logp/entropy come out; value: copies on a second "
                   "stream, double-buffered, overlapping the previous step's compute; "
                   "serial_value: copy in, compute, copy out in sequence on one stream; neither "
                   "loop records the per-kernel timing events of the device-resident loop"}

    logits_item = None
    if not args.no_logits:
        del h_host
        torch.cuda.nvtx.range_push("lp.bench.logits")
        logits_item = bench_logits(lp, synth, torch, dev, stream, peaks, peaks_kind, max_over,
                                   world, rank)
        torch.cuda.nvtx.range_pop()

    backward_item = None
    if not args.no_backward:
        torch.cuda.nvtx.range_push("lp.bench.backward")
        backward_item = bench_backward(lp, torch, x, dev, stream, peaks, peaks_kind, max_over,
                                       world)
        torch.cuda.nvtx.range_pop()

    tp_item = None
    if not args.no_tp and world == 1:
        torch.cuda.nvtx.range_push("lp.bench.vocab_parallel")
        tp_item = bench_vocab_parallel(lp, torch, x, dev, stream)
        torch.cuda.nvtx.range_pop()

    # last of the GPU items: its seconds of load would otherwise leave the
    # items after it running in a hotter, more power-capped state
    sweep_item = None
    if not args.no_sweep:
        torch.cuda.nvtx.range_push("lp.bench.batch_sweep")
        sweep_item = bench_batch_sweep(lp, torch, x, dev, stream, peaks, peaks_kind, max_over)
        torch.cuda.nvtx.range_pop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded bf16 H (RMS-normalised N(0,1)) and W ~ N(0, 0.02^2), uniform targets",
        "config": {"workload": WORKLOAD, "T": T, "d": d, "V": V, "seed": spec.seed,
                   "rows_per_gpu": T, "l2": "inputs larger than L2 (W = 1.245 GB), no flush",
                   "parallelism": f"replicas x{world} (rows partitioned, no collective)"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clocks,
        "repeats": repeats,
        "properties": properties,
        "backend": lp.lp_backend_id(),
        "logits_path": logits_item,
        "backward_path": backward_item,
        "vocab_parallel": tp_item,
        "batch_sweep": sweep_item,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_vocab_parallel(lp, torch, x, dev, stream):
    """Line item: what one rank of a 2- or 4-way vocabulary split runs at the
    headline shape, timed on this GPU (the ranks' shards are the same size):
    the forward (its shard's quarter states, then the merge of all ranks'
    states) and the training backward (its shard's backward, then the merge of
    all ranks' partial grad_H).  The all-gathers between them are not included
    (one GPU): they move 32 T bytes per quarter and 4 T d bytes per rank."""
    T, d = x.H.shape
    V = x.W.shape[0]
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    gl = torch.randn(T, generator=g, device=dev)
    ge = torch.randn(T, generator=g, device=dev)
    logp, ent, lse = lp.linear_logprob_lse(x.H, x.W, x.y)
    out = {"workload": "fused_qwen3_8b, one rank's share", "T": T, "d": d, "V": V,
           "note": "per-rank kernels and merges on one GPU; all-gathers excluded"}

    def timed(fn, n=10):
        for _ in range(2):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n * 1e3

    for n in (2, 4):
        b, e = lp.vocab_shard_range(V, 0, n)
        w0 = x.W[b:e]
        fws = torch.empty(lp.lp_linear_logprob_partials_workspace_size(T, d, V, n),
                          dtype=torch.uint8, device=dev)
        part = torch.empty((T, 4 // n, lp.STATE_FLOATS), device=dev)
        parts = [part] * n  # every rank's states have this shape; the merge reads them all
        m_lp = torch.empty(T, device=dev)
        m_ent = torch.empty(T, device=dev)
        m_lse = torch.empty(T, device=dev)

        def fwd():
            lp.lp_linear_logprob_partials(x.H, w0, x.y, V, 0, n, part, fws)
            lp.lp_merge_partials_lse(parts, T, m_lp, m_ent, m_lse)

        bws = torch.empty(lp.lp_linear_logprob_partials_backward_workspace_size(T, d, V, n),
                          dtype=torch.uint8, device=dev)
        gh_part = torch.empty((T, d), device=dev)
        gw_rows = torch.empty((e - b, d), device=dev)
        gh_parts = [gh_part] * n
        gH = torch.empty((T, d), device=dev)

        def bwd():
            lp.lp_linear_logprob_partials_backward(x.H, w0, x.y, V, 0, n, 1.0, lse, ent, gl, ge,
                                                   gh_part, gw_rows, bws)
            lp.lp_merge_grad_h_partials(gh_parts, gH)

        f_us = timed(fwd)
        b_us = timed(bwd)
        if lp.lp_get_device_error(bws) != 0 or lp.lp_get_device_error(fws) != 0:
            raise RuntimeError("device-side wait gave up in the vocabulary-parallel item")
        out[f"tp{n}"] = {"forward_us_per_rank": f_us, "backward_us_per_rank": b_us}
    return out


def bench_backward(lp, torch, x, dev, stream, peaks, peaks_kind, max_over, world):
    """Line item: lp_linear_logprob_backward (grad_H and grad_W) on the headline shape."""
    T, d = x.H.shape
    V = x.W.shape[0]
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    gl = torch.randn(T, generator=g, device=dev)
    ge = torch.randn(T, generator=g, device=dev)
    ws = torch.empty(lp.lp_linear_logprob_backward_workspace_size(T, d, V), dtype=torch.uint8,
                     device=dev)
    gH = torch.empty((T, d), device=dev)
    gW = torch.empty((V, d), device=dev)
    # entropy and log-sum-exp as a training step keeps them from its forward pass
    lse = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    logp = torch.empty(T, device=dev)
    fws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8, device=dev)
    lp.lp_linear_logprob_lse(x.H, x.W, x.y, 1.0, logp, ent, lse, fws)
    for _ in range(2):
        lp.lp_linear_logprob_backward(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, gW, ws)
    K = 10
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        lp.lp_linear_logprob_backward(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, gW, ws)
    e1.record(stream)
    torch.cuda.synchronize()
    if lp.lp_get_device_error(ws) != 0:
        raise RuntimeError("device-side wait gave up in the backward")
    ms = max_over(e0.elapsed_time(e1)) / K
    flops = 3 * 2.0 * T * d * V  # logits recompute, G W, G^T H (forward statistics saved)
    tf = flops / (ms / 1e3) / 1e12
    del gW
    # the same call with grad_W in bf16 (lp_linear_logprob_backward_ex)
    gW16 = torch.empty((V, d), device=dev, dtype=torch.bfloat16)
    for _ in range(2):
        lp.lp_linear_logprob_backward_ex(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, gW16, ws)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        lp.lp_linear_logprob_backward_ex(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, gW16, ws)
    e1.record(stream)
    torch.cuda.synchronize()
    if lp.lp_get_device_error(ws) != 0:
        raise RuntimeError("device-side wait gave up in the backward")
    ms16 = max_over(e0.elapsed_time(e1)) / K
    tf16 = flops / (ms16 / 1e3) / 1e12
    del gW16
    # grad_W added into a float32 main gradient (the accumulate mode)
    main = torch.zeros((V, d), device=dev)
    for _ in range(2):
        lp.lp_linear_logprob_backward_ex(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, main, ws,
                                         accumulate=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        lp.lp_linear_logprob_backward_ex(x.H, x.W, x.y, 1.0, lse, ent, gl, ge, gH, main, ws,
                                         accumulate=True)
    e1.record(stream)
    torch.cuda.synchronize()
    if lp.lp_get_device_error(ws) != 0:
        raise RuntimeError("device-side wait gave up in the backward")
    ms_acc = max_over(e0.elapsed_time(e1)) / K
    del ws, main
    # algorithmic bytes of one call: W read by the logits recompute and by G W,
    # H once, G (bf16 [T, V]) written once and read by both products, the
    # fp32 partial grad_H written and read (28 when V % 64 == 0, else 19),
    # grad_H and the fp32 grad_W written once
    n_part = 28 if V % 64 == 0 else 19
    alg_bytes = (2 * V * d * 2 + T * d * 2 + 3 * T * V * 2 + 2 * n_part * T * d * 4
                 + T * d * 4 + V * d * 4)
    return {"workload": "fused_qwen3_8b backward (grad_H and grad_W, fp32 out)", "T": T, "d": d,
            "V": V, "value": world * T / (ms / 1e3), "unit": "tokens/s", "us_per_call": ms * 1e3,
            "bf16_grad_W": {"us_per_call": ms16 * 1e3, "achieved_tflops": tf16,
                            "frac": tf16 / peaks["bf16_tflops"],
                            "note": "grad_W written in bf16 (lp_linear_logprob_backward_ex)"},
            "fp32_accumulate": {"us_per_call": ms_acc * 1e3,
                                "note": "grad_W added into a float32 main gradient "
                                        "(LP_GRAD_W_FLOAT32_ACCUMULATE): 4 V d more bytes read "
                                        "than writing it, and no second pass to add it"},
            "gpu_launches_per_call": 3,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                         "traffic": profile_traffic(BACKWARD_PROFILE_SUMMARY, BACKWARD_SOURCES,
                                                    "dram_bytes_per_call_full_size"),
                         "algorithmic_bytes_per_call": float(alg_bytes),
                         "kernel": "whole backward call (3 tensor-core kernels; the split sum of grad_H runs in the grad_W product)",
                         "algorithmic_flops_per_call": flops,
                         "note": "log-sum-exp and entropy saved from the forward (lp_linear_logprob_lse); one memset + 3 kernels per call",
                         "peak_source": f"{peaks_kind} bf16 burst"}}


def bench_batch_sweep(lp, torch, x, dev, stream, peaks, peaks_kind, max_over):
    """Secondary line item: the fused call at other batch sizes on the same W
    (rows of the headline H repeated; timing only), each against its own
    roofline: the slower of 2 T d V at the bf16 burst peak and W read once at
    the copy bandwidth."""
    T0, d = x.H.shape
    V = x.W.shape[0]
    sizes = (1, 16, 128, 256, 512, 2048)
    reps = (max(sizes) + T0 - 1) // T0
    H_all = torch.cat([x.H] * reps)
    y_all = torch.cat([x.y] * reps)
    out = {}
    for T in sizes:
        H = H_all[:T].contiguous()
        y = y_all[:T].contiguous()
        ws = torch.empty(lp.lp_linear_logprob_workspace_size(T, d, V), dtype=torch.uint8,
                         device=dev)
        logp = torch.empty(T, device=dev)
        ent = torch.empty(T, device=dev)
        for _ in range(3):
            lp.lp_linear_logprob(H, x.W, y, logp, ent, ws)
        K = 20
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(K):
            lp.lp_linear_logprob(H, x.W, y, logp, ent, ws)
        e1.record(stream)
        torch.cuda.synchronize()
        us = max_over(e0.elapsed_time(e1)) / K * 1e3
        flops_us = 2.0 * T * d * V / (peaks["bf16_tflops"] * 1e12) * 1e6
        bytes_us = 2.0 * V * d / (peaks["hbm_gbs"] * 1e9) * 1e6
        out[str(T)] = {"us_per_call": us, "tokens_per_s": T / (us * 1e-6),
                       "bound": "hbm" if bytes_us >= flops_us else "tensor",
                       "frac": max(flops_us, bytes_us) / us}
    return {"workload": "fused_qwen3_8b W with T rows", "d": d, "V": V,
            "timing": "20 back-to-back lp_linear_logprob calls per size (kernel + merge)",
            "roofline": "max(2 T d V / measured bf16 burst, 2 V d bytes / measured copy bandwidth)",
            "peak_source": peaks_kind, "sizes": out}


def bench_logits(lp, synth, torch, dev, stream, peaks, peaks_kind, max_over, world, rank):
    """Secondary line item: the logits-given path on the peaked workload."""
    z = synth.logits_inputs("logits_peaked", device=dev, seed=1 + 1000 * rank)
    T, V = z.z.shape
    logp = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    for _ in range(5):
        lp.lp_logprob_from_logits(z.z, z.y, logp, ent)
    K = 50
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        lp.lp_logprob_from_logits(z.z, z.y, logp, ent)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over(e0.elapsed_time(e1)) / K
    nbytes = 4.0 * T * V + 8.0 * T + 8.0 * T
    gbs = nbytes / (ms / 1e3) / 1e9
    # the backward (dL/dz) on the same logits, with the forward's log Z and entropy
    _, ent_s, lse_s = lp.logprob_from_logits_lse(z.z, z.y)
    g = torch.Generator(device=dev).manual_seed(17)
    gl = torch.randn(T, generator=g, device=dev)
    ge = torch.randn(T, generator=g, device=dev)
    grad = torch.empty_like(z.z)
    for _ in range(3):
        lp.lp_logprob_from_logits_backward(z.z, z.y, 1.0, lse_s, ent_s, gl, ge, grad)
    KB = 20
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(KB):
        lp.lp_logprob_from_logits_backward(z.z, z.y, 1.0, lse_s, ent_s, gl, ge, grad)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_b = max_over(e0.elapsed_time(e1)) / KB
    bytes_b = 8.0 * T * V + 32.0 * T
    gbs_b = bytes_b / (ms_b / 1e3) / 1e9
    del grad
    backward = {"us_per_call": ms_b * 1e3, "kernel": "lp_logits_grad_kernel",
                "achieved": gbs_b, "unit": "GB/s", "frac": gbs_b / peaks["hbm_gbs"],
                "algorithmic_bytes_per_launch": bytes_b,
                "note": "lp_logprob_from_logits_backward, fp32 dL/dz [T, V] written (logits read "
                        "once, gradient written once)"}
    return {"workload": "logits_peaked", "T": T, "V": V, "value": whole_job_throughput(T, 1, world, ms),
            "unit": "rows/s", "us_per_call": ms * 1e3, "gpu_launches_per_call": 1,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": profile_traffic(LOGITS_PROFILE_SUMMARY, LOGITS_SOURCES),
                         "kernel": "lp_logits_final_kernel",
                         "algorithmic_bytes_per_launch": nbytes,
                         "peak_source": f"{peaks_kind} copy bandwidth"},
            "backward": backward}


def run_tp(args):
    """--tp N: the vocabulary-parallel step (partials on 1/N of W, NCCL
    all-gather of the 32-byte quarter states, fixed merge) on N ranks."""
    import torch
    import torch.distributed as dist
    from invariant_token_logprobs_gb300 import lp, synth
    from invariant_token_logprobs_gb300 import vocab_parallel as vp

    world, rank, local = dist_env()
    if world != args.tp or args.tp not in (1, 2, 4):
        raise SystemExit(f"--tp {args.tp} needs exactly that many processes (1, 2 or 4); got {world}")
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lp.load()
    x = synth.fused_inputs(WORKLOAD, device=dev)  # every rank: the same rows
    T, d = x.H.shape
    V = x.W.shape[0]
    _, n, b, e = vp.shard_of_rank(V)
    w_shard = x.W[b:e].clone()
    del x.W
    ws = torch.empty(lp.lp_linear_logprob_partials_workspace_size(T, d, V, n), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step():
        return vp.vocab_parallel_linear_logprob(x.H, w_shard, x.y, V, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    K = args.steps
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        out = step()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    line = {
        "metric": METRIC, "value": T * K / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded bf16 H (RMS-normalised N(0,1)) and W ~ N(0, 0.02^2), uniform targets",
        "config": {"workload": WORKLOAD, "T": T, "d": d, "V": V, "seed": 2,
                   "parallelism": f"vocab-parallel tp{world} (1/{world} of W per rank, all-gather "
                                  f"of quarter states, fixed merge)",
                   "l2": "inputs larger than L2, no flush"},
        "gpu_launches": 3 * K, "e2e": None, "roofline": None, "cpu_baseline": None,
        "backend": lp.lp_backend_id(),
        "logp_checksum": float(out[0].double().sum()),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.tp:
        return run_tp(args)
    return run_lp(args)


if __name__ == "__main__":
    sys.exit(main())
