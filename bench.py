#!/usr/bin/env python
"""Benchmark of the exact-attention library on one GB300 (or N replicas).

Metric: attention TFLOP/s for forward and forward+backward, bf16, on the long
workload (B=2, H=16, N=8192, d=128, causal, K x 3 in heads 0-7).  FLOPs are
4*B*H*N^2*d for the forward, halved for causal, and 2.5x that for the
backward.  A step is one forward (fa_fwd) plus one backward (fa_bwd) over the
same inputs, which are resident in device memory when the timed region starts.
Q, K, V and dO are 67 MB each (268 MB together), larger than the 129 MB L2,
so no L2 flush is needed between steps.

Launch:  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
         python bench.py --case NAME [--batch B] [--iters K]   (one workload, for profilers)
For N > 1 the driver starts one process per GPU with torchrun; every rank
runs the same workload on its own GPU (independent replicas: the units of this
path, (batch, head) pairs, need no exchange), and rank 0 prints one JSON line
with the total work of all ranks divided by the slowest rank's time.

``--impl reference`` times the float64 CPU oracle (the correctness baseline)
on the machine's host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

N_CORES = len(os.sched_getaffinity(0))
# The oracle's BLAS must use exactly the host cores we report.
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(N_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(N_CORES))

METRIC = "attention TFLOP/s fwd & fwd+bwd (bf16, d=128, N=8k causal), % of tensor peak"
LONG = dict(B=2, H=16, N=8192, d=128, causal=True, k_boost=3.0)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads' sub-measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="run one workload --iters times on cuda:0 and exit (for profilers; prints no bench line)")
    ap.add_argument("--batch", type=int, default=0, help="--case: override the batch (dense, decode)")
    ap.add_argument("--iters", type=int, default=3, help="--case: calls of the workload")
    return ap.parse_args()


CASES = ["long", "mid", "varlen", "decode", "fp8", "window", "prefill"]


def run_case(a):
    """Runs one named workload a few times on cuda:0 for a profiler:
    long / mid (fa_fwd + fa_bwd), varlen (packed fwd + bwd), decode (split-KV),
    fp8 (quantise + e4m3 forward on the long shape), window (4096-key causal
    window, fwd + bwd), prefill (chunked-prefill forward).  Inputs are the
    seeded synthetic tensors of the benchmark workloads; the batch of the dense
    and decode cases can be reduced so that a profiler's save and restore of
    device memory stays small.  Returns the process exit status."""
    import torch

    import synth
    from exact_attention_94_gb300 import ops

    w = synth.WORKLOADS["long" if a.case == "fp8" else a.case]
    B = a.batch or w.B
    if a.case == "fp8":
        x = synth.make_dense(B, w.H, w.N, w.d, seed=w.seed, k_boost=w.k_boost, device="cuda", with_do=False)
        signs = synth.hadamard_signs(w.d, 0).cuda()
        for _ in range(a.iters):
            ops.fwd_fp8(x["q"], x["k"], x["v"], signs, causal=True)
    elif a.case == "window":
        x = synth.make_dense(B, w.H, w.N, w.d, seed=0, device="cuda")
        for _ in range(a.iters):
            o, lse = ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window)
            ops.bwd_masked(x["q"], x["k"], x["v"], o, lse, x["do"], window=w.window)
    elif a.case == "prefill":
        x = synth.make_masked(B, w.N, w.n_k, w.H, w.h_kv, w.d, seed=0, device="cuda", with_do=False)
        for _ in range(a.iters):
            ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window)
    elif a.case == "decode":
        x = synth.make_decode(B, w.H, w.N, w.d, seed=0, device="cuda")
        for _ in range(a.iters):
            ops.decode(x["q"], x["k"], x["v"])
    elif a.case == "varlen":
        lengths = synth.varlen_lengths(w.B, w.len_lo, w.len_hi, w.seed)
        x = synth.make_varlen(lengths, w.H, w.d, seed=0, device="cuda")
        cu = x["cu_seqlens"].cuda()
        for _ in range(a.iters):
            o, lse = ops.fwd_varlen(x["q"], x["k"], x["v"], cu, int(lengths.max()), causal=True)
            ops.bwd_varlen(x["q"], x["k"], x["v"], o, lse, x["do"], cu, int(lengths.max()), causal=True)
    else:
        x = synth.make_dense(B, w.H, w.N, w.d, seed=0, k_boost=w.k_boost, device="cuda")
        for _ in range(a.iters):
            o, lse = ops.fwd(x["q"], x["k"], x["v"], causal=w.causal)
            ops.bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=w.causal)
    torch.cuda.synchronize()
    err = ops.device_error()
    print(f"{a.case}: {a.iters} iterations, device error {err}")
    return 0 if err == 0 else 1


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                             parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 0.5 * max(x[2] for x in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_min_mhz": min(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(loaded)}


# ---------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "exact_attention_94_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_name, sources):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's sources changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", summary_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != source_sha(*sources):
        return None
    return float(m_b.group(1))


class Timer:
    """CUDA events on the current (launching) stream."""

    def __init__(self, torch):
        self.t = torch
        self.ev = []

    def mark(self):
        e = self.t.cuda.Event(enable_timing=True)
        e.record()
        self.ev.append(e)
        return e


def run_ours(args):
    import torch
    import torch.distributed as dist

    import synth
    from exact_attention_94_gb300 import _lib, accounting as acc, ops, replicas

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ops.lib()
    peaks = load_peaks()
    w = LONG
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    F = acc.fwd_flops(B, H, N, d, causal)
    x = synth.make_dense(B, H, N, d, seed=0, k_boost=w["k_boost"], device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(ops.lib().fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    have_bwd = True
    ops.fwd(q, k, v, causal=causal, out=o, lse=lse)
    try:
        ops.bwd(q, k, v, o, lse, do, causal=causal, workspace=ws)
    except _lib.FaError as e:
        if e.status != _lib.FA_ERR_UNSUPPORTED:
            raise
        have_bwd = False
    torch.cuda.synchronize()

    def step(tm=None):
        if tm is not None:
            tm.mark()
        ops.fwd(q, k, v, causal=causal, out=o, lse=lse)
        if tm is not None:
            tm.mark()
        if have_bwd:
            ops.bwd(q, k, v, o, lse, do, causal=causal, workspace=ws)
            if tm is not None:
                tm.mark()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    tm = Timer(torch)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        start = tm.mark()
        inner = Timer(torch)
        for _ in range(args.steps):
            step(inner)
        end = tm.mark()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    per = 3 if have_bwd else 2
    fwd_ms = [inner.ev[i * per].elapsed_time(inner.ev[i * per + 1]) for i in range(args.steps)]
    bwd_ms = ([inner.ev[i * per + 1].elapsed_time(inner.ev[i * per + 2]) for i in range(args.steps)]
              if have_bwd else [0.0])
    # the slowest rank sets every time (a no-op on one process)
    total_ms, fwd_mean, bwd_mean = replicas.max_over_ranks(
        [total_ms, statistics.mean(fwd_ms), statistics.mean(bwd_ms)], device="cuda")
    assert ops.device_error() == 0, "a bounded wait ran out inside a kernel"
    ms_step = total_ms / args.steps
    step_flops = F * (2.5 if have_bwd else 1.0)     # literal reading: fwd+bwd = 2.5x the forward
    value = replicas.whole_job_rate(world, step_flops, ms_step) / 1e12
    fwd_tf = F / (fwd_mean * 1e-3) / 1e12
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "long: B=2 H=16 N=8192 d=128 causal, K x3 in heads 0-7",
                   "step": "fa_fwd + fa_bwd" if have_bwd else "fa_fwd only (fa_bwd not built)",
                   "flops_convention": "fwd 4BHN^2d/2; fwd+bwd 2.5x fwd",
                   "l2": "inputs 268 MB > 129 MB L2, no flush", "parallelism": f"replicas x{world}"},
        "fwd_tflops": round(fwd_tf, 2),
        "fwd_frac_of_peak": round(fwd_tf / peaks["bf16_tflops"], 4),
        "fwdbwd_frac_of_peak": round(value / world / peaks["bf16_tflops"], 4),
    }
    if have_bwd:
        res["fwdbwd_tflops_3p5x"] = round(world * 3.5 * F / (ms_step * 1e-3) / 1e12, 2)
        res["bwd_tflops"] = round(2.5 * F / (bwd_mean * 1e-3) / 1e12, 2)
    # roofline of the dominant kernel (largest share of the step)
    if have_bwd and bwd_mean > fwd_mean:
        ach = 2.5 * F / (bwd_mean * 1e-3) / 1e12
        traffic = profiled_traffic("fa_bwd_long.md", ["fa_bwd.cu", "ptx.cuh", "fa_internal.h"])
        kname = "fa_bwd (main + pre/post kernels, timed together)"
    else:
        ach = fwd_tf
        traffic = profiled_traffic("fa_fwd_long.md", ["fa_fwd.cu", "ptx.cuh", "fa_internal.h"])
        kname = "fa_fwd_kernel"
    res["roofline"] = {"kernel": kname, "bound": "tensor", "achieved": round(ach, 2), "peak": peaks["bf16_tflops"],
                       "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": traffic,
                       "peak_source": f"{peaks['source']} bf16 burst"}
    res["clocks"] = clocks.summary()
    # The same rate against the tensor pipe's issue limit at the clock the bench
    # actually ran at: 8192 bf16 FLOP per clock per SM (an M = N = 128, K = 16
    # product issues every 64 cycles), times the SMs, times the sampled median
    # SM clock.  The measured GEMM peak above was taken at whatever clock the
    # GEMM loop held under the power cap, so the two fractions differ.
    n_sm = torch.cuda.get_device_properties(local).multi_processor_count
    mhz = res["clocks"].get("sm_mhz")
    if mhz:
        at_clock = 8192.0 * n_sm * mhz * 1e6 / 1e12
        res["roofline"]["clock_normalised"] = {
            "sm_mhz": mhz, "sms": n_sm, "flop_per_clk_per_sm": 8192, "peak_at_clock": round(at_clock, 1),
            "frac": round(ach / at_clock, 4), "fwd_frac": round(fwd_tf / at_clock, 4)}
    res["gpu_launches"] = args.steps * (1 + (3 if have_bwd else 0))
    return res, (x, o, lse, ws, have_bwd, F)


def run_e2e(args, ctx):
    """Same metric through the public API with host buffers: every step copies
    its q, k, v, dO from pinned host memory and reads its o, lse, dq, dk, dv
    back to pinned host memory.  Steps are pipelined over three streams
    (host-to-device copies of step i+1 and device-to-host copies of step i-1
    run while step i computes) with double-buffered device tensors; a step's
    forward starts once its q, k, v have landed (dO may still be on its way)
    and its o, lse go out while its backward runs.  The timed region spans
    all steps' copies and compute."""
    import torch

    from exact_attention_94_gb300 import ops

    x, o, lse, ws, have_bwd, F = ctx
    w = LONG
    names = ("q", "k", "v", "do")
    host_in = [{n: x[n].cpu().pin_memory() for n in names} for _ in range(2)]
    dev_in = [{n: torch.empty_like(x[n]) for n in names} for _ in range(2)]
    out_shapes = {"o": (x["q"].shape, torch.bfloat16), "lse": (lse.shape, torch.float32)}
    if have_bwd:
        out_shapes.update(dq=(x["q"].shape, torch.bfloat16), dk=(x["k"].shape, torch.bfloat16),
                          dv=(x["v"].shape, torch.bfloat16))
    dev_out = [{n: torch.empty(sh, dtype=dt, device="cuda") for n, (sh, dt) in out_shapes.items()} for _ in range(2)]
    host_out = [{n: torch.empty(sh, dtype=dt, pin_memory=True) for n, (sh, dt) in out_shapes.items()} for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ws2 = [ws, torch.empty_like(ws)]

    fwd_out = ("o", "lse")

    def run(steps, start=None, end=None):
        # per buffer: inputs of the forward landed, dO landed, forward done, step done,
        # results copied out (the buffer may be reused)
        ev_qkv, ev_do, ev_fwd, ev_done, ev_out = ([None, None] for _ in range(5))

        def copy_in(i):
            buf = i & 1
            with torch.cuda.stream(s_in):
                if ev_done[buf] is not None:
                    s_in.wait_event(ev_done[buf])
                for n in names:
                    dev_in[buf][n].copy_(host_in[buf][n], non_blocking=True)
                    if n == "v" or n == "do":
                        ev = torch.cuda.Event()
                        ev.record(s_in)
                        (ev_qkv if n == "v" else ev_do)[buf] = ev

        if start is not None:
            start.record(torch.cuda.current_stream())
            for st in (s_in, s_cmp, s_out):
                st.wait_event(start)
        copy_in(0)
        for i in range(steps):
            buf = i & 1
            if i + 1 < steps:
                copy_in(i + 1)
            d, out = dev_in[buf], dev_out[buf]
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_qkv[buf])  # the forward needs q, k, v only
                if ev_out[buf] is not None:
                    s_cmp.wait_event(ev_out[buf])
                ops.fwd(d["q"], d["k"], d["v"], causal=w["causal"], out=out["o"], lse=out["lse"])
                ev_fwd[buf] = torch.cuda.Event()
                ev_fwd[buf].record(s_cmp)
                if have_bwd:
                    s_cmp.wait_event(ev_do[buf])
                    ops.bwd(d["q"], d["k"], d["v"], out["o"], out["lse"], d["do"], causal=w["causal"],
                            workspace=ws2[buf], out=(out["dq"], out["dk"], out["dv"]))
                ev_done[buf] = torch.cuda.Event()
                ev_done[buf].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fwd[buf])  # o and lse go out while the backward runs
                for n in fwd_out:
                    host_out[buf][n].copy_(dev_out[buf][n], non_blocking=True)
                s_out.wait_event(ev_done[buf])
                for n in out_shapes:
                    if n not in fwd_out:
                        host_out[buf][n].copy_(dev_out[buf][n], non_blocking=True)
                ev_out[buf] = torch.cuda.Event()
                ev_out[buf].record(s_out)
        if end is not None:
            cur = torch.cuda.current_stream()
            for st in (s_in, s_cmp, s_out):
                e = torch.cuda.Event()
                e.record(st)
                cur.wait_event(e)
            end.record(cur)
        torch.cuda.synchronize()

    run(3)
    steps = max(4, args.steps)  # the pipeline's fill and drain (one step's copies each) spread over as many steps
    # the median of three timed loops: the host link is shared with the machine's other
    # GPUs, and one loop in a run has measured half the rate of the loops around it
    reps = []
    for _ in range(3):
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        run(steps, start, end)
        reps.append(start.elapsed_time(end) / steps)
    ms = sorted(reps)[1]
    flops = F * (2.5 if have_bwd else 1.0)
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    link = link_bandwidth(torch)
    # with the copies overlapped with compute and with each other, a step can go no faster
    # than its slower copy direction alone, nor than both directions' bytes at the joint rate
    copy_ms = max(h2d / link["h2d_gbs"], d2h / link["d2h_gbs"], (h2d + d2h) / link["both_directions_gbs"]) * 1e-6
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "CUDA events joined across the three streams; median of three timed loops",
            "loops_ms_per_step": [round(r, 4) for r in reps],
            "pipelining": "3 streams, double-buffered device tensors",
            "link": {**link, "copy_ms_per_step": round(copy_ms, 4),
                     "copy_bound_tflops": round(flops / (copy_ms * 1e-3) / 1e12, 2)}}


def link_bandwidth(torch, nbytes=256 << 20, reps=5, trials=3):
    """Host<->device copy rates between pinned host memory and the GPU (CUDA
    events), for judging the e2e figure: each direction alone, and both at
    once on two streams (what the pipelined e2e leg does), as total bytes
    over the joint time; the best of a few trials."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()

    def both():
        with torch.cuda.stream(s_a):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s_b):
            h_out.copy_(d_out, non_blocking=True)

    out = {}
    for name, fn, nb in (("h2d_gbs", lambda: d_in.copy_(h_in, non_blocking=True), nbytes),
                         ("d2h_gbs", lambda: h_out.copy_(d_out, non_blocking=True), nbytes),
                         ("both_directions_gbs", both, 2 * nbytes)):
        fn()
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(trials):  # the link's rate varies from run to run: keep the best trial
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream()
            s.record(cur)
            for st in (s_a, s_b):
                st.wait_event(s)
            for _ in range(reps):
                fn()
            for st in (s_a, s_b):
                ev = torch.cuda.Event()
                ev.record(st)
                cur.wait_event(ev)
            e.record(cur)
            torch.cuda.synchronize()
            best = max(best, nb * reps / (s.elapsed_time(e) * 1e-3) / 1e9)
        out[name] = round(best, 1)
    del h_in, h_out, d_in, d_out
    return out


def time_calls(torch, fn, warm=3, iters=10, reps=3):
    """ms per call: the median over `reps` timed loops of `iters` calls (CUDA
    events), after `warm` untimed calls; one disturbed loop cannot move it."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    per_call = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(iters):
            fn()
        e.record()
        torch.cuda.synchronize()
        per_call.append(s.elapsed_time(e) / iters)
    return statistics.median(per_call)


def run_extra(peaks):
    """Short measurements of the other workloads (the headline is the long one)."""
    import torch

    import synth
    from exact_attention_94_gb300 import _lib, accounting as acc, ops

    out = {}
    # fp8 first, before seconds of load bring the power cap in (the e4m3 products draw the
    # most power): the long workload's shape on e4m3 operands (quantise Q, K with the
    # Hadamard rotation and V transposed, then attend), causal
    w = synth.WORKLOADS["long"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=w.seed, k_boost=w.k_boost, device="cuda", with_do=False)
    signs = synth.hadamard_signs(w.d, 0).cuda()
    F = acc.fwd_flops(w.B, w.H, w.N, w.d, True)
    qc, qs = ops.fp8_quantize(x["q"], signs)
    kc, ks = ops.fp8_quantize(x["k"], signs)
    vc, vs = ops.fp8_quantize(x["v"], None, transpose=True)
    t_att = time_calls(torch, lambda: ops.fwd_fp8_codes(qc, kc, vc, qs, ks, vs, causal=True), warm=3, iters=20)
    t_all = time_calls(torch, lambda: ops.fwd_fp8(x["q"], x["k"], x["v"], signs, causal=True), warm=3, iters=20)
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # measured bf16 burst x the nominal e4m3 / bf16 ratio of 2
    out["fp8"] = {"attn_ms": round(t_att, 4), "attn_tflops": round(F / t_att / 1e9, 1),
                  "attn_frac_of_fp8_peak": round(F / t_att / 1e9 / fp8_peak, 4),
                  "with_quantize_ms": round(t_all, 4), "with_quantize_tflops": round(F / t_all / 1e9, 1),
                  "fp8_peak_tflops": fp8_peak, "peak_source": "measured bf16 burst x 2 (nominal ratio)"}
    del x, qc, kc, vc
    torch.cuda.empty_cache()
    # mid: B16 H16 N2048 d64 non-causal
    w = synth.WORKLOADS["mid"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=0, device="cuda")
    F = acc.fwd_flops(w.B, w.H, w.N, w.d, False)
    o, lse = ops.fwd(x["q"], x["k"], x["v"])
    t_f = time_calls(torch, lambda: ops.fwd(x["q"], x["k"], x["v"], out=o, lse=lse))
    r = {"fwd_ms": round(t_f, 4), "fwd_tflops": round(F / t_f / 1e9, 1)}
    try:
        t_b = time_calls(torch, lambda: ops.bwd(x["q"], x["k"], x["v"], o, lse, x["do"]))
        r.update(bwd_ms=round(t_b, 4), fwdbwd_tflops=round(2.5 * F / (t_f + t_b) / 1e9, 1))
    except _lib.FaError:
        pass
    out["mid"] = r
    del x, o, lse
    # varlen: 32 seeded lengths in [128, 4096], H32 d128 causal
    w = synth.WORKLOADS["varlen"]
    lengths = synth.varlen_lengths(w.B, w.len_lo, w.len_hi, w.seed)
    x = synth.make_varlen(lengths, w.H, w.d, seed=0, device="cuda")
    cu = x["cu_seqlens"].cuda()
    F = acc.varlen_fwd_flops(lengths.tolist(), w.H, w.d, True)
    mx = int(lengths.max())
    o, lse = ops.fwd_varlen(x["q"], x["k"], x["v"], cu, mx, causal=True)
    t_f = time_calls(torch, lambda: ops.fwd_varlen(x["q"], x["k"], x["v"], cu, mx, causal=True))
    r = {"tokens": int(lengths.sum()), "fwd_ms": round(t_f, 4), "fwd_tflops": round(F / t_f / 1e9, 1)}
    try:
        t_b = time_calls(torch, lambda: ops.bwd_varlen(x["q"], x["k"], x["v"], o, lse, x["do"], cu, mx, causal=True))
        r.update(bwd_ms=round(t_b, 4), fwdbwd_tflops=round(2.5 * F / (t_f + t_b) / 1e9, 1))
    except _lib.FaError:
        pass
    out["varlen"] = r
    del x, o, lse
    # window: B1 H32 N16384 d128, causal sliding window of 4096 keys (fwd and bwd)
    w = synth.WORKLOADS["window"]
    x = synth.make_dense(w.B, w.H, w.N, w.d, seed=0, device="cuda")
    F = acc.masked_fwd_flops(w.B, w.H, w.N, w.N, w.d, *w.window)
    o, lse = ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window)
    t_f = time_calls(torch, lambda: ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window))
    t_b = time_calls(torch, lambda: ops.bwd_masked(x["q"], x["k"], x["v"], o, lse, x["do"], window=w.window))
    out["window"] = {"window": list(w.window), "fwd_ms": round(t_f, 4), "fwd_tflops": round(F / t_f / 1e9, 1),
                     "bwd_ms": round(t_b, 4), "fwdbwd_tflops": round(2.5 * F / (t_f + t_b) / 1e9, 1),
                     "flops": "visible scores only, 4d per score"}
    del x, o, lse
    # prefill: 8 chunks of 2048 queries against 16384-key caches, GQA 32:8, bottom-right causal
    w = synth.WORKLOADS["prefill"]
    x = synth.make_masked(w.B, w.N, w.n_k, w.H, w.h_kv, w.d, seed=0, device="cuda", with_do=False)
    F = acc.masked_fwd_flops(w.B, w.H, w.N, w.n_k, w.d, *w.window)
    ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window)
    t_f = time_calls(torch, lambda: ops.fwd_masked(x["q"], x["k"], x["v"], window=w.window))
    out["prefill"] = {"fwd_ms": round(t_f, 4), "fwd_tflops": round(F / t_f / 1e9, 1),
                      "flops": "visible scores only, 4d per score"}
    del x
    torch.cuda.empty_cache()
    # decode: B64 L32768 H32 d128 (34.4 GB of K/V, far larger than L2)
    w = synth.WORKLOADS["decode"]
    try:
        x = synth.make_decode(w.B, w.H, w.N, w.d, seed=0, device="cuda")
        ops.decode(x["q"], x["k"], x["v"])
        t = time_calls(torch, lambda: ops.decode(x["q"], x["k"], x["v"]), warm=2, iters=5)
        byts = acc.decode_bytes(w.B, w.H, w.N, w.d)
        out["decode"] = {"ms": round(t, 4), "GB/s": round(byts / t / 1e6, 1),
                         "frac_of_hbm": round(byts / t / 1e6 / peaks["hbm_gbs"], 4)}
        del x
        torch.cuda.empty_cache()
        # the same decode over a paged cache: 16-token pages in shuffled order
        xp = synth.make_paged_decode([w.N] * w.B, w.H, w.d, page_size=16, seed=0, device="cuda")
        bt, sl = xp["block_table"].cuda(), xp["seq_lens"].cuda()
        f = lambda: ops.decode_paged(xp["q"], xp["k_pages"], xp["v_pages"], bt, sl, w.N)
        t = time_calls(torch, f, warm=2, iters=5)
        out["decode_paged"] = {"ms": round(t, 4), "GB/s": round(byts / t / 1e6, 1),
                               "frac_of_hbm": round(byts / t / 1e6 / peaks["hbm_gbs"], 4), "page_size": 16}
        del xp
    except _lib.FaError:
        pass
    torch.cuda.empty_cache()
    return out


def cpu_sample(heads):
    """Float64 oracle forward+backward on a few (b, h) heads of the long
    workload; returns (TFLOP/s under the metric's convention, seconds)."""
    import numpy as np

    import oracle
    import synth
    from exact_attention_94_gb300 import accounting as acc

    w = LONG
    if "x" not in _CPU_INPUTS:  # generated once, outside every timed region
        _CPU_INPUTS["x"] = synth.make_dense(w["B"], w["H"], w["N"], w["d"], seed=0, k_boost=w["k_boost"])
    x = _CPU_INPUTS["x"]
    scale = 1.0 / math.sqrt(w["d"])
    per_head = [tuple(synth.to_f64(x[n][b, :, h]) for n in ("q", "k", "v", "do")) for b, h in heads]
    t0 = time.perf_counter()
    for qh, kh, vh, dh in per_head:
        oracle.head_forward(qh, kh, vh, scale, True)
        oracle.head_backward(qh, kh, vh, dh, scale, True)
    sec = time.perf_counter() - t0
    flops = 2.5 * acc.fwd_flops(1, 1, w["N"], w["d"], True) * len(heads)
    return flops / sec / 1e12, sec


CPU_HEADS = [(0, 0), (0, 8), (1, 3)]
_CPU_INPUTS = {}


def run_reference(args):
    """The float64 CPU oracle timed on the host cores: each step is forward +
    backward of one (b, h) head of the long workload (rotating over the 32
    heads), reported in the same unit as the GPU arm."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import synth  # noqa: F401  (inputs are generated inside cpu_sample)

    heads = [(b, h) for b in range(LONG["B"]) for h in range(LONG["H"])]
    for i in range(max(1, args.warmup)):
        cpu_sample([heads[i % len(heads)]])
    t0 = time.perf_counter()
    tfs = []
    for i in range(args.steps):
        tf, _ = cpu_sample([heads[(args.warmup + i) % len(heads)]])
        tfs.append(tf)
    sec = time.perf_counter() - t0
    value = len(tfs) / sum(1.0 / t for t in tfs)  # total work / total time
    sample = f"one (b, h) head per step of the long workload, forward + backward in float64 ({args.steps} steps)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sec / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long: B=2 H=16 N=8192 d=128 causal, K x3 in heads 0-7",
                   "flops_convention": "fwd 4BHN^2d/2; fwd+bwd 2.5x fwd", "sample": sample},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": N_CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.case is not None:
        sys.exit(run_case(args))
    rank, world, _ = dist_env()
    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    import torch
    import torch.distributed as dist

    from exact_attention_94_gb300 import replicas

    res, ctx = run_ours(args)
    e2e = run_e2e(args, ctx)
    if world > 1:
        (slowest,) = replicas.max_over_ranks([e2e["ms_per_step"]], device="cuda")
        e2e["value"] = round(replicas.rescale_to_slowest(float(e2e["value"]), e2e["ms_per_step"], slowest, world), 2)
        e2e["ms_per_step"] = round(slowest, 4)
    res["e2e"] = e2e
    del ctx
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_extra:
        # clocks over the whole phase: each extra measurement lasts milliseconds, below
        # the sampler's 100 ms period
        with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as xclocks:
            res["extra"] = run_extra(load_peaks())
        res["extra_clocks"] = xclocks.summary()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, sec = cpu_sample(CPU_HEADS)
        res["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": N_CORES, "kind": "oracle",
                               "sample": f"{len(CPU_HEADS)} of 32 (b, h) heads of the long workload, forward + "
                                         f"backward in float64, {sec:.1f} s"}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
