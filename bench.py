#!/usr/bin/env python
"""Benchmark of the chunkwise gated delta rule forward pass (libgdn).

One step = one gdn_chunk_fwd over the training-shape workload
(B4 H16 T4096 d_k=d_v=128, C64, bf16 q/k/v/o, fp32 gates and final state),
inputs resident in HBM.  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only other implementation
of the method; there is no third-party one) on a bounded sample of the same
workload on the host cores.  Under torchrun each rank runs its own replica of
the workload (the method's (sequence, head) units are independent, so there is
no collective on the data path); ``value`` is the tokens of all ranks over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN chunk-fwd tokens/s and % bf16 tensor peak (B4 H16 T4096 d128)"
WORKLOAD = "train_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 126 * 2 ** 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_numbers(w, lengths):
    """Algorithmic FLOPs and bytes of one forward pass.

    FLOPs: per chunk of n tokens and head, 2 [3 n d_k d_v + n^2 (3 d_k + 2 d_v)]
    (K K^T, W, U, W S^T, Q S^T, Q K^T, P V_new, state update; C x C operands
    counted dense).  Bytes: q, k, v read and o written once, 8 B of gates per
    token-head, S0 read if given and S_final written, fp32.
    """
    esz = 2 if w.dtype == "bf16" else 4
    flops = 0
    for L in lengths:
        full, tail = divmod(L, w.C)
        for n in [w.C] * full + ([tail] if tail else []):
            flops += 2 * (3 * n * w.dk * w.dv + n * n * (3 * w.dk + 2 * w.dv)) * w.H
    tok_heads = sum(lengths) * w.H
    nseq = len(lengths)
    state = nseq * w.H * w.dv * w.dk * 4
    byts = tok_heads * (2 * w.dk + 2 * w.dv) * esz + tok_heads * 8 + state
    if w.s0 != "none":
        byts += state
    return flops, byts


# Source files whose code each recorded traffic figure was measured on.
KERNEL_SOURCES = {"train_bf16": ("gdn_tc.cu", "gdn_ut.cuh", "gdn_internal.h", "sm100_ptx.cuh"),
                  "decode_bf16": ("gdn_decode.cu", "gdn_internal.h")}


def triangular_flops(w, lengths):
    """The canonical count with each C x C operand counted as its lower
    triangle (n (n + 1) / 2 entries instead of n^2)."""
    flops = 0
    for L in lengths:
        full, tail = divmod(L, w.C)
        for n in [w.C] * full + ([tail] if tail else []):
            flops += 2 * (3 * n * w.dk * w.dv + (n * (n + 1) // 2) * (3 * w.dk + 2 * w.dv)) * w.H
    return flops


def kernel_source_sha(workload="train_bf16"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_09_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES.get(workload, ())):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's sources as they are now (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = kernel_source_sha(workload)
    for line in text.splitlines():
        m = re.match(r"\s*(\w+)\s+sha=(\w+)\s+dram_bytes_per_launch=(\d+)", line)
        if m and m.group(1) == workload and m.group(2) == sha:
            return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = tempfile.TemporaryFile(mode="w+")
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=timestamp," + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return []
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.seek(0)
        rows = []
        for line in self.f.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]),
                                 active=parts[5], hw=parts[6], hwt=parts[7], swt=parts[8],
                                 pcap=parts[9]))
            except (ValueError, IndexError):
                continue
        return rows

    @staticmethod
    def summarise(rows, t_start, t_end):
        win = [r for r in rows if t_start - 0.1 <= r["ts"] <= t_end + 0.1]
        if not win and rows:  # very short timed region: nearest samples
            win = sorted(rows, key=lambda r: abs(r["ts"] - (t_start + t_end) / 2))[:3]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for r in win:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in win),
                "sm_max_mhz": max(r["smax"] for r in win),
                "reasons": sorted(reasons), "samples": len(win)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_baseline(w, x, sample_tokens, min_seconds=0.0):
    """Oracle on the first ``sample_tokens`` tokens of every sequence x all heads,
    repeated until ``min_seconds`` of wall time have passed (at least once)."""
    from oracle import gdn_recurrence_f64
    sl = (slice(None), slice(0, sample_tokens))
    cores = os.cpu_count() or 1
    args = [x[k][sl] for k in ("q", "k", "v", "log_alpha", "beta")]
    reps, t0 = 0, time.perf_counter()
    while True:
        gdn_recurrence_f64(*args, n_threads=cores)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    tokens = reps * w.B * sample_tokens
    # one thread on one (sequence, head) of the same sample, for the per-core rate
    one = [t[:1, :, :1] for t in args]
    t1 = time.perf_counter()
    gdn_recurrence_f64(*one, n_threads=1)
    dt1 = time.perf_counter() - t1
    return dict(value=tokens / dt, unit="tokens/s", cores=min(cores, w.B * w.H), kind="oracle",
                sample="%d x (%d sequences x %d heads x first %d of %d tokens) of %s, fp64, "
                       "%.2f s" % (reps, w.B, w.H, sample_tokens, w.T, w.name, dt),
                one_thread={"value": sample_tokens / dt1, "unit": "token-heads/s",
                            "sample": "1 sequence x 1 head x %d tokens, %.3f s"
                                      % (sample_tokens, dt1)})


def run_reference(args, world, rank):
    from gated_delta_rule_09_gb300 import inputs as I
    if rank != 0:
        return
    w = I.WORKLOADS[args.workload]
    x = I.generate(w, seed=0)
    sample = args.ref_tokens
    for _ in range(args.warmup):
        cb = cpu_baseline(w, x, sample)
    times = []
    for _ in range(args.steps):
        cb = cpu_baseline(w, x, sample)
        times.append(w.B * sample / cb["value"])
    total = sum(times)
    value = args.steps * w.B * sample / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "%s: B%d H%d T%d d_k=%d d_v=%d C%d, each step the oracle "
                                   "on the first %d tokens of each sequence, all heads"
                                   % (w.name, w.B, w.H, w.T, w.dk, w.dv, w.C, sample)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cb["cores"],
                             "kind": "oracle", "sample": cb["sample"],
                             "one_thread": cb["one_thread"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch
    import gated_delta_rule_09_gb300 as gdn
    from gated_delta_rule_09_gb300 import inputs as I

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = I.WORKLOADS[args.workload]
    x = I.generate(w, seed=rank)
    lengths = x["lengths"]
    flops, byts = workload_numbers(w, lengths)
    tokens = sum(lengths)
    keys = ("q", "k", "v", "log_alpha", "beta")
    # two resident copies, used alternately, so no step finds its inputs in L2
    sets = []
    for _ in range(2):
        d = {kk: x[kk].to(dev) for kk in keys}
        d["S0"] = None if x["S0"] is None else x["S0"].to(dev)
        d["cu"] = None if x["cu_seqlens"] is None else x["cu_seqlens"].to(dev)
        d["o"] = torch.empty(x["v"].shape, dtype=x["v"].dtype, device=dev)
        d["Sf"] = torch.empty((x["N"], w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
        sets.append(d)
    stream = torch.cuda.Stream(dev)

    def step(i):
        d = sets[i & 1]
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                          o=d["o"], S_final=d["Sf"], C=w.C, cu_seqlens=d["cu"], stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    assert gdn.gdn_get_device_status(stream) == 0
    launches_per_step, path = gdn.gdn_last_launch_count()

    sampler = ClockSampler(local)
    sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(world)
    rows = sampler.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms, world)
    clocks = ClockSampler.summarise(rows, t_start, t_end)
    # the same steps again, each between its own pair of events, for the median
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        evs[i][0].record(stream)
        step(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    per_step = sorted(e0_.elapsed_time(e1_) for e0_, e1_ in evs)
    ms_median = max_over_ranks(per_step[len(per_step) // 2], world)

    # end to end through the public call: every step copies its inputs from
    # pinned host memory, runs the forward pass and copies o and S_final back
    # to pinned host memory.  Consecutive steps are independent, so they
    # overlap as a stream of jobs would: step i + 1's inputs go in on one copy
    # stream while step i computes and step i - 1's results come out on
    # another, with the two device buffer sets used alternately.
    host = {kk: x[kk].pin_memory() for kk in keys}
    host_S0 = None if x["S0"] is None else x["S0"].pin_memory()
    host_cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].pin_memory()
    out_o = [torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory() for _ in range(2)]
    out_S = [torch.empty((x["N"], w.H, w.dv, w.dk), dtype=torch.float32).pin_memory()
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    h2d += 0 if host_S0 is None else host_S0.numel() * 4
    h2d += 0 if host_cu is None else host_cu.numel() * 4
    d2h = out_o[0].numel() * out_o[0].element_size() + out_S[0].numel() * 4
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_in):  # inputs once step i - 2 has consumed this set
            if used[b]:
                s_in.wait_event(ev_comp[b])
            for kk in keys:
                d[kk].copy_(host[kk], non_blocking=True)
            if host_S0 is not None:
                d["S0"].copy_(host_S0, non_blocking=True)
            if host_cu is not None:
                d["cu"].copy_(host_cu, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:  # this set's previous results have been copied out
            stream.wait_event(ev_out[b])
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                          o=d["o"], S_final=d["Sf"], C=w.C, cu_seqlens=d["cu"], stream=stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            out_o[b].copy_(d["o"], non_blocking=True)
            out_S[b].copy_(d["Sf"], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_event(ev_out[(e2e_steps - 1) & 1])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    # the host link alone: the same input copies, no compute and no results
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(s_in)
    for i in range(e2e_steps):
        d = sets[i & 1]
        with torch.cuda.stream(s_in):
            for kk in keys:
                d[kk].copy_(host[kk], non_blocking=True)
            if host_S0 is not None:
                d["S0"].copy_(host_S0, non_blocking=True)
            if host_cu is not None:
                d["cu"].copy_(host_cu, non_blocking=True)
    c1.record(s_in)
    torch.cuda.synchronize(dev)
    h2d_only_ms = max_over_ranks(c0.elapsed_time(c1) / e2e_steps, world)
    barrier(world)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    kernel_s = ms * 1e-3 / max(launches_per_step, 1)  # one launch per step on both paths
    gbs = byts / kernel_s / 1e9
    tflops = flops / (ms * 1e-3) / 1e12
    value = world * tokens / (ms_max * 1e-3)
    cb = (cpu_baseline(w, x, min(args.cpu_tokens, w.T or tokens), args.cpu_seconds)
          if (world == 1 and not args.no_cpu_baseline) else None)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "ms_per_step_median": ms_median,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": "%s: B%d H%d T%d d_k=%d d_v=%d C%d, %s q/k/v/o, fp32 gates "
                               "and final state, %s" % (
                                   w.name, w.B, w.H, w.T, w.dk, w.dv, w.C, w.dtype,
                                   "no S0" if x["S0"] is None else "fp32 S0 (%s)" % w.s0),
                   "tokens_per_step": tokens,
                   "l2": ("inputs larger than L2 (%.0f MB moved per step vs %.0f MB L2), two "
                          "resident input copies used alternately" if byts > L2_BYTES else
                          "inputs fit in L2 (%.0f MB moved per step vs %.0f MB L2; not flushed, "
                          "so warm-cache figures), two resident copies used alternately")
                   % (byts / 1e6, L2_BYTES / 1e6),
                   "parallelism": "replicas x%d" % world,
                   "kernel_path": "tcgen05" if path == 1 else "fp32 cuda-core"},
        "tflops": tflops,
        "pct_bf16_peak": 100.0 * tflops / peaks["bf16_tflops"],
        "pct_bf16_sustained_peak": 100.0 * tflops / peaks.get("bf16_tflops_sustained",
                                                                peaks["bf16_tflops"]),
        "tflops_triangular": triangular_flops(w, lengths) / (ms * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": recorded_traffic(w.name),
                     "algorithmic_bytes": byts, "peak_source": peak_src,
                     "tensor": {"achieved": tflops, "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                                "algorithmic_flops": flops}},
        "clocks": clocks,
        "e2e": {"value": world * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "h2d_only_ms_per_step": h2d_only_ms,
                "overlap": "consecutive steps: inputs in, compute, results out on three streams"},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cb,
    }
    print(json.dumps(line), flush=True)


DECODE_METRIC = "GDN decode-step tokens/s and % of HBM bandwidth (N256 H16 d128, fp32 state in place)"


def decode_numbers(N, H, T, dk, dv, esz):
    """Algorithmic bytes and FLOPs of one decode call: the fp32 state read and
    written once, q, k, v read and o written once, 8 B of gates per
    token-head; per token-head 2 d_k d_v FLOP for each of r = S k, the rank-1
    update and o = S q, plus d_k d_v for the decay."""
    byts = 2 * N * H * dv * dk * 4 + N * T * H * ((2 * dk + 2 * dv) * esz + 8)
    flops = N * T * H * 7 * dk * dv
    return flops, byts


def run_decode(args, world, rank, local):
    import torch
    import gated_delta_rule_09_gb300 as gdn
    from gated_delta_rule_09_gb300 import inputs as I

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = I.decode_inputs(seed=rank)
    N, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    esz = x["q"].element_size()
    flops, byts = decode_numbers(N, H, T, dk, dv, esz)
    keys = ("q", "k", "v", "log_alpha", "beta")
    d = {kk: x[kk].to(dev) for kk in keys}
    S = x["S0"].to(dev)                     # the cache, updated in place every step
    o = torch.empty(x["v"].shape, dtype=x["v"].dtype, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S_in=S, o=o,
                            S_out=S, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize(dev)
    assert gdn.gdn_get_device_status(stream) == 0
    launches_per_step, path = gdn.gdn_last_launch_count()

    sampler = ClockSampler(local)
    sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(world)
    rows = sampler.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms, world)
    clocks = ClockSampler.summarise(rows, t_start, t_end)

    # end to end: the step's token inputs from pinned host memory, the call,
    # its outputs back to pinned host memory; the state is the device-resident
    # cache and does not move.  The steps are ordered by the state, but step
    # i + 1's inputs go in while step i runs and step i's outputs come out
    # while step i + 1 runs (two device buffer sets, three streams).
    host = {kk: x[kk].pin_memory() for kk in keys}
    out_o = [torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_o[0].numel() * out_o[0].element_size()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    dsets = [d, {kk: torch.empty_like(d[kk]) for kk in keys}]
    osets = [o, torch.empty_like(o)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        db, ob = dsets[b], osets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_comp[b])
            for kk in keys:
                db[kk].copy_(host[kk], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])
        gdn.gdn_decode_step(db["q"], db["k"], db["v"], db["log_alpha"], db["beta"], S_in=S,
                            o=ob, S_out=S, stream=stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            out_o[b].copy_(ob, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_event(ev_out[(e2e_steps - 1) & 1])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    barrier(world)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    gbs = byts / (ms * 1e-3) / 1e9
    tokens = N * T
    cb = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle import gdn_recurrence_f64
        cores = os.cpu_count() or 1
        reps, t0 = 0, time.perf_counter()
        while True:
            gdn_recurrence_f64(*[x[kk] for kk in keys], S0=x["S0"], n_threads=cores)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= args.cpu_seconds:
                break
        cb = {"value": reps * tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
              "sample": "%d x the whole decode batch (%d sequences x %d heads x %d token), "
                        "fp64, %.2f s" % (reps, N, H, T, dt)}
    line = {
        "metric": DECODE_METRIC, "value": world * tokens / (ms_max * 1e-3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "decode_bf16: N%d H%d T%d d_k=%d d_v=%d, bf16 q/k/v/o, fp32 "
                               "state updated in place" % (N, H, T, dk, dv),
                   "tokens_per_step": tokens,
                   "l2": "inputs larger than L2 (%.0f MB of state read and written per step "
                         "vs %.0f MB L2)" % (byts / 1e6, L2_BYTES / 1e6),
                   "parallelism": "replicas x%d" % world, "kernel_path": "recurrent decode"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": recorded_traffic("decode_bf16"),
                     "algorithmic_bytes": byts, "peak_source": peak_src,
                     "algorithmic_flops": flops},
        "clocks": clocks,
        "e2e": {"value": world * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "overlap": "next inputs in and previous outputs out while a step runs (the state stays in place)"},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cb,
    }
    print(json.dumps(line), flush=True)


SCAN_METRIC = "GDN chunk-fwd tokens/s on one long sequence (B1 H8 T131072 d128), chunk-level scan"


def run_scan(args, world, rank, local):
    """The chunk-level scan on few long sequences, against the plain pass on
    the same inputs (one unit per (sequence, head) leaves most SMs idle)."""
    import torch
    import gated_delta_rule_09_gb300 as gdn
    from gated_delta_rule_09_gb300 import inputs as I

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, H, T, dk, dv = 1, 8, args.scan_tokens, 128, 128
    x = I.custom(B, H, T, dk, dv, 64, dtype="bf16", seed=rank)
    keys = ("q", "k", "v", "log_alpha", "beta")
    d = {kk: x[kk].to(dev) for kk in keys}
    o = torch.empty(x["v"].shape, dtype=x["v"].dtype, device=dev)
    Sf = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    need = gdn.gdn_chunk_fwd_scan_workspace_size(B, H, T, dk, dv, 64, 0)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    flops, byts = workload_numbers(I.Workload("long", B, H, T, dk, dv, 64, "bf16", True,
                                              "sigmoid_normal", "softplus_0.1", "none"), [T] * B)

    def scan_step():
        gdn.gdn_chunk_fwd_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], o=o,
                               S_final=Sf, segments=0, workspace=ws, stream=stream)

    def plain_step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], o=o, S_final=Sf,
                          stream=stream)

    def timed(fn, steps):
        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    plain_ms = timed(plain_step, max(1, args.steps // 10))
    sampler = ClockSampler(local)
    sampler.start()
    t_start = time.time()
    ms = timed(scan_step, args.steps)
    t_end = time.time()
    rows = sampler.stop()
    assert gdn.gdn_get_device_status(stream) == 0
    launches, path = gdn.gdn_last_launch_count()
    ms_max = max_over_ranks(ms, world)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    gbs = byts / (ms * 1e-3) / 1e9
    line = {
        "metric": SCAN_METRIC.replace("T131072", "T%d" % T), "value": world * B * T / (ms_max * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "long_bf16: B%d H%d T%d d_k=%d d_v=%d C64, bf16, no S0" % (B, H, T, dk, dv),
                   "segments_workspace_bytes": need, "plain_pass_ms": plain_ms,
                   "speedup_vs_plain": plain_ms / ms,
                   "l2": "inputs larger than L2 (%.0f MB moved per step vs %.0f MB L2)"
                         % (byts / 1e6, L2_BYTES / 1e6),
                   "parallelism": "replicas x%d" % world, "kernel_path": "chunk-level scan"},
        "tflops": flops / (ms * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes": byts,
                     "peak_source": peak_src},
        "clocks": ClockSampler.summarise(rows, t_start, t_end),
        "gpu_launches": launches * args.steps,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


INV_METRIC = "UT inverse (I + A)^{-1}, 64 x 64 matrices/s, doubling product on the tensor cores"


def run_inverse(args, world, rank, local):
    """The batched UT inverse by both methods on the same matrices: the
    doubling product on the tensor cores (the line's value) and the blocked
    forward substitution on CUDA cores, with their errors against fp64."""
    import numpy as np
    import torch
    import gated_delta_rule_09_gb300 as gdn
    from gated_delta_rule_09_gb300 import inputs as I

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    count, C = 16384, 64
    A = I.ut_matrices(count, C, 0.04, seed=rank)
    Ad = A.to(dev)
    T = torch.empty_like(Ad)
    stream = torch.cuda.Stream(dev)

    def timed(method, steps):
        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                gdn.gdn_ut_inverse(Ad, T, method=method, stream=stream)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        for _ in range(steps):
            gdn.gdn_ut_inverse(Ad, T, method=method, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    def error(method):
        from oracle.chunk_reference import forward_substitution
        gdn.gdn_ut_inverse(Ad, T, method=method, stream=stream)
        torch.cuda.synchronize(dev)
        Tc = T[:64].double().cpu().numpy()
        An = A[:64].double().numpy()
        worst = 0.0
        for n in range(64):
            ref = forward_substitution(-An[n])
            worst = max(worst, float(np.abs(Tc[n] - ref).max() / np.abs(ref).max()))
        return worst

    fs_ms = timed(0, args.steps)
    sampler = ClockSampler(local)
    sampler.start()
    t_start = time.time()
    tc_ms = timed(1, args.steps)
    t_end = time.time()
    rows = sampler.stop()
    assert gdn.gdn_get_device_status(stream) == 0
    ms_max = max_over_ranks(tc_ms, world)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    byts = 2 * count * C * C * 4
    flops = count * 9 * 2 * C ** 3  # nine 64 x 64 x 64 products
    line = {
        "metric": INV_METRIC, "value": world * count / (ms_max * 1e-3), "unit": "matrices/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32",
        "data": "synthetic",
        "config": {"workload": "ut_inverse: %d strictly lower 64 x 64 fp32 matrices, entries "
                               "N(0, 0.04^2)" % count,
                   "forward_substitution_ms": fs_ms,
                   "forward_substitution_matrices_per_s": count / (fs_ms * 1e-3),
                   "max_rel_error_tensor": error(1), "max_rel_error_forward_substitution": error(0),
                   "l2": "inputs larger than L2 (%.0f MB read and written per call)" % (byts / 1e6),
                   "parallelism": "replicas x%d" % world},
        "roofline": {"bound": "hbm", "achieved": byts / (tc_ms * 1e-3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": byts / (tc_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes": byts, "peak_source": peak_src,
                     "tensor_tflops": flops / (tc_ms * 1e-3) / 1e12},
        "clocks": ClockSampler.summarise(rows, t_start, t_end),
        "gpu_launches": args.steps,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["chunk", "decode", "scan", "inverse"], default="chunk",
                    help="chunk: the chunkwise forward (default); decode: the recurrent "
                         "decode step on the decode batch; scan: the chunk-level scan on "
                         "one long sequence, beside the plain pass; inverse: the batched UT "
                         "inverse by both methods")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--scan-tokens", type=int, default=131072,
                    help="--op scan: tokens of the one long sequence (smaller for profiling)")
    ap.add_argument("--ref-tokens", type=int, default=256,
                    help="tokens of each sequence per oracle step (all sequences, all heads)")
    ap.add_argument("--cpu-tokens", type=int, default=4096,
                    help="tokens of each sequence in the oracle sample for the cpu_baseline key")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="the cpu_baseline sample repeats until this much wall time has passed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.op == "decode":
        run_decode(args, world, rank, local)
    elif args.op == "scan":
        run_scan(args, world, rank, local)
    elif args.op == "inverse":
        run_inverse(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
