#!/usr/bin/env python3
"""Benchmark of the per-layer mixed-precision AdamW step on GB300.

Workload of the headline (default): one h=5120 decoder layer (330,311,680
parameters), R = 8 BF16 gradient replicas averaged in the kernel, per-tensor
gradient scales drawn log-uniform in [1e-5, 1e-2], lr 1e-5, betas
0.9/0.999, eps 1e-8, weight decay 0.01.  This is the largest HBM-resident
workload.  A step is one slide_layer_step: the fused grad_reduce_adamw_cast
kernel (plus the clip pre-pass when the workload clips) over one batch of R
synthetic replicas (pre-generated batches are cycled; every step touches
13.9 GB, far more than the 129 MB L2).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Output: detail lines (one per leg, prefixed "detail ") and, LAST, one compact
JSON line (under 4 KB) with the headline, the roofline, the baselines, the
end-to-end figure and a short summary of every other leg.  --detail-out PATH
also writes the whole record as one JSON file.  Under torchrun each rank
updates its own layer (independent problems, no collective on the data path:
weak scaling); the value is all ranks' parameters over the slowest rank's
time.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LayerAdam Gparam/s & HBM GB/s vs ~8 TB/s; host-streamed s/step vs link BW"
UNIT = "Gparam/s"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="h5120_R8_logscale",
                    choices=["h2560_R1", "h2560_R4_clip", "h5120_R8_logscale"],
                    help="HBM-resident workload of the headline")
    ap.add_argument("--detail-out", default="",
                    help="also write the whole record (every leg in full) to this JSON file")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the FP32-gradient variant, the other HBM workloads and the CPU-route legs")
    ap.add_argument("--no-streamed", action="store_true",
                    help="skip the host-streamed legs (8-layer h=8192 model, ~98 GB pinned host memory; "
                         "40-layer h=5120 model, ~177 GB pinned)")
    ap.add_argument("--streamed-workload", default="h8192x8_streamed",
                    choices=["h8192x8_streamed", "h5120x40_streamed"],
                    help="host-streamed workload of the 'streamed' key")
    ap.add_argument("--streamed-also", default="h5120x40_streamed,h8192x8_streamed+bf16hbm",
                    help="comma-separated further host-streamed workloads, each under 'streamed_also' "
                         "('' for none); a '+bf16hbm' suffix keeps the BF16 copy in HBM")
    ap.add_argument("--streamed-steps", type=int, default=5)
    ap.add_argument("--streamed-bf16-in-hbm", action="store_true",
                    help="keep the BF16 copy in HBM (host holds 12 B/param); implied for h5120x40_streamed")
    ap.add_argument("--pinned-guard-gib", type=int, default=8,
                    help="pin this many GiB first and hold them for the run (0: none); see PinnedArena")
    ap.add_argument("--streamed-arena", choices=["hostalloc", "hugepages"], default="hostalloc",
                    help="pinned host arena of the streamed legs: cudaHostAlloc, or an anonymous mapping "
                         "advised for transparent huge pages and registered with cudaHostRegister")
    ap.add_argument("--streamed-chunk-mib", type=int, default=256,
                    help="host->device copy chunk of the streamed engine (the library's default, 256 MiB, "
                         "from the chunk sweep; the pages use 64 MiB)")
    ap.add_argument("--streamed-chunk-d2h-mib", type=int, default=0,
                    help="device->host write-back chunk of the streamed engine (0: as the copy-in chunk)")
    ap.add_argument("--chunk-sweep", default="32:32,64:64,128:128,256:256,512:512,64:256,256:64,128:512",
                    help="copy-in:write-back chunk sizes (MiB) swept on each --chunk-sweep-workloads "
                         "workload ('' for none)")
    ap.add_argument("--chunk-sweep-workloads", default="h8192x8_streamed,h5120x40_streamed",
                    help="streamed workloads of the chunk sweep (each must fit the run's pinned arena)")
    ap.add_argument("--batches", type=int, default=4,
                    help="pre-generated gradient batches cycled by the steps (1 for small profiling runs)")
    ap.add_argument("--slice-params", type=int, default=0,
                    help="profiling only: cut the main workload's unit to its first N parameters (the line "
                         "then carries config.slice_params and is not a full-size measurement)")
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="seconds of untimed steps before the timed region (clocks settle, samples)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


# ---------------------------------------------------------------- env ----

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            out = self.parse(f.readlines())
        os.unlink(self.path)
        return out

    @staticmethod
    def parse(lines):
        """Median SM clock, max clock and the throttle reasons seen in the
        nvidia-smi CSV lines (fields as in FIELDS, no header, no units)."""
        sms, maxs, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxs) if maxs else None,
                "reasons": sorted(reasons), "samples": n}


def max_over_ranks(x: float, dist=None) -> float:
    """The largest value of x over all ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload(name):
    from synth import workloads as W
    return W.ALL[name]()


def slice_unit(unit, n):
    """The first n parameters of a unit: its tensors in order, the last one cut."""
    from synth import workloads as W
    tensors, left = [], n
    for name, k in unit.tensors:
        if left <= 0:
            break
        tensors.append((name, min(k, left)))
        left -= k
    return W.Unit(unit.name, tensors)


# ------------------------------------------------------------ oracle ----

def oracle_sample_rate(w, n_sample, steps_budget_s, max_steps, seed_offset=0, openmp=False):
    """Time the oracle (single thread, as it stands; openmp=True: the same
    source built with -fopenmp, on all host cores) on a contiguous slice of
    the workload's unit treated as a layer of its own (the clip, when on,
    is over the slice).  Inputs are generated before each timed call."""
    import numpy as np
    import oracle
    import synth

    sp = synth.spec(w.seed, w.grad_kind, w.zero_prob)
    hp = oracle.hparams(*w.hparams_tuple())
    th = synth.master(n_sample, w.seed)
    m, v = np.zeros(n_sample, np.float32), np.zeros(n_sample, np.float32)
    wb = np.zeros(n_sample, np.uint16)
    scale = w.tensor_scales(0)[0]
    batches = [[synth.grad(n_sample, sp, 0, b + 1 + seed_offset, r, scale) for r in range(w.R)]
               for b in range(2)]
    elapsed, steps = 0.0, 0
    # a time budget > 0 stops early once spent (at least 2 steps); 0 runs max_steps
    while steps < max_steps and (steps_budget_s <= 0 or elapsed < steps_budget_s or steps < 2):
        g = batches[steps % 2]
        t0 = time.perf_counter()
        oracle.layer_step(g, th, m, v, wb, hp, steps + 1, openmp=openmp)
        elapsed += time.perf_counter() - t0
        steps += 1
    return n_sample * steps / elapsed / 1e9, steps, elapsed


def cpu_model():
    """The host CPU's model name (lscpu; /proc/cpuinfo on x86)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = workload(args.workload)
    # calibrate, then size each step's sample so the whole run takes ~2 minutes
    rate, _, _ = oracle_sample_rate(w, 1 << 20, 0.5, 3, seed_offset=1000)
    per_step_s = 120.0 / (args.steps + args.warmup)
    n_s = int(rate * 1e9 * per_step_s) // 4096 * 4096
    n_s = max(4096, min(n_s, w.units[0].numel, 1 << 24))
    oracle_sample_rate(w, n_s, 0.0, args.warmup, seed_offset=2000)  # untimed warm-up
    value, steps, elapsed = oracle_sample_rate(w, n_s, 0.0, args.steps)
    sample = (f"first {n_s} parameters of the {w.name} unit treated as a layer of their own "
              f"(R={w.R}{', clip over the sample' if w.max_grad_norm > 0 else ''}), "
              f"{steps} steps; inputs generated outside the timed calls")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "params_per_step": n_s},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------- FP32-gradient variant ----

def measure_hbm_workload(args, S, torch, synth, peak, w, max_steps=500):
    """One HBM-resident workload timed like the main line: per-launch events
    on the launching stream, back-to-back steps over two pre-generated
    gradient batches, inputs larger than L2."""
    n, R = w.units[0].numel, w.R
    clip = w.max_grad_norm > 0
    gsize = 4 if w.fp32_grads else 2
    hp = S.hparams(*w.hparams_tuple())
    stream = torch.cuda.Stream()
    st = S.slide_state_create([n], R, flags=S.SLIDE_FLAG_FP32_GRADS if w.fp32_grads else 0)
    try:
        synth.dev_master(S.slide_layer_ptrs(st, 0)[0], n, w.seed, stream=stream.cuda_stream)
        sp = synth.spec(w.seed, w.grad_kind, w.zero_prob)
        fill = synth.dev_grad_f32 if w.fp32_grads else synth.dev_grad
        batches = []
        for b in range(2):
            reps = [torch.empty(n + 64, dtype=torch.float32 if w.fp32_grads else torch.int16, device="cuda")
                    for _ in range(R)]
            for r, t in enumerate(reps):
                for (off, ln), sc in zip(w.units[0].segments(), w.tensor_scales(0)):
                    fill(t.data_ptr() + gsize * off, ln, sp, 0, b + 1, r, sc, offset=off, stream=stream.cuda_stream)
            batches.append(reps)
        torch.cuda.synchronize()
        for i in range(max(3, args.warmup)):
            S.slide_layer_step(st, 0, batches[i % 2], hp, stream)
        K = min(args.steps, max_steps)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for trio in ev:
            for e in trio:
                e.record(stream)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(K):
            S.slide_trace_events(st, ev[k][0], ev[k][1], ev[k][2])
            S.slide_layer_step(st, 0, batches[k % 2], hp, stream)
        stop.record(stream)
        torch.cuda.synchronize()
        S.slide_trace_events(st)
        ms = start.elapsed_time(stop)
        upd = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        pre = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        # The steps above carry trace events (with the clip, between pre-pass
        # and update, which serialises them); the step as a caller runs it (with
        # the clip, the update launched behind the pre-pass, overlapping its
        # end) is timed here.
        ms_traced = ms
        start.record(stream)
        for k in range(K):
            S.slide_layer_step(st, 0, batches[k % 2], hp, stream)
        stop.record(stream)
        torch.cuda.synchronize()
        ms = start.elapsed_time(stop)
    finally:
        S.slide_state_destroy(st)
    b_upd, b_pre = (26 + gsize * R) * n, (gsize * R * n if clip else 0)
    traffic, traffic_note = recorded_traffic(w.name)
    return {"workload": w.name, "description": w.description, "params": n, "replicas": R, "steps": K,
            "value": n * K / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms / K,
            "hbm_gbs": (b_upd + b_pre) / (ms / K * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": "grad_reduce_adamw_cast", "achieved": b_upd / (upd * 1e-3) / 1e9,
                         "peak": peak, "unit": "GB/s", "frac": b_upd / (upd * 1e-3) / 1e9 / peak,
                         "traffic": traffic, "traffic_note": traffic_note, "bytes_per_launch": b_upd,
                         "bytes_per_param": 26 + gsize * R, "avg_launch_ms": upd, "launches": K},
            "prepass": ({"achieved": b_pre / (pre * 1e-3) / 1e9, "frac": b_pre / (pre * 1e-3) / 1e9 / peak,
                         "avg_launch_ms": pre, "bytes_per_param": gsize * R} if clip else None),
            "step_roofline_frac": (b_upd + b_pre) / (ms / K * 1e-3) / 1e9 / peak,
            "serialised_step_frac": ((b_upd + b_pre) / (ms_traced / K * 1e-3) / 1e9 / peak
                                     if clip else None),
            "traced_step_frac": (b_upd + b_pre) / (ms_traced / K * 1e-3) / 1e9 / peak}


# ----------------------------------------------------------- streamed ----

def kernel_source_sha256():
    import hashlib
    p = os.path.join(ROOT, "mixed_precision_adam_grad_gb300", "csrc", "grad_reduce_adamw_cast.cu")
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(name):
    """DRAM bytes per launch of the fused kernel on a workload, from the ncu
    summary committed under profiles/ (traffic_<workload>.json), and where
    they come from; (None, reason) when there is none or the kernel source
    changed since the capture."""
    prof = os.path.join(ROOT, "profiles", f"traffic_{name}.json")
    if not os.path.exists(prof):
        return None, "no ncu capture recorded for this workload"
    with open(prof) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256") != kernel_source_sha256():
        return None, "the kernel changed since the ncu capture: traffic withheld"
    return rec.get("grad_reduce_adamw_cast_bytes_per_launch"), rec.get("source", "")


def mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def release_pinned_cache(torch):
    """Return the pinned host buffers that torch keeps cached after their
    tensors are freed, so the streamed legs can pin the host state."""
    import gc
    gc.collect()
    fn = getattr(torch._C, "_host_emptyCache", None)
    if fn is not None:
        fn()


def anon_huge_kb(addr):
    """AnonHugePages (kB) of the mapping of this process that holds addr
    (from /proc/self/smaps), or None where that cannot be read."""
    try:
        with open("/proc/self/smaps") as f:
            inside = False
            for line in f:
                head = line.split()
                if head and "-" in head[0] and len(head) >= 5 and not head[0].endswith(":"):
                    lo, hi = (int(x, 16) for x in head[0].split("-"))
                    inside = lo <= addr < hi
                elif inside and line.startswith("AnonHugePages:"):
                    return int(line.split()[1])
    except (OSError, ValueError):
        pass
    return None


def pinned_empty(torch, arena=None):
    """Allocator of pinned host tensors: carved from the run's arena when
    there is one, else torch's pinned allocator."""
    if arena is not None:
        return lambda shape, dtype: arena.tensor(shape, dtype)
    return lambda shape, dtype: torch.empty(shape, dtype=dtype, pin_memory=True)


PROBE_BYTES = (2 << 30) + (1 << 30) + (1 << 20)   # link probe and link monitor buffers


def link_probe(torch, nbytes=1 << 30, reps=20, arena=None):
    """Pinned host <-> device copy bandwidth (GB/s): each direction alone,
    then both at once on two streams (per direction and aggregate); medians."""
    alloc = pinned_empty(torch, arena)
    h_src = alloc(nbytes, torch.uint8)
    h_dst = alloc(nbytes, torch.uint8)
    d_dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def one(direction):
        a, b = ev(), ev()
        st = s1 if direction == "h2d" else s2
        with torch.cuda.stream(st):
            a.record(st)
            if direction == "h2d":
                d_dst.copy_(h_src, non_blocking=True)
            else:
                h_dst.copy_(d_src, non_blocking=True)
            b.record(st)
        torch.cuda.synchronize()
        return nbytes / (a.elapsed_time(b) * 1e-3) / 1e9

    def both():
        a, b1, b2 = ev(), ev(), ev()
        a.record(s1)
        s2.wait_event(a)
        with torch.cuda.stream(s1):
            d_dst.copy_(h_src, non_blocking=True)
            b1.record(s1)
        with torch.cuda.stream(s2):
            h_dst.copy_(d_src, non_blocking=True)
            b2.record(s2)
        torch.cuda.synchronize()
        t1, t2 = a.elapsed_time(b1) * 1e-3, a.elapsed_time(b2) * 1e-3
        return nbytes / t1 / 1e9, nbytes / t2 / 1e9, 2 * nbytes / max(t1, t2) / 1e9

    for _ in range(2):
        one("h2d"), one("d2h"), both()
    h2d = statistics.median(one("h2d") for _ in range(reps))
    d2h = statistics.median(one("d2h") for _ in range(reps))
    bi = [both() for _ in range(reps)]
    out = {"h2d_gbs": h2d, "d2h_gbs": d2h,
           "h2d_concurrent_gbs": statistics.median(x[0] for x in bi),
           "d2h_concurrent_gbs": statistics.median(x[1] for x in bi),
           "bidir_gbs": statistics.median(x[2] for x in bi),
           "probe": f"{nbytes >> 20} MiB pinned<->device cudaMemcpyAsync, {reps} reps, medians"}
    del h_src, h_dst, d_dst, d_src
    return out


def link_monitor(torch, seconds=2.0, chunk=64 << 20, slots=8, arena=None):
    """Both directions of the host link kept busy for `seconds` with
    back-to-back pinned <-> device copies of `chunk` bytes, every copy timed
    by its own pair of events.  The per-copy rates over time show whether the
    link held its rate for the whole window: on a host shared with other
    work it can drop for stretches of a few hundred ms, which a median-based
    probe hides.  Rates in GB/s; a copy is "slow" below 0.8 x the median."""
    alloc = pinned_empty(torch, arena)
    h_src = alloc((slots, chunk), torch.uint8)
    h_dst = alloc((slots, chunk), torch.uint8)
    d_dst = torch.empty(slots, chunk, dtype=torch.uint8, device="cuda")
    d_src = torch.empty(slots, chunk, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    n = max(8, int(seconds * 175e9 / chunk))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(2)]
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    start.record(s1)
    s2.wait_event(start)
    ev[0][0].record(s1)
    ev[1][0].record(s2)
    for i in range(n):
        j = i % slots
        with torch.cuda.stream(s1):
            d_dst[j].copy_(h_src[j], non_blocking=True)
            ev[0][i + 1].record(s1)
        with torch.cuda.stream(s2):
            h_dst[j].copy_(d_src[j], non_blocking=True)
            ev[1][i + 1].record(s2)
    torch.cuda.synchronize()
    out = {"seconds": seconds, "copy_mib": chunk >> 20}
    for d, name in ((0, "h2d"), (1, "d2h")):
        ms = [ev[d][i].elapsed_time(ev[d][i + 1]) for i in range(n)]
        gbs = [chunk / (t * 1e-3) / 1e9 for t in ms]
        med = statistics.median(gbs)
        srt = sorted(gbs)
        slow_ms = sum(t for t, g in zip(ms, gbs) if g < 0.8 * med)
        longest = run = 0.0
        for t, g in zip(ms, gbs):
            run = run + t if g < 0.8 * med else 0.0
            longest = max(longest, run)
        out[name] = {"median_gbs": med, "p5_gbs": srt[len(srt) // 20], "min_gbs": srt[0],
                     "slow_ms": slow_ms, "longest_slow_stretch_ms": longest, "window_ms": sum(ms)}
    del h_src, h_dst, d_dst, d_src
    return out


def unit_spread(units, sizes=None):
    """Slowest unit copy-in of a streamed step against the median unit, per
    parameter (sizes: parameters per unit; equal sizes if None): a ratio near
    1 means every unit met the same link rate.  Every unit of the sweep
    counts, the first and the last included."""
    import math
    sizes = sizes or [1] * len(units)
    rates = [(i, (u["h2d_end"] - u["h2d_begin"]) / max(1, sizes[i])) for i, u in enumerate(units)
             if not math.isnan(u["h2d_begin"]) and sizes[i] > 0]
    if len(rates) < 2:
        return {"unit_max_over_median": None, "slowest_unit": None}
    med = statistics.median(t for _, t in rates)
    i, t = max(rates, key=lambda x: x[1])
    return {"unit_max_over_median": t / med if med > 0 else None, "slowest_unit": i,
            "median_unit_copy_in_ms_per_gparam": med * 1e9}


def _union(intervals):
    out = []
    for a, b in sorted(intervals):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return out


def timeline_overlap(units, fwd_end):
    """Busy time of the host->device and device->host copies in the last
    streamed step (from the engine's per-unit events) and how much of it ran
    at the same time."""
    import math
    h2d = _union([(0.0, fwd_end)] + [(u["h2d_begin"], u["h2d_end"]) for u in units
                                     if not math.isnan(u["h2d_begin"])])
    d2h = _union([(u["d2h_begin"], u["d2h_end"]) for u in units if not math.isnan(u["d2h_begin"])])
    both = 0.0
    for a, b in h2d:
        for c, d in d2h:
            both += max(0.0, min(b, d) - max(a, c))
    end = max(iv[1] for iv in h2d + d2h)
    return {"step_ms": end, "h2d_busy_ms": sum(b - a for a, b in h2d), "d2h_busy_ms": sum(b - a for a, b in d2h),
            "both_busy_ms": both, "forward_sweep_ms": fwd_end,
            "units_ms": [{k: round(v, 3) for k, v in u.items()} for u in units]}


def measure_delivery(S, torch, st, layer, n, R, reps=3):
    """Delivery of one unit's BF16 copy from the pinned host mirror to R
    consumer buffers: full (R copies over the host link) against sharded (one
    copy's worth over the link, then an on-device all-gather)."""
    dst = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
    stream = torch.cuda.Stream()
    out = {"params": n, "consumers": R}
    for name, route in (("full", S.SLIDE_DELIVER_FULL), ("sharded", S.SLIDE_DELIVER_SHARDED)):
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            S.slide_deliver_bf16(st, layer, dst, route=route, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        out[name] = {"ms": best, "host_link_bytes": (R if route == S.SLIDE_DELIVER_FULL else 1) * 2 * n,
                     "device_bytes": 0 if route == S.SLIDE_DELIVER_FULL else 2 * (R - 1) * 2 * n}
    del dst
    return out


class PinnedArena:
    """The run's one pinned host allocation, of an exact size (cudaHostAlloc,
    portable and mapped), made before anything else is pinned.  The legs take
    their DMA-only host buffers from it in turn: the end-to-end leg's replicas
    and copy, the link probes' buffers and each streamed state's host state
    (handed to the library as its host_arena).  So the streamed states get
    pages that no earlier buffer used and that the CPU never touched: on these
    hosts, pinned pages that the CPU had read or written, including pages that
    earlier pinned buffers had left behind, were read several times slower by
    the copy engines for a while afterwards.

    The same class pins the run's guard block first of all: on these hosts
    (virtual machines) a fixed set of about 7 GiB of guest memory, which a
    fresh machine hands to the first pinned allocation, decays within a minute
    of being pinned to about 15 GB/s of copy-engine reads while the rest holds
    210 GB/s.  The guard holds those pages for the run and is not used."""

    def __init__(self, nbytes):
        import ctypes as C
        import ctypes.util
        lib = None
        for name in ("libcudart.so.13", ctypes.util.find_library("cudart") or "", "libcudart.so"):
            if not name:
                continue
            try:
                lib = C.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise OSError("libcudart not found")
        self._lib = lib
        lib.cudaHostAlloc.argtypes = [C.POINTER(C.c_void_p), C.c_size_t, C.c_uint]
        lib.cudaFreeHost.argtypes = [C.c_void_p]
        p = C.c_void_p()
        t0 = time.time()
        rc = lib.cudaHostAlloc(C.byref(p), C.c_size_t(nbytes), 1 | 2)   # portable | mapped
        if rc != 0 or not p.value:
            raise MemoryError(f"cudaHostAlloc({nbytes}) failed with {rc}")
        self.addr, self.nbytes, self.pin_s = p.value, nbytes, time.time() - t0
        self.top = 0

    def mark(self):
        return self.top

    def reset(self, mark=0):
        self.top = mark

    def carve(self, nbytes):
        """Address of the next nbytes (256-byte aligned) of the arena."""
        a = (self.top + 255) // 256 * 256
        if a + nbytes > self.nbytes:
            raise MemoryError(f"pinned arena: {nbytes} bytes do not fit ({self.nbytes - a} left)")
        self.top = a + nbytes
        return self.addr + a

    def tensor(self, shape, dtype):
        """A CPU tensor over the next bytes of the arena (pinned memory)."""
        import ctypes as C
        import torch
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
        numel = 1
        for d in shape:
            numel *= d
        nbytes = numel * torch.empty((), dtype=dtype).element_size()
        addr = self.carve(max(nbytes, 1))
        buf = (C.c_uint8 * max(nbytes, 1)).from_address(addr)
        return torch.frombuffer(buf, dtype=torch.uint8)[:nbytes].view(dtype).view(shape)

    def free(self):
        if self.addr:
            self._lib.cudaFreeHost(self.addr)
            self.addr = 0


def streamed_host_bytes(S, key, args):
    """Pinned host bytes of a streamed leg (its workload and layout)."""
    name, _, layout = key.partition("+")
    w = workload(name)
    in_hbm = args.streamed_bf16_in_hbm or name == "h5120x40_streamed" or layout == "bf16hbm"
    flags = S.SLIDE_FLAG_BF16_COPY_IN_HBM if in_hbm else 0
    return S.slide_state_bytes([u.numel for u in w.units], w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED,
                               flags=flags)[1]


def grad_pool(torch, synth, w, maxn, n_pool=2):
    """Pre-generated replicas in HBM (the workload's distribution) and the
    callback argument that copies them into the window for every unit."""
    import ctypes as C
    sp = synth.spec(w.seed, w.grad_kind, w.zero_prob)
    pool = [torch.empty(maxn + 64, dtype=torch.int16, device="cuda") for _ in range(n_pool * w.R)]
    for k in range(n_pool):
        for r in range(w.R):
            synth.dev_grad(pool[k * w.R + r].data_ptr(), maxn, sp, 1000 + k, 0, r, w.grad_scale)
    torch.cuda.synchronize()
    sizes = [u.numel for u in w.units]
    numel = (C.c_int64 * len(sizes))(*sizes)
    pool_ptrs = (C.c_void_p * len(pool))(*[t.data_ptr() for t in pool])
    pg = synth.PoolGrads(w.R, n_pool, 0, 0, C.cast(numel, C.c_void_p), C.cast(pool_ptrs, C.c_void_p))
    return pg, (pool, numel, pool_ptrs)


def link_roofline_s(link, N, in_hbm):
    """T_roof of one streamed step of N parameters for the measured link."""
    G = 1e9
    if in_hbm:   # the BF16 copy's delivery and write-back stay inside HBM
        return max(12 * N / (link["h2d_concurrent_gbs"] * G), 12 * N / (link["d2h_concurrent_gbs"] * G),
                   24 * N / (link["bidir_gbs"] * G))
    return (2 * N / (link["h2d_gbs"] * G)
            + max(12 * N / (link["h2d_concurrent_gbs"] * G), 14 * N / (link["d2h_concurrent_gbs"] * G),
                  26 * N / (link["bidir_gbs"] * G)))


LINK_KEYS = ("h2d_gbs", "d2h_gbs", "h2d_concurrent_gbs", "d2h_concurrent_gbs", "bidir_gbs")


def best_link(links):
    """Per rate, the highest that the run's link probes measured (each
    probe is a median of 20 copies).  That is the link's capability: the
    host's pinned memory can slow down for a while (see the link monitors), so
    a probe taken in a slow moment would lower the roofline of its leg and
    raise that leg's fraction.  Rooflines computed from it are the tightest
    the run supports."""
    out = {k: max(x[k] for x in links) for k in LINK_KEYS}
    out["probe"] = f"highest of the run's {len(links)} link probes, per rate"
    return out


def rebase_streamed(leg, link):
    """Roofline and fractions of a streamed leg against `link` (the run's
    best probe); the figures against the leg's own probe stay under
    own_probe."""
    N, in_hbm = leg["params"], leg["bf16_copy_in_hbm"]
    t = link_roofline_s(link, N, in_hbm)
    leg["own_probe"] = {"roofline_s": leg["roofline_s"], "frac": leg["frac"]}
    leg["roofline_link"] = link
    leg["roofline_s"], leg["frac"] = t, t / leg["s_per_step"]
    leg["frac_fastest_step"] = t / leg["s_per_step_min"]
    pp = leg.get("pipelined")
    if pp:
        per_dir, G = leg["link_bytes_per_step"]["h2d"], 1e9
        tp = max(per_dir / (link["h2d_concurrent_gbs"] * G), per_dir / (link["d2h_concurrent_gbs"] * G),
                 2 * per_dir / (link["bidir_gbs"] * G))
        pp["roofline_s"] = tp
        pp["frac"] = tp / pp["s_per_step"] if pp.get("s_per_step") else None


def e2e_link_roofline(e2e, link, n):
    """The fastest the host link allows for one end-to-end step of n
    parameters: the BF16 copy's device-to-host bytes run beside part of the
    replicas' host-to-device bytes, at the rates measured with both directions
    busy, and the rest of the larger direction runs alone (running the two
    directions one after the other is slower on this link).  Returns the
    bound in seconds and the measured step's fraction of it."""
    G = 1e9
    h2d, d2h = e2e["h2d_bytes_per_step"], e2e["d2h_bytes_per_step"]
    ch, cd = link["h2d_concurrent_gbs"] * G, link["d2h_concurrent_gbs"] * G
    t_both = min(h2d / ch, d2h / cd)             # both directions busy
    t = t_both + (h2d - ch * t_both) / (link["h2d_gbs"] * G) + (d2h - cd * t_both) / (link["d2h_gbs"] * G)
    measured = n / (e2e["value"] * G)
    return {"s": t, "frac": t / measured,
            "model": "device-to-host bytes beside host-to-device bytes at the concurrent rates, the rest alone; "
                     "link rates from the run's probe"}


def run_chunk_sweep(args, S, torch, synth, key, arena, link, points, steps=2):
    """TuneChunks-style sweep of the streamed engine's copy-in (host->device)
    and write-back (device->host) chunk sizes on one streamed workload: per
    point, a state on the run's pinned arena, one warm-up step and `steps`
    timed steps; s/step (median) against the link roofline of the run."""
    name, _, layout = key.partition("+")
    w = workload(name)
    sizes = [u.numel for u in w.units]
    N = sum(sizes)
    in_hbm = name == "h5120x40_streamed" or layout == "bf16hbm"
    flags = S.SLIDE_FLAG_BF16_COPY_IN_HBM if in_hbm else 0
    pg, keep = grad_pool(torch, synth, w, max(sizes))
    hp = S.hparams(*w.hparams_tuple())
    t_roof = link_roofline_s(link, N, in_hbm)
    out = []
    for h2d_mib, d2h_mib in points:
        host_b = S.slide_state_bytes(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, flags=flags)[1]
        st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED,
                                  chunk_bytes=h2d_mib << 20, chunk_bytes_d2h=d2h_mib << 20, flags=flags,
                                  host_arena=arena.addr, host_arena_bytes=host_b)
        try:
            S.slide_model_step_streamed(st, synth.pool_grad_fn_address(), pg, hp)     # warm-up
            times, spreads = [], []
            for k in range(steps):
                pg.step = 1 + k
                t0 = time.perf_counter()
                S.slide_model_step_streamed(st, synth.pool_grad_fn_address(), pg, hp)
                times.append(time.perf_counter() - t0)
                spreads.append(unit_spread(S.slide_streamed_timeline(st)[0], sizes)["unit_max_over_median"])
        finally:
            S.slide_state_destroy(st)
        med = statistics.median(times)
        out.append({"h2d_mib": h2d_mib, "d2h_mib": d2h_mib, "s_per_step": med, "frac": t_roof / med,
                    "unit_max_over_median": max(x for x in spreads if x is not None) if any(spreads) else None})
    del keep
    best = max(out, key=lambda p: p["frac"])
    return {"workload": key, "roofline_s": t_roof, "steps_per_point": steps, "points": out,
            "chosen": [best["h2d_mib"], best["d2h_mib"]],
            "note": "every point runs on the run's one pinned arena; master, m and v start at zero"}


def run_streamed(args, S, torch, synth, key, arena=None):
    """Host-resident streamed step of a whole model: s/step against the
    host-link roofline measured in the same run.  The gradient callback stands
    in for the backward pass; in the timed steps it copies pre-generated
    replicas (the workload's distribution) from a pool in HBM into the window,
    so the time is the engine's copies and update; one more step with the
    on-the-fly generator as the callback is reported beside it.  `arena`: a
    PinnedArena to hold the host state (else the state pins its own)."""
    import ctypes as C
    name, _, layout = key.partition("+")
    if layout not in ("", "bf16hbm"):
        raise ValueError(f"unknown streamed layout suffix in {key!r}")
    w = workload(name)
    sizes = [u.numel for u in w.units]
    N = sum(sizes)
    maxn = max(sizes)
    in_hbm = args.streamed_bf16_in_hbm or name == "h5120x40_streamed" or layout == "bf16hbm"
    flags = S.SLIDE_FLAG_BF16_COPY_IN_HBM if in_hbm else 0
    arena_kind = "the run's one pinned arena (state handed over as host_arena)" if arena else \
        getattr(args, "streamed_arena", "hostalloc")
    if arena_kind == "hugepages":
        flags |= S.SLIDE_FLAG_HOST_HUGE_PAGES
    _, host_b = S.slide_state_bytes(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, flags=flags)
    if arena is not None and arena.nbytes < host_b:
        return {"workload": w.name, "skipped": f"the run's pinned arena ({arena.nbytes / 1e9:.1f} GB) is smaller "
                                                f"than this leg's {host_b / 1e9:.1f} GB"}
    # with the run's arena the host state is pinned already: only working room is needed
    headroom = (6 << 30) if arena is not None else (24 << 30)
    need = (0 if arena is not None else host_b) + headroom
    if mem_available_bytes() < need:
        return {"workload": w.name, "skipped": f"host memory: {(need - headroom) / 1e9:.1f} GB to pin + "
                                                f"{headroom >> 30} GiB headroom needed, "
                                                f"{mem_available_bytes() / 1e9:.1f} GB available"}
    leg_mark = arena.mark() if arena is not None else 0
    state_addr = arena.carve(host_b) if arena is not None else None
    probe_mark = arena.mark() if arena is not None else 0
    link = link_probe(torch, arena=arena)
    if arena is not None:
        arena.reset(probe_mark)
    monitor_before = link_monitor(torch, arena=arena)
    if arena is not None:
        arena.reset(probe_mark)
    release_pinned_cache(torch)
    n_pool = 2
    sp = synth.spec(w.seed, w.grad_kind, w.zero_prob)
    pg, pool_keep = grad_pool(torch, synth, w, maxn, n_pool)
    numel = (C.c_int64 * len(sizes))(*sizes)
    mg = synth.ModelGrads(sp, len(sizes), w.R, 1, 0, C.cast(numel, C.c_void_p), None, None, None, None,
                          w.grad_scale)
    chunk_h2d = args.streamed_chunk_mib
    chunk_d2h = getattr(args, "streamed_chunk_d2h_mib", 0) or chunk_h2d
    t0 = time.time()
    st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED,
                              chunk_bytes=chunk_h2d << 20, chunk_bytes_d2h=chunk_d2h << 20, flags=flags,
                              host_arena=state_addr, host_arena_bytes=host_b if arena else 0)
    create_s = time.time() - t0
    arena_hp_kb = anon_huge_kb(S.slide_layer_ptrs(st, 0)[0])
    try:
        for ui, u in enumerate(w.units):
            synth.dev_master(S.slide_layer_ptrs(st, ui)[0], u.numel, w.seed, unit=ui)
        torch.cuda.synchronize()
        hp = S.hparams(*w.hparams_tuple())
        fn_pool, fn_gen = synth.pool_grad_fn_address(), synth.grad_fn_address()
        S.slide_model_step_streamed(st, fn_pool, pg, hp)          # warm-up step
        times, per_step, tls = [], [], []
        for k in range(args.streamed_steps):
            pg.step = 1 + k
            t0 = time.perf_counter()
            S.slide_model_step_streamed(st, fn_pool, pg, hp)      # returns after the last write-back
            times.append(time.perf_counter() - t0)
            units_tl, fwd_end = S.slide_streamed_timeline(st)
            tls.append((units_tl, fwd_end))
            per_step.append(dict(s=times[-1], **unit_spread(units_tl, sizes)))
        # steps enqueued back to back (slide_model_step_streamed_async): each
        # call returns once the step before has finished its updates, so the
        # interval between returns is the steady-state step; the next step's
        # forward sweep overlaps this step's last write-backs
        pipe_returns = []
        t_pipe0 = time.perf_counter()
        for k in range(args.streamed_steps + 1):
            pg.step = 100 + k
            S.slide_model_step_streamed_async(st, fn_pool, pg, hp)
            pipe_returns.append(time.perf_counter())
        S.slide_streamed_sync(st)
        t_pipe1 = time.perf_counter()
        pipe_steps = [b - a for a, b in zip(pipe_returns[1:], pipe_returns[2:])]
        monitor_after = link_monitor(torch, arena=arena)
        if arena is not None:
            arena.reset(probe_mark)
        fastest, slowest = times.index(min(times)), times.index(max(times))
        overlap_fast = timeline_overlap(*tls[fastest])
        overlap_slow = timeline_overlap(*tls[slowest])
        delivery = measure_delivery(S, torch, st, 0, sizes[0], w.R)
        t0 = time.perf_counter()
        S.slide_model_step_streamed(st, fn_gen, mg, hp)
        gen_s = time.perf_counter() - t0
        dev_b = S.slide_state_bytes(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, flags=flags)[0]
    finally:
        S.slide_state_destroy(st)
        del pool_keep
        if arena is not None:
            arena.reset(leg_mark)
    s_step = statistics.median(times)
    cpu = None
    if not args.no_cpu_baseline:
        n_s = min(1 << 22, maxn)
        rate, c_steps, c_el = oracle_sample_rate(w, n_s, 4.0, 100, seed_offset=3000)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "s_per_step_extrapolated": N / (rate * 1e9),
               "sample": f"first {n_s} parameters of one unit as a layer of their own, R={w.R}, "
                         f"{c_steps} steps ({c_el:.1f} s of single-thread CPU time); the per-parameter rate "
                         f"is extrapolated to the whole model's {N} parameters"}
    t_roof = link_roofline_s(link, N, in_hbm)
    per_dir = 12 * N if in_hbm else 14 * N
    G = 1e9
    # with steps overlapped, the forward sweep shares the link with the write-back
    t_roof_pipe = max(per_dir / (link["h2d_concurrent_gbs"] * G), per_dir / (link["d2h_concurrent_gbs"] * G),
                      2 * per_dir / (link["bidir_gbs"] * G))
    s_pipe = statistics.median(pipe_steps) if pipe_steps else None
    return {"workload": w.name, "description": w.description, "params": N, "replicas": w.R,
            "steps": args.streamed_steps, "s_per_step": s_step, "s_per_step_each": times,
            "s_per_step_min": min(times), "s_per_step_mean": statistics.mean(times),
            "gparam_s": N / s_step / 1e9, "roofline_s": t_roof, "frac": t_roof / s_step,
            "frac_fastest_step": t_roof / min(times), "per_step": per_step,
            "link_bytes_per_step": {"h2d": per_dir, "d2h": per_dir}, "bf16_copy_in_hbm": in_hbm,
            "achieved_link_gbs_each_way": per_dir / s_step / 1e9,
            "link": link, "link_monitor_before": monitor_before, "link_monitor_after": monitor_after,
            "host_pinned_gb": host_b / 1e9, "window_gb": dev_b / 1e9,
            "create_s": create_s, "chunk_mib": chunk_h2d, "chunk_h2d_mib": chunk_h2d, "chunk_d2h_mib": chunk_d2h,
            "pinned_arena": arena_kind, "arena_pin_s": arena.pin_s if arena else None,
            "arena_huge_page_kb": arena_hp_kb,
            "grad_callback": f"copies pre-generated replicas ({n_pool} sets, the workload's distribution) "
                             "from HBM into the window",
            "s_per_step_with_generator_callback": gen_s,
            "cpu_baseline": cpu,
            "timeline_fastest_step": overlap_fast, "timeline_slowest_step": overlap_slow,
            "bf16_delivery": delivery,
            "timing": "host wall clock around each synchronous model step; s_per_step is the median",
            "pipelined": {"s_per_step": s_pipe, "roofline_s": t_roof_pipe,
                          "frac": (t_roof_pipe / s_pipe) if s_pipe else None,
                          "s_per_step_each": pipe_steps,
                          "s_per_step_incl_last_drain": (t_pipe1 - t_pipe0) / (args.streamed_steps + 1),
                          "roofline": "max(B/B'_h2d, B/B'_d2h, 2B/B_bidir), B the bytes each way per step",
                          "timing": "intervals between the returns of slide_model_step_streamed_async calls "
                                    "(each returns once the step before has finished its updates)"}}


# --------------------------------------------------------------- ours ----

def run_ours(args):
    import torch

    import mixed_precision_adam_grad_gb300 as S
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    w = workload(args.workload)
    if args.slice_params > 0:
        w.units[0] = slice_unit(w.units[0], args.slice_params)
    n = w.units[0].numel
    R = w.R
    clip = w.max_grad_norm > 0
    hp = S.hparams(*w.hparams_tuple())
    stream = torch.cuda.Stream()

    # The run's one pinned host arena, pinned before anything else: large
    # enough for the end-to-end leg and the largest streamed leg that fits the
    # host (legs use it one after another; only DMA touches it).
    arena = guard = None
    streamed_keys = []
    if world == 1:
        also = [x for x in args.streamed_also.split(",") if x and x != args.streamed_workload]
        streamed_keys = [] if args.no_streamed else [args.streamed_workload] + also
        needs = [0 if args.no_e2e else 2 * (2 * R * n + 2 * n) + (1 << 20)]
        try:
            if args.pinned_guard_gib > 0 and (streamed_keys or not args.no_e2e):
                guard = PinnedArena(args.pinned_guard_gib << 30)
            avail = mem_available_bytes() - (16 << 30)
            needs += [b for b in (streamed_host_bytes(S, k, args) + PROBE_BYTES for k in streamed_keys)
                      if b <= avail]
            if args.streamed_arena == "hostalloc" and max(needs) > 0:
                arena = PinnedArena(max(needs))
        except (OSError, MemoryError) as exc:   # no arena: every state pins its own host memory
            print(f"detail {json.dumps({'pinned_arena_unavailable': str(exc)})}", flush=True)
            arena = None

    st = S.slide_state_create([n], R, device=local, flags=0 if args.no_e2e else S.SLIDE_FLAG_HOST_INPUTS)
    try:
        th_d = S.slide_layer_ptrs(st, 0)[0]
        synth.dev_master(th_d, n, w.seed + 100 * rank, stream=stream.cuda_stream)
        batches = []
        for b in range(args.batches):
            reps = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
            for r, t in enumerate(reps):
                for (off, ln), sc in zip(w.units[0].segments(), w.tensor_scales(0)):
                    synth.dev_grad(t.data_ptr() + 2 * off, ln, synth.spec(w.seed + 100 * rank, w.grad_kind,
                                                                          w.zero_prob),
                                   0, b + 1, r, sc, offset=off, stream=stream.cuda_stream)
            batches.append(reps)
        torch.cuda.synchronize()

        def step(i):
            S.slide_layer_step(st, 0, batches[i % len(batches)], hp, stream)

        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()

        gpu_index = local
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            try:
                gpu_index = int(vis.split(",")[local])
            except ValueError:
                pass
        sampler = ClockSampler(gpu_index)
        sampler.start()
        # soak: same steps, untimed, so clocks settle and the sampler sees load
        t_end = time.time() + args.soak_s
        i = 0
        while time.time() < t_end:
            for _ in range(20):
                step(i)
                i += 1
            stream.synchronize()

        K = args.steps
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for trio in ev:          # create the CUDA events (torch creates them on first record)
            for e in trio:
                e.record(stream)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(K):
            if not clip:   # with the clip, an event between pre-pass and update would serialise them
                S.slide_trace_events(st, ev[k][0], ev[k][1], ev[k][2])
            step(k)
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clocks = sampler.stop()
        S.slide_trace_events(st)
        ms_total = start.elapsed_time(stop)
        serialised_ms = None
        if clip:
            # The kernel split: K more steps, each with its trace events, which
            # make the update wait for the pre-pass's end.
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for k in range(K):
                S.slide_trace_events(st, ev[k][0], ev[k][1], ev[k][2])
                step(K + k)
            s1.record(stream)
            torch.cuda.synchronize()
            S.slide_trace_events(st)
            serialised_ms = s0.elapsed_time(s1) / K
        pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
        upd_ms = [e[1].elapsed_time(e[2]) for e in ev]
        ms_total = max_over_ranks(ms_total, dist)

        # End to end through the C ABI with host buffers: every step is one
        # slide_layer_step_host call on the step's R replicas in pinned host
        # memory and a pinned host buffer for its BF16 copy.  The library copies
        # the replicas into one of its two device staging sets on its copy
        # stream (the copy-in of step k+1 overlaps the update of step k), runs
        # the step behind the copy and copies the BF16 copy back on `stream`.
        e2e = None
        if not args.no_e2e:
            Ke = max(3, min(args.e2e_steps, K))
            alloc = pinned_empty(torch, arena)
            host_reps = [[alloc(n, torch.int16) for _ in range(R)] for _ in range(2)]
            for b in range(2):
                for r in range(R):
                    host_reps[b][r].copy_(batches[b % len(batches)][r][:n])
            out_host = [alloc(n, torch.int16) for _ in range(2)]
            torch.cuda.synchronize()

            def run_e2e(steps):
                for k in range(steps):
                    S.slide_layer_step_host(st, 0, host_reps[k % 2], hp, stream, out_host[k % 2])

            run_e2e(3)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run_e2e(Ke)
            e1.record(stream)        # behind the last step's copy-out, which is behind its copy-in
            torch.cuda.synchronize()
            ms_e2e = e0.elapsed_time(e1)
            ms_e2e = max_over_ranks(ms_e2e, dist)
            e2e = {"value": n * Ke * world / (ms_e2e * 1e-3) / 1e9, "unit": UNIT,
                   "h2d_bytes_per_step": 2 * R * n, "d2h_bytes_per_step": 2 * n, "steps": Ke,
                   "call": "slide_layer_step_host (host replicas in, host BF16 copy out)",
                   "pipelining": "the library's copy stream: the copy-in of step k+1 overlaps step k's update"}
            del host_reps, out_host
            if arena is not None:
                arena.reset()
    finally:
        S.slide_state_destroy(st)

    del batches
    release_pinned_cache(torch)
    torch.cuda.empty_cache()
    variant = None
    cpu_route = None
    others = None
    if not args.no_variants and world == 1:
        from synth import workloads as W
        peak0 = measured_peaks()[0]
        variant = measure_hbm_workload(args, S, torch, synth, peak0, W.h2560_r4_clip_fp32grads())
        others = {name: measure_hbm_workload(args, S, torch, synth, peak0, W.ALL[name](),
                                             max_steps=200 if name == "h5120_R8_logscale" else 500)
                  for name in W.HBM_RESIDENT if name != args.workload}
        import reduce_routes
        # the host reduction reads and writes these buffers with the CPU, so
        # they come from torch's pinned memory, not from the arena that the
        # streamed states use (pinned pages the CPU has touched are read
        # slowly by the copy engines for a while on these hosts)
        # on the h2560 R = 4 layer (the headline layer's buffers would crowd the
        # host next to the largest streamed leg's pinned state)
        w_route = W.h2560_r4_clip()
        cpu_route = reduce_routes.measure_cpu_reduce_route(S, torch, synth, w_route.units[0].numel, w_route.R)
        cpu_route["workload"] = w_route.name
    streamed = streamed_also = chunk_sweep = None
    release_pinned_cache(torch)
    try:
        if streamed_keys:
            streamed = run_streamed(args, S, torch, synth, args.streamed_workload, arena)
            also = streamed_keys[1:]
            if also:
                streamed_also = {x: run_streamed(args, S, torch, synth, x, arena) for x in also}
            legs = [x for x in [streamed] + list((streamed_also or {}).values()) if "link" in x]
            link = best_link([x["link"] for x in legs]) if legs else None
            for leg in legs:
                rebase_streamed(leg, link)
            if e2e is not None and link:
                e2e["link_roofline"] = e2e_link_roofline(e2e, link, n)
            if args.chunk_sweep and arena is not None and link:
                pts = [tuple(int(v) for v in p.split(":")) for p in args.chunk_sweep.split(",")]
                chunk_sweep = {}
                for key in [k for k in args.chunk_sweep_workloads.split(",") if k]:
                    if streamed_host_bytes(S, key, args) <= arena.nbytes:
                        chunk_sweep[key] = run_chunk_sweep(args, S, torch, synth, key, arena, link, pts)
    finally:
        if arena is not None:
            arena.free()
        if guard is not None:
            guard.free()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    bytes_upd = (26 + 2 * R) * n
    bytes_pre = 2 * R * n if clip else 0
    upd_avg = statistics.mean(upd_ms)
    pre_avg = statistics.mean(pre_ms) if clip else 0.0
    ach_upd = bytes_upd / (upd_avg * 1e-3) / 1e9
    ach_pre = bytes_pre / (pre_avg * 1e-3) / 1e9 if clip else None
    ms_step = ms_total / K
    value = n * K * world / (ms_total * 1e-3) / 1e9
    step_bytes = bytes_upd + bytes_pre

    cpu = cpu_all = None
    if not args.no_cpu_baseline and world == 1:
        rate, steps, el = oracle_sample_rate(w, 1 << 24 if n >= (1 << 24) else n, 12.0, 1000)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "gbs": rate * (26 + 2 * R), "gbs_bytes_per_param": 26 + 2 * R, "cpu_model": cpu_model(),
               "sample": f"first {min(n, 1 << 24)} parameters of the layer as a layer of their own, "
                         f"R={R}{', clip over the sample' if clip else ''}, {steps} steps "
                         f"({el:.1f} s of single-thread CPU time; inputs generated outside the timed calls)"}
        import oracle
        rate_all, steps_all, el_all = oracle_sample_rate(w, 1 << 24 if n >= (1 << 24) else n, 6.0, 1000,
                                                         openmp=True)
        cpu_all = {"value": rate_all, "unit": UNIT, "cores": oracle.threads(True), "kind": "oracle_openmp",
                   "gbs": rate_all * (26 + 2 * R), "gbs_bytes_per_param": 26 + 2 * R, "cpu_model": cpu_model(),
                   "sample": f"the same slice, the oracle source built with -fopenmp (element loops split "
                             f"across threads), {steps_all} steps in {el_all:.1f} s"}
    traffic, traffic_note = (recorded_traffic(w.name) if args.slice_params <= 0
                             else (None, "profiling slice: no full-launch capture applies"))


    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "params": n, "replicas": R,
                   "max_grad_norm": w.max_grad_norm, "parallelism": f"replicas-only x{world}",
                   "l2": f"inputs larger than L2: each step touches {step_bytes / 1e9:.2f} GB; "
                         f"{args.batches} gradient batches cycled",
                   "clock_samples": "nvidia-smi every 200 ms over a soak of the same step and the "
                                    "timed region",
                   **({"slice_params": n, "note": "profiling slice of the unit, not a full-size measurement"}
                      if args.slice_params > 0 else {})},
        "hbm_gbs": step_bytes / (ms_step * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "grad_reduce_adamw_cast",
                     "achieved": ach_upd, "peak": peak, "unit": "GB/s", "frac": ach_upd / peak,
                     "traffic": traffic, "traffic_note": traffic_note, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "bytes_per_launch": bytes_upd, "avg_launch_ms": upd_avg,
                     "bytes_per_param": 26 + 2 * R, "launches": K},
        "prepass": ({"kernel": "grad_sqnorm_pipe", "achieved": ach_pre, "unit": "GB/s", "frac": ach_pre / peak,
                     "bytes_per_launch": bytes_pre, "avg_launch_ms": pre_avg,
                     "split_note": "pre-pass and update timed in K further steps with trace events between "
                                   "them, which serialise them; the timed region runs the steps without them",
                     "serialised_step_frac": step_bytes / (serialised_ms * 1e-3) / 1e9 / peak}
                    if clip else None),
        "step_roofline_frac": (step_bytes / (ms_step * 1e-3) / 1e9) / peak,
        "gpu_launches": K * (2 if clip else 1),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "fp32_grad_variant": variant,
        "other_hbm_workloads": others,
        "cpu_reduce_route": cpu_route,
        "streamed": streamed,
        "streamed_also": streamed_also,
        "chunk_sweep": chunk_sweep,
    }
    report(line, args.detail_out)
    if dist:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------- report ----

def _r(x, digits=4):
    """x rounded to `digits` significant digits (None and non-floats as is)."""
    if isinstance(x, float):
        if x != x or x in (float("inf"), float("-inf")):
            return None
        return float(f"{x:.{digits}g}")
    return x


def _pick(d, keys):
    return {k: _r(d[k]) for k in keys if d is not None and k in d and d[k] is not None}


def compact_hbm_leg(leg):
    """One HBM-resident leg in a few fields: rate, kernel and step fractions."""
    if leg is None:
        return None
    out = {"value": _r(leg["value"]), "frac": _r(leg["roofline"]["frac"]),
           "step_frac": _r(leg["step_roofline_frac"]), "launches": leg["steps"]}
    if leg.get("prepass"):
        out["prepass_frac"] = _r(leg["prepass"]["frac"])
    if leg.get("serialised_step_frac") is not None:
        out["serialised_step_frac"] = _r(leg["serialised_step_frac"])
    return out


def compact_streamed(leg):
    """One host-streamed leg: median s/step against the link roofline, the
    concurrent link rates it was measured against and the unit spread (median
    over the steps, and the worst step)."""
    if leg is None:
        return None
    if "skipped" in leg:
        return {"skipped": leg["skipped"][:160]}
    spreads = sorted(p["unit_max_over_median"] for p in leg.get("per_step", [])
                     if p.get("unit_max_over_median") is not None)
    link = leg.get("roofline_link", leg.get("link", {}))
    out = {"bf16_in_hbm": leg["bf16_copy_in_hbm"], "s_per_step": _r(leg["s_per_step"]),
           "roofline_s": _r(leg["roofline_s"]), "frac": _r(leg["frac"]),
           "frac_fastest": _r(leg["frac_fastest_step"]),
           "link_gbs_each_way": _r(leg["achieved_link_gbs_each_way"]),
           "link_concurrent_gbs": [_r(link.get("h2d_concurrent_gbs"), 3), _r(link.get("d2h_concurrent_gbs"), 3)],
           "unit_max_over_median": _r(statistics.median(spreads), 3) if spreads else None,
           "unit_max_over_median_worst": _r(spreads[-1], 3) if spreads else None,
           "chunk_mib": [leg.get("chunk_h2d_mib", leg.get("chunk_mib")), leg.get("chunk_d2h_mib", leg.get("chunk_mib"))]}
    if "pinned_arena" in leg:   # "shared": the run's one pinned arena; else how the state pinned its own
        a = leg["pinned_arena"]
        out["arena"] = "shared" if a.startswith("the run's") else a
    if leg.get("cpu_baseline"):
        out["cpu_s_per_step"] = _r(leg["cpu_baseline"]["s_per_step_extrapolated"], 3)
    pp = leg.get("pipelined")
    if pp and pp.get("s_per_step"):
        out["async_s_per_step"] = _r(pp["s_per_step"])
    return out


HEADLINE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data")


def compact_headline(full):
    """The last stdout line: the headline workload and the roofline of its
    dominant kernel, the CPU baselines, the end-to-end figure, the clocks and
    one short summary per other leg; the timelines, per-step arrays and link
    monitors stay in the detail lines."""
    line = {k: _r(full[k]) for k in HEADLINE_KEYS}
    cfg = full["config"]
    line["config"] = {k: cfg[k] for k in ("workload", "description", "params", "replicas", "max_grad_norm",
                                          "parallelism", "l2") if k in cfg}
    if "slice_params" in cfg:
        line["config"]["slice_params"] = cfg["slice_params"]
    rf = full["roofline"]
    line["roofline"] = {k: _r(rf[k]) for k in ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic",
                                               "bytes_per_launch", "bytes_per_param", "avg_launch_ms",
                                               "launches")}
    line["roofline"]["peak_kind"] = "measured" if rf.get("peak_kind", "").startswith("measured") else "fallback"
    line["hbm_gbs"] = _r(full["hbm_gbs"])
    line["step_roofline_frac"] = _r(full["step_roofline_frac"])
    if full.get("prepass"):
        line["prepass"] = _pick(full["prepass"], ("kernel", "achieved", "frac", "avg_launch_ms", "serialised_step_frac"))
    line["gpu_launches"] = full["gpu_launches"]
    ck = full.get("clocks") or {}
    line["clocks"] = {"sm_mhz": ck.get("sm_mhz"), "sm_max_mhz": ck.get("sm_max_mhz"),
                      "reasons": ck.get("reasons", []), "samples": ck.get("samples")}
    if full.get("e2e"):
        line["e2e"] = _pick(full["e2e"], ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "steps"))
        if full["e2e"].get("link_roofline"):
            line["e2e"]["link_frac"] = _r(full["e2e"]["link_roofline"]["frac"])
    for k in ("cpu_baseline", "cpu_baseline_all_cores"):
        c = full.get(k)
        if c:
            line[k] = {"value": _r(c["value"]), "unit": c["unit"], "cores": c["cores"], "kind": c["kind"],
                       "gbs": _r(c.get("gbs")), "sample": c["sample"][:160]}
    legs = {}
    for name, leg in (full.get("other_hbm_workloads") or {}).items():
        legs[name] = compact_hbm_leg(leg)
    if full.get("fp32_grad_variant"):
        legs[full["fp32_grad_variant"]["workload"]] = compact_hbm_leg(full["fp32_grad_variant"])
    if legs:
        line["hbm_legs"] = legs
    st = {}
    if full.get("streamed"):
        st[full["streamed"]["workload"] + ("+bf16hbm" if full["streamed"].get("bf16_copy_in_hbm") else "")] = \
            compact_streamed(full["streamed"])
    for name, leg in (full.get("streamed_also") or {}).items():
        st[name] = compact_streamed(leg)
    if st:
        line["streamed"] = st
    cr = full.get("cpu_reduce_route")
    if cr:
        line["cpu_reduce_route"] = {"workload": cr.get("workload"),
                                    "cpu_route_s": _r(cr["cpu_route"]["s"]), "gpu_route_s": _r(cr["gpu_route"]["s"]),
                                    "cpu_route_d2h_bytes": cr["cpu_route"]["d2h_bytes"],
                                    "identical_results": cr["identical_results"]}
    sw = full.get("chunk_sweep")
    if sw:
        line["chunk_sweep"] = {k: {"chosen": v.get("chosen"),
                                   "points": [[p["h2d_mib"], p["d2h_mib"], _r(p["frac"], 3)] for p in v["points"]]}
                               for k, v in sw.items()}
    return line


def report(full, detail_out=""):
    """Print every leg in full on its own "detail" line, then the compact
    headline as the last line of stdout; optionally write the whole record."""
    for key in ("other_hbm_workloads", "fp32_grad_variant", "cpu_reduce_route", "chunk_sweep", "streamed",
                "streamed_also"):
        if full.get(key) is not None:
            print("detail " + json.dumps({key: full[key]}), flush=True)
    if detail_out:
        with open(detail_out, "w") as f:
            json.dump(full, f, indent=1)
    line = compact_headline(full)
    print(json.dumps(line, separators=(",", ":")), flush=True)
    return line


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
