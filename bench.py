#!/usr/bin/env python3
"""Benchmark of exact attention (FlashAttention-2 style) on one GB300.

One step = one forward plus one backward pass of causal bf16 attention over
the B4 H32 S4096 d80 2.7B-LM workload (``c4``, Q, K, V ~ 2 N(0,1)), inputs
resident in HBM.  Prints ONE JSON line (rank 0):

  value        fwd+bwd TFLOP/s, FLOPs = 3.5 * 4*B*H*S^2*d * 1/2 (causal), whole job
  e2e          the same metric through fa_fwd_bwd_host, the C-ABI entry on pinned
               host buffers: H2D of q, k, v, dO and D2H of o, lse, dq, dk, dv
               inside the timing, steps rotating over three streams
  roofline     the dominant kernel's algorithmic TFLOP/s against the measured peak
  cpu_baseline the fp64 oracle timed on this host's cores on a bounded sample
  target_shapes  fwd, bwd and fwd+bwd TFLOP/s of B1 H16 S4096/8192 d64/d128
               causal bf16, with their fractions of the measured bf16 peak

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
        [--workload c2|c3|c4|sweep:S:d] [--no-target-shapes]
Under torchrun every rank runs its own copy of the workload (independent
(batch, head) slices: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from seeded_inputs import WORKLOADS, Workload, make_inputs  # noqa: E402

L2_FLUSH_BYTES = 256 << 20          # > the 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c4")
    ap.add_argument("--no-target-shapes", action="store_true",
                    help="skip the B1 H16 S4096/8192 d64/d128 points reported beside the workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lean", action="store_true",
                    help="only the fwd+bwd steps of --workload (warm-up and timed), one short JSON line: "
                         "the command the ncu captures run, with nothing else on the device")
    ap.add_argument("--non-causal", action="store_true",
                    help="with --lean: the workload without the causal mask")
    ap.add_argument("--deterministic", action="store_true",
                    help="with --lean: the step's backward through fa_bwd_deterministic")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--memory", action="store_true",
                    help="instead of timing: peak device memory of fwd+bwd against a materialised-score "
                         "PyTorch baseline on --workload (one JSON line)")
    return ap.parse_args()


def workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep:"):           # sweep:S:d[:dtype]
        parts = name.split(":")
        S, d = int(parts[1]), int(parts[2])
        dt = parts[3] if len(parts) > 3 else "bf16"
        return Workload(name, 1, 16, S, d, dt, (True,), 1.0, 4242)
    raise SystemExit(f"unknown workload {name}")


def flops_fwd(w: Workload, causal=True) -> float:
    f = 4.0 * w.B * w.H * w.S * w.S * w.d
    return f / 2 if causal else f


def workload_config(w: Workload, causal: bool) -> dict:
    """The keys of the JSON line's `config` that name the workload; both arms
    report them alike and add their own timing keys."""
    return {"workload": f"{w.name}: B{w.B} H{w.H} S{w.S} d{w.d} {'causal' if causal else 'non-causal'} {w.dtype}",
            "B": w.B, "H": w.H, "S": w.S, "d": w.d, "causal": causal}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a window."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for (_, r) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(w: Workload, seconds: float):
    """Time the fp64 oracle (fwd + standard bwd) on whole (b, h) slices of the
    workload until `seconds` have passed; returns (TFLOP/s on the bench's FLOP
    count, slices done, elapsed seconds, threads)."""
    import numpy as np
    import oracle
    q, k, v, do = make_inputs(w.B, w.H, w.S, w.d, w.dtype, w.seed, w.qkv_scale)
    f64 = lambda t: t.to(torch.float64).numpy()
    per_slice = 3.5 * flops_fwd(Workload("s", 1, 1, w.S, w.d, w.dtype, (True,)), True)
    done, t0 = 0, time.perf_counter()
    slices = [(b, h) for b in range(w.B) for h in range(w.H)]
    while True:
        b, h = slices[done % len(slices)]
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        oracle.attention_fwd(sl(q), sl(k), sl(v), True, w.scale)
        oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), True, w.scale)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", "0")) or len(os.sched_getaffinity(0))
    return per_slice * done / el / 1e12, done, el, threads


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = workload(args.workload)
    import numpy as np  # noqa: F401
    import oracle
    q, k, v, do = make_inputs(w.B, w.H, w.S, w.d, w.dtype, w.seed, w.qkv_scale)
    f64 = lambda t: t.to(torch.float64).numpy()
    per_slice = 3.5 * flops_fwd(Workload("s", 1, 1, w.S, w.d, w.dtype, (True,)), True)
    slices = [(b, h) for b in range(w.B) for h in range(w.H)]

    def step(i):
        b, h = slices[i % len(slices)]
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        oracle.attention_fwd(sl(q), sl(k), sl(v), True, w.scale)
        oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), True, w.scale)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = per_slice * args.steps / el / 1e12
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", "0")) or len(os.sched_getaffinity(0))
    sample = f"one (b,h) slice of {w.name} (S={w.S}, d={w.d}) per step: fp64 fwd + standard bwd"
    print(json.dumps({
        "impl": "reference", "metric": "attention fwd+bwd TFLOP/s (bf16, causal)", "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**workload_config(w, True), "sample": "one (b,h) slice per step",
                   "parallelism": "rank 0 alone, on the host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def sources_sha16(paths) -> str:
    """First 16 hex digits of the SHA-256 of the listed files, concatenated in
    order (a kernel source and the headers it includes)."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(kernel_name: str, workload_name: str):
    """DRAM bytes per launch from a committed ncu summary, only if the kernel
    source and the headers it was built from are unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        j = json.load(open(p))
        ent = j.get(kernel_name, {}).get(workload_name)
        if not ent:
            return None
        paths = ent["sources"] if "sources" in ent else [ent["source"]]
        return ent["dram_bytes_per_launch"] if sources_sha16(paths) == ent["source_sha256_16"] else None
    except Exception:
        return None


def time_steps(step, n, flush, stream):
    """Device time (ms) of each of n calls of `step`, CUDA events on the
    launching stream, L2 flushed before each (outside the events)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def kernel_times(fa, step, n, flush):
    """{kernel: (total ms, launches)} over n steps from the library's own
    events around every launch (they serialise the kernels; step times are
    taken without them)."""
    fa.profile_read()                      # drop anything recorded so far
    fa.profile_enable(True)
    for _ in range(n):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    fa.profile_enable(False)
    prof = fa.profile_read()
    fa.check_status()
    return prof


def per_launch_ms(prof, name):
    tot, n = prof.get(name, (0.0, 0))
    return tot / n if n else None


def bwd_rates(f_fwd, prof):
    """Backward TFLOP/s on the backward's FLOP count (2.5x the forward's):
    of the main backward kernel alone, and of the whole backward step
    (D preprocess + main kernel + dQ conversion, from their own events)."""
    main = per_launch_ms(prof, "bwd_main")
    parts = [per_launch_ms(prof, k) for k in ("bwd_preprocess", "bwd_main", "dq_convert")]
    step_ms = sum(x for x in parts if x) if main else None
    rate = lambda ms: 2.5 * f_fwd / (ms * 1e-3) / 1e12 if ms else None
    return {"bwd_kernel_tflops": rate(main), "bwd_step_ms": step_ms, "bwd_step_tflops": rate(step_ms)}


TARGET_SHAPES = [(4096, 64), (4096, 128), (8192, 64), (8192, 128)]


def measure_target_shapes(fa, dev, flush, stream, peaks, seed_offset):
    """Causal bf16 B1 H16 at S = 4096, 8192 and d = 64, 128: the shapes the
    throughput target is stated for.  Each point: whole fwd+bwd steps timed
    as the main measurement is, then per-kernel times from the library's
    events."""
    out = []
    for S, d in TARGET_SHAPES:
        w = Workload(f"B1 H16 S{S} d{d}", 1, 16, S, d, "bf16", (True,), 1.0, 4300 + S + d + seed_offset)
        q, k, v, do = (t.to(dev) for t in make_inputs(w.B, w.H, w.S, w.d, w.dtype, w.seed))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
        g = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        ws = torch.empty(fa.bwd_workspace_size(w.B, w.H, w.S, w.d, q.dtype), device=dev, dtype=torch.uint8)

        def step():
            fa.fwd(q, k, v, True, w.scale, out=o, lse=lse)
            fa.bwd(q, k, v, o, do, lse, True, w.scale, workspace=ws, out=g)

        for _ in range(3):
            step()
        fa.check_status()
        ms = time_steps(step, 20, flush, stream)
        prof = kernel_times(fa, step, 10, flush)
        f_fwd = flops_fwd(w, True)
        ms_step = sum(ms) / len(ms)
        fwd_ms = per_launch_ms(prof, "fwd")
        step_tf = 3.5 * f_fwd / (ms_step * 1e-3) / 1e12
        out.append({"shape": f"B1 H16 S{S} d{d} causal bf16", "fwd_bwd_step_ms": ms_step,
                    "fwd_bwd_step_tflops": step_tf,
                    "frac_of_burst_peak": step_tf / peaks["bf16_tflops"],
                    "frac_of_sustained_peak": step_tf / peaks["bf16_tflops_sustained"],
                    "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None,
                    **bwd_rates(f_fwd, prof)})
        del q, k, v, do, o, lse, g, ws
    return out


def run_ours(args, world, rank, local):
    import exact_attention_fa2_gb300 as fa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load_library()
    w = workload(args.workload)
    if (args.non_causal or args.deterministic) and not args.lean:
        raise SystemExit("--non-causal and --deterministic are options of --lean")
    causal = not args.non_causal
    scale = w.scale
    q, k, v, do = make_inputs(w.B, w.H, w.S, w.d, w.dtype, w.seed + 7919 * rank, w.qkv_scale)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    dqd, dkd, dvd = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(fa.bwd_workspace_size(w.B, w.H, w.S, w.d, qd.dtype), device=dev, dtype=torch.uint8)
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def step():
        fa.fwd(qd, kd, vd, causal, scale, out=od, lse=lsed)
        fa.bwd(qd, kd, vd, od, dod, lsed, causal, scale, workspace=ws, out=(dqd, dkd, dvd),
               deterministic=args.deterministic)

    for _ in range(max(3, args.warmup)):
        step()
    fa.check_status()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    step_ms = time_steps(step, args.steps, flush, stream)    # L2 flushed between timed steps
    barrier(world)
    t1 = time.time()
    fa.check_status()
    ms_per_step = max_over_ranks(sum(step_ms) / len(step_ms), world)

    if args.lean:
        if rank == 0:
            f = 3.5 * flops_fwd(w, causal)
            print(json.dumps({"lean": True, "workload": workload_config(w, causal)["workload"],
                              "deterministic_bwd": args.deterministic,
                              "ms_per_step": ms_per_step, "value": world * f / (ms_per_step * 1e-3) / 1e12,
                              "unit": "TFLOP/s", "steps": args.steps, "warmup": args.warmup}), flush=True)
        sampler.stop()
        return 0

    # Per-kernel device times from a separate pass with the library's timing
    # events around every launch (they serialise the kernels, so the step
    # time above is taken without them).
    prof_steps = max(5, min(args.steps, 50))
    prof = kernel_times(fa, step, prof_steps, flush)
    launches_per_step = sum(v[1] for v in prof.values()) / prof_steps

    # The same step with the deterministic backward (fa_bwd_deterministic:
    # dK/dV-only kernel plus the query-tile-outer dQ pass), timed the same way
    # after the main measurement, and its kernels from the library's events.
    def step_det():
        fa.fwd(qd, kd, vd, causal, scale, out=od, lse=lsed)
        fa.bwd(qd, kd, vd, od, dod, lsed, causal, scale, workspace=ws, out=(dqd, dkd, dvd), deterministic=True)

    for _ in range(3):
        step_det()
    det_steps = max(5, min(args.steps, 50))
    barrier(world)
    det_ms = time_steps(step_det, det_steps, flush, stream)
    fa.check_status()
    det_ms_per_step = max_over_ranks(sum(det_ms) / det_steps, world)
    prof_det = kernel_times(fa, step_det, 5, flush)

    # End to end through the C ABI with host buffers (fa_fwd_bwd_host): every
    # step copies q, k, v, dO from pinned host memory, runs forward and
    # backward, and copies o, lse, dq, dk, dv back.  Steps rotate over three
    # streams, each with its own device buffer and host outputs, so one step's
    # copies overlap another's kernels (as a training loop with a data loader
    # would run); the figure is the whole run's device time over its steps.
    # The three device buffers (> 129 MB together at c2) keep each step's
    # inputs out of L2 when it starts.
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    NR = 3
    streams = [torch.cuda.Stream(device=dev) for _ in range(NR)]
    bufs = [torch.empty(fa.fwd_bwd_host_buffer_size(w.B, w.H, w.S, w.d, qd.dtype), device=dev, dtype=torch.uint8)
            for _ in range(NR)]
    houts = []
    for _ in range(NR):
        houts.append((torch.empty_like(hq).pin_memory(), torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory(),
                      torch.empty_like(hq).pin_memory(), torch.empty_like(hq).pin_memory(), torch.empty_like(hq).pin_memory()))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in houts[0])
    e2e_steps = max(6, min(args.steps, 60))

    def e2e_run(n):
        for i in range(n):
            r = i % NR
            fa.fwd_bwd_host(hq, hk, hv, hdo, houts[r], bufs[r], causal, scale, stream=streams[r])

    e2e_run(NR)
    torch.cuda.synchronize()
    fa.check_status()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for st in streams:
        st.wait_event(start)
    e2e_run(e2e_steps)
    for st in streams:
        stream.wait_stream(st)
    end.record(stream)
    end.synchronize()
    fa.check_status()
    barrier(world)
    e2e_ms_step = max_over_ranks(start.elapsed_time(end) / e2e_steps, world)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    targets = None
    if not args.no_target_shapes:
        targets = measure_target_shapes(fa, dev, flush, stream, load_peaks(), 7919 * rank)

    f_fwd = flops_fwd(w, causal)
    step_flops = 3.5 * f_fwd
    value = world * step_flops / (ms_per_step * 1e-3) / 1e12
    e2e_value = world * step_flops / (e2e_ms_step * 1e-3) / 1e12
    peaks = load_peaks()

    # Dominant kernel: the one with the largest share of timed device time.
    kern_flops = {"fwd": f_fwd, "bwd_main": 2.5 * f_fwd}
    shares = {k: v[0] for k, v in prof.items()}
    dom = max(("fwd", "bwd_main"), key=lambda k: shares[k])
    dom_ms, dom_n = prof[dom]
    achieved = kern_flops[dom] / (dom_ms / max(dom_n, 1) * 1e-3) / 1e12 if dom_n else None
    peak = peaks["bf16_tflops"]
    kernel_names = {"fwd": "fa_fwd_kernel", "bwd_main": "fa_bwd_kernel"}
    traffic = load_traffic(kernel_names[dom], w.name)
    per = lambda k: (prof[k][0] / max(prof[k][1], 1)) if prof[k][1] else None
    fwd_ms, bwd_ms = per("fwd"), per("bwd_main")
    total_kernel_ms = sum(v[0] for v in prof.values())
    rows_all = w.B * w.H * w.S
    elt = 2 if w.dtype == "bf16" else 4
    pre_bytes = rows_all * (2 * w.d * elt + 4 + 4 * w.d)      # read O, dO; write D; zero dQacc
    conv_bytes = rows_all * w.d * (4 + elt)                    # read dQacc; write dq

    line = {
        "metric": "attention fwd+bwd TFLOP/s (bf16, causal)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {**workload_config(w, causal),
                   "l2": "flushed between timed steps (256 MiB write outside the events)",
                   "parallelism": f"replica per GPU x{world} (independent heads, no collective)"},
        "frac_of_peak": {"burst": value / peaks["bf16_tflops"],
                         "sustained": value / peaks["bf16_tflops_sustained"], "peaks": peaks["source"]},
        "kernels": {"fwd_ms": fwd_ms, "bwd_main_ms": bwd_ms,
                    "bwd_preprocess_ms": per("bwd_preprocess"), "dq_convert_ms": per("dq_convert"),
                    # HBM-bound helpers: algorithmic bytes over time against the measured copy rate.
                    "bwd_preprocess_gbs": (pre_bytes / (per("bwd_preprocess") * 1e-3) / 1e9) if per("bwd_preprocess") else None,
                    "dq_convert_gbs": (conv_bytes / (per("dq_convert") * 1e-3) / 1e9) if per("dq_convert") else None,
                    "hbm_peak_gbs": peaks["hbm_gbs"],
                    "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None,
                    **bwd_rates(f_fwd, prof),
                    "shares": {k: (v[0] / total_kernel_ms if total_kernel_ms else None) for k, v in prof.items()}},
        "roofline": {"kernel": kernel_names[dom], "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 burst"},
        "deterministic_bwd": {
            "api": "fa_bwd_deterministic (Algorithm 2's separate dQ loop, no atomics)",
            "ms_per_step": det_ms_per_step,
            "value": world * step_flops / (det_ms_per_step * 1e-3) / 1e12, "unit": "TFLOP/s",
            "dkdv_ms": (prof_det["bwd_main"][0] / prof_det["bwd_main"][1]) if prof_det["bwd_main"][1] else None,
            "dq_pass_ms": (prof_det["dq_pass"][0] / prof_det["dq_pass"][1]) if prof_det["dq_pass"][1] else None,
            "steps": det_steps},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "fa_fwd_bwd_host (host buffers)", "pipelining": f"steps rotate over {NR} streams"},
        "gpu_launches": int(round(launches_per_step * args.steps)),
    }
    if targets is not None:
        line["target_shapes"] = {
            "what": "causal bf16 B1 H16 at the sequence lengths and head dims the throughput target names; "
                    "fwd+bwd step timed like `value` (L2 flushed, 20 steps), fwd and bwd from the "
                    "library's per-kernel events; fractions of the measured bf16 peaks",
            "points": targets}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, n_sl, el, thr = cpu_oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{n_sl} whole (b,h) slices of {w.name}, cycling over its "
                                          f"{w.B * w.H}; fp64 fwd + standard bwd, {el:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def peak_memory_bytes(fn):
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    fn()
    torch.cuda.synchronize()
    return torch.cuda.max_memory_allocated() - base


def run_memory(args):
    """Peak device memory above the inputs of one fwd+bwd step: this library
    against the materialised computation (QK^T -> masked softmax -> PV in the
    storage dtype, PyTorch autograd), which holds S x S score tensors."""
    import exact_attention_fa2_gb300 as fa
    dev = torch.device("cuda", 0)
    fa.load_library()
    w = workload(args.workload)
    q, k, v, do = (t.to(dev) for t in make_inputs(w.B, w.H, w.S, w.d, w.dtype, w.seed, w.qkv_scale))

    def ours():
        o, lse = fa.fwd(q, k, v, True, w.scale)
        fa.bwd(q, k, v, o, do, lse, True, w.scale)

    def materialised():
        qq, kk, vv = (t.detach().requires_grad_() for t in (q, k, v))
        s_ = torch.matmul(qq, kk.transpose(-1, -2)) * w.scale
        mask = torch.ones(w.S, w.S, device=dev, dtype=torch.bool).triu(1)
        p_ = torch.softmax(s_.masked_fill(mask, float("-inf")), dim=-1)
        out = torch.matmul(p_, vv)
        out.backward(do)

    ours()
    fa.check_status()
    m_ours = peak_memory_bytes(ours)
    fa.check_status()
    m_mat = peak_memory_bytes(materialised)
    line = {"memory": {"workload": f"{w.name}: B{w.B} H{w.H} S{w.S} d{w.d} causal {w.dtype}",
                       "ours_peak_bytes": m_ours, "materialised_peak_bytes": m_mat,
                       "ratio": m_mat / max(m_ours, 1),
                       "what": "torch.cuda.max_memory_allocated above the resident inputs, one fwd+bwd"}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.memory:
            return run_memory(args)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
