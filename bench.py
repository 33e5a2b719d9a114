#!/usr/bin/env python3
"""Benchmark of the tiled-attention hot path on GB300 (one JSON line on rank 0).

A step is one pass of the whole path over one batch: fa_fwd (O, L) followed by
fa_bwd (Dlt/lse preprocess, the recompute-P backward kernel, dQ conversion) on
the multi-head LLM-shaped layer B=4, H=32, Nq=Nk=4096, D=128, causal, bf16
Q/K/V/dO ~ N(0,1)*0.5 from the seeded recipe.  FLOPs per step follow the
4*B*H*Nq*Nk*D forward convention (halved for causal) plus 2.5x that for the
backward.  Inputs (4 x 134 MB) exceed the 129 MB L2, so no flush is needed.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--no-cpu-baseline]

Multi-GPU: one process per GPU (torchrun); every rank runs the same per-GPU
workload (weak scaling, no collective on the data path); the step time is the
max over ranks and `value` the work of all ranks over it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s (bf16 causal H=32 N=4096 D=128), % of TC peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BWD_SOURCES = ["tiled_attention_11_gb300/csrc/bwd_sm103a.cu", "tiled_attention_11_gb300/csrc/ptx_sm103a.cuh",
               "tiled_attention_11_gb300/csrc/fa_kernels.h"]
FWD_SOURCES = ["tiled_attention_11_gb300/csrc/fwd_sm103a.cu", "tiled_attention_11_gb300/csrc/ptx_sm103a.cuh",
               "tiled_attention_11_gb300/csrc/fa_kernels.h"]


# ------------------------------------------------------------------ host helpers (CPU-testable)
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's step time."""
    return flops_per_step_per_rank * world / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def sources_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, sources) -> float | None:
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_sha") != sources_sha(sources):
        return None
    return float(d["dram_bytes_per_launch"])


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else the platform string)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self, gpu_index: int = 0):
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != 9:
                    continue
                try:
                    if int(parts[0]) != gpu_index:
                        continue
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        reasons = sorted({n for r in rows for n, v in zip(self.NAMES, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ CPU oracle timing
def oracle_sample(p, seconds_target: float, max_heads: int, seed: int = 0):
    """Time the fp64 oracle (fwd + bwd) on whole heads of the workload until about
    `seconds_target` of CPU work; returns (TFLOP/s by the path's convention, heads, seconds)."""
    import oracle
    from tiled_attention_11_gb300 import inputs as I
    q, k, v, do = I.draw(p, seed)
    per_head = (I.flops_fwd(p) + I.flops_bwd(p)) / (p.B * p.H)
    t_total, n = 0.0, 0
    while n < max_heads and (n == 0 or t_total < seconds_target):
        b, h = divmod(n % (p.B * p.H), p.H)
        qd, kd, vd, dod = (I.as_f64(t[b, h]) for t in (q, k, v, do))
        t0 = time.perf_counter()
        oracle.forward_head(qd, kd, vd, p.scale, p.causal)
        oracle.backward_head(qd, kd, vd, dod, p.scale, p.causal)
        t_total += time.perf_counter() - t0
        n += 1
    return per_head * n / t_total / 1e12, n, t_total


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    from tiled_attention_11_gb300 import _lib
    from tiled_attention_11_gb300 import inputs as I

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(_lib.LIB_PATH):
        if local == 0:
            from tiled_attention_11_gb300.build import build
            build()
        if world > 1:
            dist.barrier()
    _lib.lib()

    p = I.LAYER
    flops_fwd, flops_bwd = I.flops_fwd(p), I.flops_bwd(p)
    flops_step = flops_fwd + flops_bwd
    q, k, v, do = I.draw(p, seed=rank)
    pin = [t.pin_memory() for t in (q, k, v, do)]
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qg)
    lse = torch.empty((p.B, p.H, p.Nq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
    ws = torch.empty(_lib.fa_bwd_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D), dtype=torch.uint8, device=dev)

    def fwd():
        _lib.fa_fwd(qg, kg, vg, o, lse, p.causal, p.scale)

    def bwd():
        _lib.fa_bwd(qg, kg, vg, o, lse, dog, dq, dk, dv, p.causal, p.scale, workspace=ws)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()

    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    fb, fe, bb, be, mb, me = ([ev() for _ in range(K)] for _ in range(6))
    s = torch.cuda.current_stream()
    for e in fb + fe + bb + be + mb + me:
        e.record(s)  # create the underlying CUDA events before the timed region
    start, end = ev(), ev()
    torch.cuda.synchronize()

    clocks = ClockSampler()
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(s)
    for i in range(K):
        fb[i].record(s)
        fwd()
        fe[i].record(s)
        _lib.fa_set_bwd_main_events(mb[i], me[i])
        bb[i].record(s)
        bwd()
        be[i].record(s)
    end.record(s)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    _lib.fa_set_bwd_main_events(None, None)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = int(visible.split(",")[local]) if visible and visible.split(",")[local].isdigit() else local
    clk = clocks.stop(smi_index)

    ms_step = max_over_ranks(start.elapsed_time(end) / K, dev)
    fwd_ms = statistics.mean(fb[i].elapsed_time(fe[i]) for i in range(K))
    bwd_ms = statistics.mean(bb[i].elapsed_time(be[i]) for i in range(K))
    main_ms = statistics.mean(mb[i].elapsed_time(me[i]) for i in range(K))
    rc, site = _lib.fa_device_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} (wait site {site}) after the timed region")

    if args.no_e2e:  # (profiling runs: only the device-resident steps)
        if world > 1:
            dist.destroy_process_group()
        return
    # ---------------- end to end through fa_step_host: pinned host inputs -> device, fwd + bwd,
    # every output -> pinned host.  Several steps are in flight on their own streams (own
    # device buffer and host output set each), so copies overlap kernels and each other
    # (three measured best: 569 TFLOP/s against 463 with two, the same with four).
    del qg, kg, vg, dog, o, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()
    n_dev = _lib.step_host_device_bytes(p.B, p.H, p.Nq, p.Nk, p.D)
    lanes = []
    for _ in range(args.e2e_lanes):
        outs_host = [torch.empty(shape, dtype=dt, pin_memory=True)
                     for shape, dt in (((p.B, p.H, p.Nq, p.D), torch.bfloat16), ((p.B, p.H, p.Nq), torch.float32),
                                       ((p.B, p.H, p.Nq, p.D), torch.bfloat16), ((p.B, p.H, p.Nk, p.D), torch.bfloat16),
                                       ((p.B, p.H, p.Nk, p.D), torch.bfloat16))]
        lanes.append((torch.cuda.Stream(device=dev), torch.empty(n_dev, dtype=torch.uint8, device=dev), outs_host))
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in lanes[0][2])

    def host_step(i):
        st, buf, outs = lanes[i % len(lanes)]
        _lib.step_host(*pin, *outs, buf, p.causal, p.scale, stream=st)

    for i in range(len(lanes)):  # warm-up of every lane
        host_step(i)
    torch.cuda.synchronize()
    K2 = max(len(lanes), min(K, args.e2e_steps))
    if world > 1:
        dist.barrier()
    e2e_s, e2e_e = ev(), ev()
    e2e_s.record(s)
    for st, _, _ in lanes:
        st.wait_event(e2e_s)
    for i in range(K2):
        host_step(i)
    for st, _, _ in lanes:
        s.wait_stream(st)
    e2e_e.record(s)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e2e_ms = max_over_ranks(e2e_s.elapsed_time(e2e_e) / K2, dev)
    # the host link's own rates (pinned buffers of the step's size, copy engines, best of 5):
    # no step can move its inputs in and its outputs out faster than both directions at once
    del lanes
    torch.cuda.empty_cache()
    link = link_rates(dev, h2d)
    e2e_floor_ms = max(h2d, d2h) / (link["both_gbs"] * 1e9) * 1e3

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    timed_s = ms_step * K * 1e-3
    fwd_tf = flops_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = flops_bwd / (bwd_ms * 1e-3) / 1e12
    main_tf = flops_bwd / (main_ms * 1e-3) / 1e12
    if main_ms >= fwd_ms:
        dom, dom_ms, dom_flops, dom_src = "fa_bwd main kernel (bwd_persist_kernel<128,causal>)", main_ms, flops_bwd, BWD_SOURCES
        traffic = traffic_for("bwd_main_layer", BWD_SOURCES)
    else:
        dom, dom_ms, dom_flops, dom_src = "fa_fwd kernel (fwd_persist_kernel<128,causal>)", fwd_ms, flops_fwd, FWD_SOURCES
        traffic = traffic_for("fwd_layer", FWD_SOURCES)
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12

    out = {
        "metric": METRIC,
        "value": round(job_throughput(flops_step, world, ms_step), 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)*0.5 bf16 Q/K/V/dO; no dataset)",
        "config": {"workload": "multi-head LLM-shaped attention layer fwd+bwd: B=4 H=32 Nq=Nk=4096 D=128 causal",
                   "B": p.B, "H": p.H, "Nq": p.Nq, "Nk": p.Nk, "D": p.D, "causal": True,
                   "flops_per_step": flops_step, "l2": "inputs larger than L2 (Q,K,V,dO = 537 MB), no flush"},
        "fwd": {"ms": round(fwd_ms, 4), "tflops": round(fwd_tf, 1), "pct_peak": round(100 * fwd_tf / burst, 1)},
        "bwd": {"ms": round(bwd_ms, 4), "tflops": round(bwd_tf, 1), "pct_peak": round(100 * bwd_tf / burst, 1),
                "main_kernel_ms": round(main_ms, 4), "main_kernel_tflops": round(main_tf, 1),
                "main_kernel_pct_peak": round(100 * main_tf / burst, 1)},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": burst, "unit": "TFLOP/s", "frac": round(achieved / burst, 4),
                     "peak_kind": f"bf16_tflops, burst ({peak_src}): the timed region lasts {timed_s:.2f} s, "
                                  "far from the seconds-long power-capped loop of the sustained figure",
                     "frac_of_sustained": round(achieved / sustained, 4),
                     "traffic": traffic, "algorithmic_flops_per_launch": dom_flops},
        "e2e": {"value": round(job_throughput(flops_step, world, e2e_ms), 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "steps": K2, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": f"fa_step_host (pinned host buffers), {args.e2e_lanes} steps in flight on {args.e2e_lanes} streams",
                "link_gbs": link, "floor_ms": round(e2e_floor_ms, 4),
                "frac_of_floor": round(e2e_floor_ms / e2e_ms, 4)},
        "gpu_launches": 4 * K,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        val, n, secs = oracle_sample(p, args.cpu_seconds, max_heads=p.B * p.H)
        out["cpu_baseline"] = {"value": round(val, 6), "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                               "cpu_model": cpu_model(),
                               "sample": f"fp64 numpy oracle fwd+bwd on {n} whole head(s) of the workload "
                                         f"({secs:.1f} s of CPU work), FLOPs by the same convention"}
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def link_rates(dev, nbytes: int) -> dict:
    """Host <-> device copy rates (GB/s) for pinned buffers of nbytes: host to device,
    device to host, and each direction while both run at once (two streams)."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def best(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            fn()
            e1.record(s1)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return min(ts)

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s1):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        s2.wait_stream(s1)
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)
        s1.wait_stream(s2)

    r = {k: round(nbytes / (best(f) * 1e-3) / 1e9, 1) for k, f in (("h2d_gbs", h2d), ("d2h_gbs", d2h),
                                                                 ("both_gbs", both))}
    del h_in, h_out, d_in, d_out
    torch.cuda.empty_cache()
    return r


# ------------------------------------------------------------------ per-workload table
def run_table(args):
    """Time fa_fwd and fa_bwd on every workload (median of `--steps` reps after 3
    warm-ups); shapes whose inputs fit in L2 get an L2 flush (a 256 MB write)
    before every timed call.  Prints one markdown row per workload."""
    import torch
    from tiled_attention_11_gb300 import _lib
    from tiled_attention_11_gb300 import inputs as I

    dev = torch.device("cuda", 0)
    _lib.lib()
    peaks, _ = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    dense_rows = not (args.varlen_only or args.window_only or args.fp8_only)
    ex2 = 0.0
    if dense_rows:
        from tiled_attention_11_gb300 import probe
        probe.lib()
        ex2 = probe.ex2_rate(dev)
        print(f"exp2 roof (special-function units, measurement library): {ex2 / 1e12:.2f} T exp2/s; "
              f"tensor roof for the score GEMM's UMMA shape: {probe.umma_rate(dev) / 1e12:.0f} "
              f"TFLOP/s at the running clock; % peak columns use the measured burst cuBLAS bf16 peak "
              f"{peak:.1f} TFLOP/s")
    print("| workload | fwd ms | fwd TFLOP/s | fwd % peak | bwd ms | bwd TFLOP/s | bwd % peak | fwd GB/s (% HBM) "
          "| step ms direct / CUDA graph | L2 flush | exp2 % of roof fwd / bwd |")
    print("|---|---|---|---|---|---|---|---|---|---|---|")
    for p in (I.SWEEP + I.SWEEP_X8[-2:] + I.LONG + [I.LAYER, I.LONG_RAGGED] if dense_rows else []):
        if args.only and p.name() != args.only:
            continue
        q, k, v, do = (t.to(dev) for t in I.draw(p, 0))
        o = torch.empty_like(q)
        lse = torch.empty((p.B, p.H, p.Nq), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(_lib.fa_bwd_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D), 256), dtype=torch.uint8,
                         device=dev)
        in_bytes = 2 * p.D * p.B * p.H * (2 * p.Nq + 2 * p.Nk) + 4 * p.B * p.H * p.Nq
        small = 4 * q.numel() * 2 < (129 << 20)
        fwd = lambda: _lib.fa_fwd(q, k, v, o, lse, p.causal, p.scale)  # noqa: E731
        bwd = lambda: _lib.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, p.causal, p.scale, workspace=ws)  # noqa: E731
        res = []
        for fn in (fwd, bwd):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(args.steps):
                if small:
                    flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            res.append(statistics.median(ts))
        # whole step (fwd + bwd) as direct calls and as a CUDA graph replay
        graph = _lib.StepGraph(q, k, v, o, lse, do, dq, dk, dv, p.causal, p.scale, workspace=ws)
        steps = []
        for fn in (lambda: (fwd(), bwd()), graph.launch):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(args.steps):
                if small:
                    flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            steps.append(statistics.median(ts))
        graph.close()
        ff, fb = I.flops_fwd(p), I.flops_bwd(p)
        tf, tb = ff / res[0] / 1e9, fb / res[1] / 1e9
        gbs = in_bytes / res[0] / 1e6
        exps = ff / (4.0 * p.D)  # one exp2 per unmasked score in each pass (same causal convention)
        xf, xb = 100 * exps / (res[0] * 1e-3) / ex2, 100 * exps / (res[1] * 1e-3) / ex2
        print(f"| {p.name()} | {res[0]:.4f} | {tf:.1f} | {100 * tf / peak:.1f}% | {res[1]:.4f} | {tb:.1f} | "
              f"{100 * tb / peak:.1f}% | {gbs:.0f} ({100 * gbs / hbm:.1f}%) | {steps[0]:.4f} / {steps[1]:.4f} "
              f"| {'yes' if small else 'no'} | {xf:.1f}% / {xb:.1f}% |", flush=True)
        del q, k, v, do, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
    if args.only:
        return
    if args.fp8_only:
        _table_fp8(args, dev, peak, hbm)
        return
    if not args.window_only:
        _table_varlen(args, dev, peak, hbm)
    if not args.varlen_only:
        _table_window(args, dev, peak)
    if not (args.window_only or args.varlen_only):
        _table_fp8(args, dev, peak, hbm)


def window_pairs(Nq: int, Nk: int, causal: bool, window_left: int, window_right: int, n_global: int) -> int:
    """(query, key) pairs the local-window + global-token mask allows, row by row in closed
    form: a global row sees every key up to its last visible one (hi); another row sees its
    window [wlo, whi] plus the global keys [0, g) not already in it, all clipped to hi."""
    import numpy as np
    i = np.arange(Nq, dtype=np.int64)
    hi = np.full(Nq, Nk - 1, np.int64)
    if causal:
        hi = np.minimum(hi, i)
    wlo = np.zeros(Nq, np.int64) if window_left < 0 else np.maximum(i - window_left, 0)
    whi = hi if window_right < 0 else np.minimum(hi, i + window_right)
    win = np.maximum(whi - wlo + 1, 0)
    a = np.minimum(min(n_global, Nk) - 1, hi)                 # last global key a row may see
    overlap = np.maximum(np.minimum(a, whi) - wlo + 1, 0)
    cnt = win + np.maximum(a + 1, 0) - overlap
    cnt = np.where(i < n_global, hi + 1, cnt)
    return int(np.maximum(cnt, 0).sum())


# Local-window workloads of --table: (B, H, N, D, causal, window_left, window_right, n_global)
WINDOW_TABLE = [(1, 32, 32768, 128, True, 4096, -1, 0), (1, 32, 32768, 128, True, 1024, -1, 64),
                (1, 16, 65536, 64, False, 512, 512, 128)]


def _table_window(args, dev, peak):
    """Local-window + global-token rows: FLOPs count only the allowed (query, key) pairs."""
    import torch
    from tiled_attention_11_gb300 import _lib
    from tiled_attention_11_gb300 import inputs as I

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for (B, H, N, D, causal, wl, wr, g) in WINDOW_TABLE:
        p = I.Problem(B, H, N, N, D, causal, factor=0.5)
        q, k, v, do = (t.to(dev) for t in I.draw(p, 0))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(_lib.fa_bwd_window_workspace_size(B, H, N, N, D, wl, wr, g), dtype=torch.uint8, device=dev)
        fws = torch.empty(max(_lib.fa_fwd_window_workspace_size(B, H, N, N, D, causal, wl, wr, g), 256),
                          dtype=torch.uint8, device=dev)
        fwd = lambda: _lib.fa_fwd_window(q, k, v, o, lse, causal, wl, wr, g, p.scale, workspace=fws)  # noqa: E731
        bwd = lambda: _lib.fa_bwd_window(q, k, v, o, lse, do, dq, dk, dv, causal, wl, wr, g, p.scale,  # noqa: E731
                                         workspace=ws)
        res = []
        for fn in (fwd, bwd, lambda: (fwd(), bwd())):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(args.steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            res.append(statistics.median(ts))
        ff = 4.0 * B * H * D * window_pairs(N, N, causal, wl, wr, g)
        tf, tb = ff / res[0] / 1e9, 2.5 * ff / res[1] / 1e9
        gbs = (2 * D * B * H * 4 * N + 4 * B * H * N) / res[0] / 1e6
        name = f"window B{B}H{H}N{N}D{D}{'c' if causal else 'n'} wl{wl} wr{wr} g{g}"
        print(f"| {name} | {res[0]:.4f} | {tf:.1f} | {100 * tf / peak:.1f}% | {res[1]:.4f} | {tb:.1f} | "
              f"{100 * tb / peak:.1f}% | {gbs:.0f} | {res[2]:.4f} / - | yes |", flush=True)
        del q, k, v, do, o, lse, dq, dk, dv, ws, fws
        torch.cuda.empty_cache()


def _table_fp8(args, dev, peak, hbm):
    """FP8 forward rows: the e4m3 kernel alone (inputs quantised once), and the three
    per-tensor quantisations; % of the e4m3 dense peak = 2 x the measured bf16 peak (the
    nominal fp8 / bf16 ratio)."""
    import torch
    from tiled_attention_11_gb300 import _lib
    from tiled_attention_11_gb300 import inputs as I

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for p in (I.LAYER, I.Problem(8, 1, 16384, 16384, 128, True), I.Problem(1, 8, 65537, 65537, 128, True)):
        q, k, v, _ = (t.to(dev) for t in I.draw(p, 0))
        q8, _, qd = _lib.quantize_e4m3(q)
        k8, _, kd = _lib.quantize_e4m3(k)
        vt8, ldv, _, vd = _lib.quantize_e4m3_transposed(v)
        o = torch.empty_like(q)
        lse = torch.empty((p.B, p.H, p.Nq), dtype=torch.float32, device=dev)
        fwd = lambda: _lib.fa_fwd_fp8(q8, k8, vt8, ldv, qd, kd, vd, o, lse, p.causal, p.scale)  # noqa: E731
        quant = lambda: _lib.quantize_qkv_e4m3(q, k, v)  # noqa: E731
        quant3 = lambda: (_lib.quantize_e4m3(q), _lib.quantize_e4m3(k), _lib.quantize_e4m3_transposed(v))  # noqa: E731
        res = []
        for fn in (fwd, quant, quant3):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(args.steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            res.append(statistics.median(ts))
        tf = I.flops_fwd(p) / res[0] / 1e9
        qbytes = 3 * q.numel() * (2 + 2 + 1)  # amax read, quantise read + 1-byte write, per tensor
        print(f"| fp8 fwd {p.name()} | {res[0]:.4f} | {tf:.1f} | {100 * tf / (2 * peak):.1f}% of e4m3 | "
              f"quantise q,k,v {res[1]:.4f} ms ({qbytes / res[1] / 1e6:.0f} GB/s, {100 * qbytes / res[1] / 1e6 / hbm:.0f}% HBM; "
              f"three separate calls {res[2]:.4f} ms) |",
              flush=True)
        del q, k, v, q8, k8, vt8, o, lse
        torch.cuda.empty_cache()


def _table_varlen(args, dev, peak, hbm):
    """Packed variable-length row: fa_fwd_varlen / fa_bwd_varlen on the document mix."""
    import torch
    from tiled_attention_11_gb300 import _lib
    from tiled_attention_11_gb300 import inputs as I

    w = I.VARLEN_DOCS
    lens, H, D, causal = w["lens"], w["H"], w["D"], w["causal"]
    q, k, v, do, cu_q, cu_k = I.draw_varlen(lens, lens, H, D, 0, w["factor"])
    q, k, v, do, cu_q, cu_k = (t.to(dev) for t in (q, k, v, do, cu_q, cu_k))
    total, mx = sum(lens), max(lens)
    scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_bwd_varlen_workspace_size(len(lens), H, total, mx, D), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    fwd = lambda: _lib.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, mx, mx, causal, scale)  # noqa: E731
    bwd = lambda: _lib.fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu_q, cu_k, mx, mx, causal, scale,  # noqa: E731
                                     workspace=ws)
    res = []
    for fn in (fwd, bwd, lambda: (fwd(), bwd())):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        res.append(statistics.median(ts))
    ff, fb = I.flops_varlen(lens, lens, H, D, causal), I.flops_varlen(lens, lens, H, D, causal, backward=True)
    tf, tb = ff / res[0] / 1e9, fb / res[1] / 1e9
    gbs = (2 * D * H * 4 * total + 4 * H * total) / res[0] / 1e6
    name = f"varlen docs {len(lens)} seqs, {total} tok (max {mx}) H{H}D{D}{'c' if causal else 'n'}"
    print(f"| {name} | {res[0]:.4f} | {tf:.1f} | {100 * tf / peak:.1f}% | {res[1]:.4f} | {tb:.1f} | "
          f"{100 * tb / peak:.1f}% | {gbs:.0f} ({100 * gbs / hbm:.1f}%) | {res[2]:.4f} / - | yes |", flush=True)


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args):
    from tiled_attention_11_gb300 import inputs as I
    import oracle

    rank, world, _ = dist_env()
    if rank != 0:
        return
    p = I.LAYER
    q, k, v, do = I.draw(p, 0)
    per_head = (I.flops_fwd(p) + I.flops_bwd(p)) / (p.B * p.H)

    def step(i):
        b, h = divmod(i % (p.B * p.H), p.H)
        qd, kd, vd, dod = (I.as_f64(t[b, h]) for t in (q, k, v, do))
        oracle.forward_head(qd, kd, vd, p.scale, p.causal)
        oracle.backward_head(qd, kd, vd, dod, p.scale, p.causal)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    secs = time.perf_counter() - t0
    ms = secs * 1e3 / args.steps
    val = per_head / (ms * 1e-3) / 1e12
    cores = blas_threads()
    sample = "fp64 numpy oracle fwd+bwd on one whole head of the workload per step"
    out = {
        "metric": METRIC, "value": round(val, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1)*0.5 bf16 Q/K/V/dO; no dataset)",
        "impl": "reference",
        "config": {"workload": "multi-head LLM-shaped attention layer fwd+bwd: B=4 H=32 Nq=Nk=4096 D=128 causal",
                   "B": p.B, "H": p.H, "Nq": p.Nq, "Nk": p.Nk, "D": p.D, "causal": True,
                   "sample": "one head (1/128 of the layer) per step"},
        "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-lanes", type=int, default=3, help="steps in flight in the end-to-end measurement")
    ap.add_argument("--no-e2e", action="store_true",
                    help="stop after the device-resident steps, printing nothing (for profiler captures)")
    ap.add_argument("--table", action="store_true", help="time every workload, print a markdown table")
    ap.add_argument("--varlen-only", action="store_true", help="with --table: only the packed variable-length row")
    ap.add_argument("--window-only", action="store_true", help="with --table: only the local-window rows")
    ap.add_argument("--only", default="", help="with --table: only the dense row of this workload name "
                                               "(e.g. B8H1q256k256D16n)")
    ap.add_argument("--fp8-only", action="store_true", help="with --table: only the FP8 forward rows")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.table:
        run_table(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
