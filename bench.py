#!/usr/bin/env python3
"""Benchmark: ring-allreduce gradient sync of N logical ranks on one GB300.

    python bench.py [--gpus G] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: N = 8 logical ranks, one 1 GiB fp32 bucket per rank
(268,435,456 elements, N(0, 1e-2^2) from seed r), ring allreduce divided by
8.  A step is one ring_allreduce_fused call over the resident bucket (the
bucket is the rank's whole gradient vector, so the pack and unpack copies
are identities here; the bucketed DDP step with pack/unpack is timed on the
355M-parameter decoder and reported under "ddp_step").

Prints ONE JSON line.  value = bus bandwidth 2(N-1)/N * S_bytes / t summed
over GPUs (GB/s, 1e9 B/s); roofline.achieved = algorithmic HBM bytes
2*N*S_bytes per launch / average launch time.  With G > 1 (torchrun, one
process per GPU) each GPU runs an independent replica of the workload
(the N logical ranks never span GPUs); time is the max over GPUs.

--impl reference times the CPU oracle (the plain ring simulation) on a
bounded sample of the same workload on the host cores, as the comparison arm.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ring allreduce busbw GB/s and achieved HBM GB/s vs peak, N logical ranks, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
N_RANKS = 8
NUMEL = 1 << 28
MiB = 1 << 20


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_digest() -> str:
    h = hashlib.sha256()
    for f in ("ring_kernels.cu", "ddp_device.cuh", "ddp_internal.h"):       # the headline kernel's sources
        with open(os.path.join(ROOT, "gradient_sync_plan_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(name: str):
    """DRAM bytes per full-size launch recorded from an ncu capture in the data
    file profiles/<name> (JSON), or None if absent or taken on a different
    version of the kernel sources."""
    p = os.path.join(ROOT, "profiles", name)
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, None
    if d.get("kernel_sources_digest") != kernel_sources_digest():
        return None, p
    v = d.get("traffic_bytes_per_full_launch")
    return (float(v) if v is not None else None), p


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-i", str(self.gpu_index), "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark_start(self):
        self.t0 = _dt.datetime.now()

    def mark_end(self):
        self.t1 = _dt.datetime.now()

    def stop(self):
        time.sleep(0.15)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if self.t0 and self.t1 and self.t0 <= ts <= self.t1]
        use = inside if inside else [p for _, p in rows]

        def num(s):
            m = re.match(r"([0-9.]+)", s)
            return float(m.group(1)) if m else None

        sm = sorted(v for v in (num(p[2]) for p in use) if v is not None)
        mx = [v for v in (num(p[3]) for p in use) if v is not None]
        reasons = set()
        for p in use:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max((num(p[4]) or 0.0) for p in use) if use else None}


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    management library, loaded with ctypes) every `period_s` seconds while the
    timed region runs; reading only, no setting is changed.  Falls back to
    nvidia-smi when NVML cannot be loaded."""

    # clock-event reason bits of NVML's public API
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str, gpu_index: int, period_s: float = 0.005):
        self.uuid, self.gpu_index, self.period_s = uuid, gpu_index, period_s
        self.samples = []            # (t, sm_mhz, max_mhz, power_w, reasons)
        self.t0 = self.t1 = None
        self._stop = threading.Event()
        self._thread = None
        self._fallback = None

    def _open(self):
        import ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        rc = L.nvmlDeviceGetHandleByUUID(("GPU-" + self.uuid).encode(), ctypes.byref(h))
        if rc != 0:
            rc = L.nvmlDeviceGetHandleByIndex_v2(self.gpu_index, ctypes.byref(h))
        if rc != 0:
            raise OSError("no NVML handle")
        reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons
        return L, h, reasons_fn

    def start(self):
        try:
            L, h, reasons_fn = self._open()
        except Exception:
            self._fallback = ClockSampler(self.gpu_index)
            self._fallback.start()
            return
        import ctypes

        def loop():
            sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            while not self._stop.is_set():
                ok = (L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and
                      L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0)
                if L.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) != 0:
                    pw.value = 0
                if reasons_fn(h, ctypes.byref(rs)) != 0:
                    rs.value = 0
                if ok:
                    self.samples.append((time.perf_counter(), sm.value, mx.value, pw.value / 1000.0, rs.value))
                time.sleep(self.period_s)
            L.nvmlShutdown()

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        time.sleep(0.05)

    def mark_start(self):
        self.t0 = time.perf_counter()
        if self._fallback:
            self._fallback.mark_start()

    def mark_end(self):
        self.t1 = time.perf_counter()
        if self._fallback:
            self._fallback.mark_end()

    def stop(self):
        if self._fallback:
            self._fallback.stop()
            return
        time.sleep(0.02)
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=2)

    def summary(self):
        if self._fallback:
            return self._fallback.summary()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "no NVML samples"}
        inside = [x for x in self.samples if self.t0 is not None and self.t0 <= x[0] <= self.t1]
        use = inside if inside else self.samples
        sm = sorted(x[1] for x in use)
        reasons = sorted({name for x in use for bit, name in self.REASONS.items() if x[4] & bit})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(x[2] for x in use), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside), "period_ms": self.period_s * 1e3,
                "power_w_max": max(x[3] for x in use), "source": "NVML (ctypes), read-only"}


def run_metadata(torch, dev, n_ranks: int) -> dict:
    """What the line was measured on and with: GPU, host CPU, input seeds."""
    props = torch.cuda.get_device_properties(dev)
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    import platform
    return {"gpu": {"name": torch.cuda.get_device_name(dev), "uuid": str(getattr(props, "uuid", "")),
                    "sms": props.multi_processor_count, "memory_gib": round(props.total_memory / 2**30, 1),
                    "cc": f"{props.major}.{props.minor}"},
            "host": {"nproc": os.cpu_count(), "cores_available": host_cores(), "cpu_model": model,
                     "arch": platform.machine()},
            "inputs": {"generator": "torch.Generator(device='cuda').manual_seed(seed), torch.randn float32 * 1e-2",
                       "seeds": list(range(n_ranks)), "seed_rule": "rank r draws from seed r"},
            "torch": torch.__version__}


def host_link_bench(torch, dev, host_src, dev_dst, host_dst, dev_src, reps: int = 3) -> dict:
    """The CPU-GPU link's own throughput through the copy engines: pinned
    host -> device alone, device -> pinned host alone, and both at once on two
    streams (CUDA events around each), best of `reps`."""
    nbytes = host_src.numel() * host_src.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cur = torch.cuda.current_stream(dev)

    def timed(both, h2d=True):
        best = None
        for _ in range(reps):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            torch.cuda.synchronize(dev)
            e0.record(cur)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
            if both or h2d:
                with torch.cuda.stream(s_in):
                    dev_dst.copy_(host_src, non_blocking=True)
            if both or not h2d:
                with torch.cuda.stream(s_out):
                    host_dst.copy_(dev_src, non_blocking=True)
            e1.record(s_in)
            e2.record(s_out)
            cur.wait_event(e1)
            cur.wait_event(e2)
            torch.cuda.synchronize(dev)
            ms = max(e0.elapsed_time(e1), e0.elapsed_time(e2))
            best = ms if best is None else min(best, ms)
        return best

    h2d = timed(False, True)
    d2h = timed(False, False)
    both = timed(True)
    return {"bytes_each_way": nbytes, "h2d_gbs": nbytes / (h2d / 1e3) / 1e9, "d2h_gbs": nbytes / (d2h / 1e3) / 1e9,
            "both_gbs": 2 * nbytes / (both / 1e3) / 1e9, "both_ms": both,
            "how": "pinned host memory, copy engines, both directions on two streams at once, CUDA events, "
                   f"best of {reps}"}


def cpu_oracle_run(n_ranks: int, budget_s: float, max_numel: int, reps_cap: int = 1000):
    """Time the CPU oracle's ring on a bounded sample; returns a dict."""
    import numpy as np
    import oracle
    import workloads
    oracle.build()
    # calibrate on a small sample, then size the sample to the budget
    cal = 1 << 18
    x = workloads.rank_vectors(n_ranks, cal, "randn", std=1e-2).numpy()
    rows = [x[r] for r in range(n_ranks)]
    t = time.perf_counter()
    oracle.ring_allreduce(rows, oracle.F32, n_ranks)
    per_elem = max((time.perf_counter() - t) / cal, 1e-10)
    numel = int(min(max_numel, max(1 << 16, budget_s / 3.0 / per_elem)))
    numel = 1 << int(math.log2(numel))
    x = workloads.rank_vectors(n_ranks, numel, "randn", std=1e-2).numpy()
    rows = [x[r] for r in range(n_ranks)]
    times = []
    t_start = time.perf_counter()
    while len(times) < reps_cap and (time.perf_counter() - t_start) < budget_s:
        t = time.perf_counter()
        oracle.ring_allreduce(rows, oracle.F32, n_ranks)
        times.append(time.perf_counter() - t)
    tm = sorted(times)[len(times) // 2]
    s_bytes = numel * 4
    return {"numel": numel, "reps": len(times), "median_s": tm, "total_s": sum(times),
            "busbw_gbs": 2 * (n_ranks - 1) / n_ranks * s_bytes / tm / 1e9,
            "hbm_equiv_gbs": 2 * n_ranks * s_bytes / tm / 1e9}


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# --------------------------------------------------------------------------

def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    import numpy as np
    import oracle
    import workloads
    oracle.build()
    # per-step sample sized so that warmup + steps fit in about two minutes
    cal = 1 << 18
    x = workloads.rank_vectors(N_RANKS, cal, "randn", std=1e-2).numpy()
    rows = [x[r] for r in range(N_RANKS)]
    t = time.perf_counter()
    oracle.ring_allreduce(rows, oracle.F32, N_RANKS)
    per_elem = max((time.perf_counter() - t) / cal, 1e-10)
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    numel = int(min(args.numel, max(1 << 12, budget / per_elem)))
    numel = 1 << int(math.log2(numel))
    x = workloads.rank_vectors(N_RANKS, numel, "randn", std=1e-2).numpy()
    rows = [x[r] for r in range(N_RANKS)]
    for _ in range(args.warmup):
        oracle.ring_allreduce(rows, oracle.F32, N_RANKS)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.ring_allreduce(rows, oracle.F32, N_RANKS)
    dt = time.perf_counter() - t0
    s_bytes = numel * 4
    value = 2 * (N_RANKS - 1) / N_RANKS * s_bytes * args.steps / dt / 1e9
    part = "the whole" if numel == args.numel else "a bounded sample of the"
    sample = (f"N={N_RANKS} ranks x {numel} fp32 per rank ({s_bytes / MiB:.2f} MiB) per step, {part} "
              f"{args.numel * 4 / MiB:.0f} MiB-per-rank bucket; single-threaded C oracle")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": f"N={N_RANKS} logical ranks, one fp32 bucket of {args.numel} elements "
                                  f"({args.numel * 4 / MiB:.0f} MiB) per rank, fused ring allreduce / {N_RANKS}",
                      "ranks": N_RANKS, "numel": args.numel, "bucket_bytes": args.numel * 4,
                      "algorithm": "CPU oracle ring simulation", "sample_numel": numel,
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist
    import gradient_sync_plan_gb300 as ddp
    import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ddp.lib()
    numel = args.numel
    N = N_RANKS
    s_bytes = numel * 4
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    x = torch.empty((N, numel), dtype=torch.float32, device=dev)
    for r in range(N):
        x[r].copy_(workloads.randn_f32(numel, r, 1e-2, device=str(dev)))
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        ddp.ring_allreduce_fused(x, N)
    torch.cuda.synchronize()

    sampler = None
    if rank == 0 and not args.no_clocks:
        phys = local_rank
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            try:
                phys = int(vis.split(",")[local_rank])
            except Exception:
                phys = local_rank
        sampler = NvmlSampler(str(getattr(torch.cuda.get_device_properties(dev), "uuid", "")), phys)
        sampler.start()

    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    # one event after every step as well: the per-step distribution (median,
    # p90) beside the whole-region mean; recording events adds no device work
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev0.record(stream)
    for i in range(args.steps):
        ddp.ring_allreduce_fused(x, N)
        step_ev[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    per_step = sorted([ev0.elapsed_time(step_ev[0])] +
                      [step_ev[i - 1].elapsed_time(step_ev[i]) for i in range(1, args.steps)])
    step_median = per_step[len(per_step) // 2]
    step_p90 = per_step[min(len(per_step) - 1, (len(per_step) * 9) // 10)]
    if sampler:
        sampler.stop()
    ms_step = ms / args.steps
    busbw_total = world * 2 * (N - 1) / N * s_bytes * args.steps / (ms / 1e3) / 1e9
    hbm = 2 * N * s_bytes / (ms_step / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    traffic, traffic_src = profiled_traffic("ring_fused_n8_1gib.json")
    if traffic is not None and numel != NUMEL:
        traffic = traffic * numel / NUMEL

    out = {"metric": METRIC, "value": busbw_total, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_median": step_median,
           "ms_per_step_p90": step_p90, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": f"N={N} logical ranks, one fp32 bucket of {numel} elements "
                                  f"({s_bytes / MiB:.0f} MiB) per rank, fused ring allreduce / {N}",
                      "ranks": N, "numel": numel, "bucket_bytes": s_bytes, "algorithm": "ring_allreduce_fused",
                      "l2": f"inputs {N * s_bytes / 2**30:.2f} GiB per step, larger than L2; no flush",
                      "parallelism": "replicas" if world > 1 else "single GPU"},
           "algbw_gbs": s_bytes / (ms_step / 1e3) / 1e9,
           "hbm_gbs": hbm,
           "hbm_frac_of_nominal_8tbs": hbm / NOMINAL_HBM_GBS,
           "roofline": {"bound": "hbm", "achieved": hbm, "peak": peak, "unit": "GB/s", "frac": hbm / peak,
                        "traffic": traffic, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                        if peak_kind == "measured" else "fallback 6.8 TB/s",
                        "kernel": "k_ring_fused (vector, one block per tile)",
                        "algorithmic_bytes_per_launch": 2 * N * s_bytes},
           "gpu_launches": args.steps}
    if sampler:
        out["clocks"] = sampler.summary()
    out["run"] = run_metadata(torch, dev, N)

    # ---- end to end through the C ABI with host buffers ----------------------
    if not args.no_e2e:
        host = torch.empty((N, numel), dtype=torch.float32).pin_memory()
        host.copy_(x)
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        def timed(fn, steps):
            fn()
            torch.cuda.synchronize()
            barrier()
            ev0.record(stream)
            for _ in range(steps):
                fn()
            ev1.record(stream)
            torch.cuda.synchronize()
            return max_over_ranks(ev0.elapsed_time(ev1), world, dev) / steps

        # the kernel reads the pinned host buffers and writes the result back
        # to them over the CPU-GPU link: both directions at once, no device copy
        d_ms = timed(lambda: ddp.ring_allreduce_fused_host_direct(host, host, N), e2e_steps)
        # copy engines: host -> device buffers, kernel, device -> host
        c_ms = timed(lambda: ddp.ring_allreduce_fused_from_host(host, host, x, N), e2e_steps)
        out["e2e"] = {"value": world * 2 * (N - 1) / N * s_bytes / (d_ms / 1e3) / 1e9, "unit": "GB/s",
                      "h2d_bytes_per_step": N * s_bytes, "d2h_bytes_per_step": N * s_bytes,
                      "steps": e2e_steps, "ms_per_step": d_ms,
                      "api": "ring_allreduce_fused_host_direct (pinned host buffers in and out; the kernel moves "
                             "the bytes over the CPU-GPU link)",
                      "host_link_gbs": 2 * N * s_bytes / (d_ms / 1e3) / 1e9}
        out["e2e_copy_engines"] = {"value": world * 2 * (N - 1) / N * s_bytes / (c_ms / 1e3) / 1e9, "unit": "GB/s",
                                   "ms_per_step": c_ms, "steps": e2e_steps,
                                   "api": "ring_allreduce_fused_from_host (pinned host buffers; 32 MiB pieces "
                                          "copied in, reduced and copied out on overlapping streams)"}
        out["e2e"]["gpu_launches"] = e2e_steps          # one fused kernel per direct call
        # the link's own ceiling, measured the same run: copy engines in both
        # directions at once over the same 8 GiB (a second pinned host buffer
        # and a second device buffer)
        host2 = torch.empty_like(host).pin_memory()
        dev2 = torch.empty_like(x)
        link = host_link_bench(torch, dev, host, dev2, host2, x)
        del dev2
        # the same link driven by a kernel's own loads and stores, as the
        # direct path drives it: one rank, so the "allreduce" is a copy of the
        # 8 GiB from one pinned buffer to the other, read and written at once
        flat_in, flat_out = host.view(1, -1), host2.view(1, -1)
        k_ms = timed(lambda: ddp.ring_allreduce_fused_host_direct(flat_in, flat_out, 0), e2e_steps)
        link["kernel_copy_gbs"] = 2 * N * s_bytes / (k_ms / 1e3) / 1e9
        link["kernel_copy_how"] = ("ring_allreduce_fused_host_direct with one rank of 8 GiB: the kernel reads one "
                                   "pinned buffer and writes another over the CPU-GPU link")
        del host2, flat_in, flat_out
        peak_link = max(link["both_gbs"], link["kernel_copy_gbs"])
        out["e2e"]["host_link_peak_gbs"] = peak_link
        out["e2e"]["host_link_frac"] = out["e2e"]["host_link_gbs"] / peak_link
        out["e2e"]["host_link"] = link
        del host

    # ---- extra measurements ------------------------------------------------
    if not args.no_extras:
        extra_steps = max(3, min(20, args.steps // 10))
        a = x
        for _ in range(max(3, args.warmup)):       # untimed: first calls set up the hop kernel's launch state
            ddp.ring_allreduce_staged(a, N)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(extra_steps):
            ddp.ring_allreduce_staged(a, N)
        ev1.record(stream)
        torch.cuda.synchronize()
        st_ms = ev0.elapsed_time(ev1) / extra_steps
        out["staged"] = {"ms_per_step": st_ms, "launches_per_step": 2 * (N - 1),
                         "busbw_gbs": 2 * (N - 1) / N * s_bytes / (st_ms / 1e3) / 1e9,
                         "hbm_alg_gbs": 5 * (N - 1) * s_bytes / (st_ms / 1e3) / 1e9,
                         "useful_gbs": 2 * N * s_bytes / (st_ms / 1e3) / 1e9}
        del a, x
        torch.cuda.empty_cache()
        out["ddp_step"] = ddp_step_bench(ddp, workloads, torch, dev, stream, extra_steps)
        out["ddp_step"]["overlap"] = overlap_bench(ddp, workloads, torch, dev, 5)

    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_oracle_run(N, args.cpu_budget, NUMEL)
        out["cpu_baseline"] = {"value": cpu["busbw_gbs"], "unit": "GB/s", "cores": 1, "kind": "oracle",
                               "sample": f"N={N} ranks x {cpu['numel']} fp32 per rank "
                                         f"({cpu['numel'] * 4 // MiB} MiB), {cpu['reps']} runs, median; "
                                         f"single-threaded C ring simulation on the host "
                                         f"({host_cores()} cores present)",
                               "median_s": cpu["median_s"]}
    if rank == 0:
        print(json.dumps(out), flush=True)


def ddp_step_bench(ddp, workloads, torch, dev, stream, steps):
    """The bucketed DDP step on the 355M-parameter decoder, N = 8, fp32."""
    numels = workloads.param_numels(workloads.decoder_param_shapes())
    N, total = N_RANKS, sum(numels)
    p_bytes = total * 4
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, MiB, 25 * MiB)
    g = torch.empty((N, total), dtype=torch.float32, device=dev)
    for r in range(N):
        g[r].copy_(workloads.randn_f32(total, r, 1e-2, device=str(dev)))
    offs = [0]
    for n in numels:
        offs.append(offs[-1] + n)
    views = [[g[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
    buckets = [[torch.empty(int(n), dtype=torch.float32, device=dev) for n in plan[2]] for _ in range(N)]
    res = {"workload": "decoder 24x1024, 292 tensors, 354,823,168 fp32 params, N=8, caps 1 MiB / 25 MiB",
           "buckets": int(len(plan[2])), "bucket_sizes_bytes_first_last": [int(plan[2][0]) * 4, int(plan[2][-1]) * 4]}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, algo, bytes_alg in (("fused", ddp.DDP_ALGO_FUSED, 6 * N * p_bytes),
                                  ("staged", ddp.DDP_ALGO_STAGED, (2 * N + 5 * (N - 1)) * p_bytes + 2 * N * p_bytes),
                                  ("view", ddp.DDP_ALGO_VIEW, 2 * N * p_bytes)):
        call = ddp.SyncCall(views, plan, None if algo == ddp.DDP_ALGO_VIEW else buckets, N, algo)
        for _ in range(2):
            call()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(steps):
            call()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        res[name] = {"ms_per_step": ms, "hbm_alg_gbs": bytes_alg / (ms / 1e3) / 1e9,
                     "grad_bytes_synced_gbs": N * p_bytes / (ms / 1e3) / 1e9}
    # bf16 compression hook: float32 grads -> bf16 buckets -> bf16 ring -> float32
    bk16 = [[torch.empty(int(n), dtype=torch.bfloat16, device=dev) for n in plan[2]] for _ in range(N)]
    call = ddp.SyncCall(views, plan, bk16, N, ddp.DDP_ALGO_BF16_HOOK)
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    # pack: read 4 + write 2, ring: 2 + 2, unpack: read 2 + write 4 bytes per element and rank
    res["bf16_hook"] = {"ms_per_step": ms, "hbm_alg_gbs": 16 * N * total / (ms / 1e3) / 1e9,
                        "grad_bytes_synced_gbs": N * p_bytes / (ms / 1e3) / 1e9}
    del bk16
    # the same hook fused into one pass over the float32 gradients
    call = ddp.SyncCall(views, plan, None, N, ddp.DDP_ALGO_BF16_HOOK_VIEW)
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    res["bf16_hook_view"] = {"ms_per_step": ms, "hbm_alg_gbs": 2 * N * p_bytes / (ms / 1e3) / 1e9,
                             "grad_bytes_synced_gbs": N * p_bytes / (ms / 1e3) / 1e9}
    # the fp16 compression hook, fused the same way
    call = ddp.SyncCall(views, plan, None, N, ddp.DDP_ALGO_FP16_HOOK_VIEW)
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    res["fp16_hook_view"] = {"ms_per_step": ms, "hbm_alg_gbs": 2 * N * p_bytes / (ms / 1e3) / 1e9,
                             "grad_bytes_synced_gbs": N * p_bytes / (ms / 1e3) / 1e9}
    # no_sync: 3 local accumulations of a micro-batch, then one sync (view)
    scratch = torch.empty_like(g)
    scratch.copy_(g)
    call = ddp.SyncCall(views, plan, None, N, ddp.DDP_ALGO_VIEW)
    ev0.record(stream)
    for _ in range(steps):
        for _m in range(3):
            ddp.ddp_grad_accumulate(g, scratch)
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    res["no_sync_4_micro_view"] = {"ms_per_step": ms,
                                   "hbm_alg_gbs": (3 * 3 * N * p_bytes + 2 * N * p_bytes) / (ms / 1e3) / 1e9,
                                   "allreduce_calls_per_step": int(len(plan[2]))}
    del g, scratch, buckets, views
    torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """Message-size sweep: 4 KiB .. 256 MiB per rank, fp32 U[-1,1), N = 8 and 64,
    fused vs staged.  Each point replays a CUDA graph of R back-to-back calls
    (so the host's call overhead is not timed); buffers below the L2 size stay
    resident between calls, which is the latency regime the sweep exposes.
    One JSON line per point."""
    import torch
    import gradient_sync_plan_gb300 as ddp
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ddp.lib()
    for N in (4, 8, 64):
        for k in range(17):
            S = 1024 << k
            s_bytes = S * 4
            x = torch.empty((N, S), dtype=torch.float32, device=dev)
            for r in range(N):
                x[r].copy_(workloads.uniform_pm1_f32(S, r, device=str(dev)))
            reps = int(max(2, min(200, (1 << 28) // (N * S))))
            row = {"sweep": "message size", "ranks": N, "bytes_per_rank": s_bytes, "reps_per_graph": reps}
            status = torch.zeros(2, dtype=torch.int32, device=dev)
            persistent = lambda b, d: ddp.ring_allreduce_persistent(b, d, status=status)   # noqa: E731
            for name, fn in (("fused", ddp.ring_allreduce_fused), ("staged", ddp.ring_allreduce_staged),
                             ("persistent", persistent), ("tree_fused", ddp.tree_allreduce_fused),
                             ("tree_staged", ddp.tree_allreduce_staged)):
                s = torch.cuda.Stream()
                with torch.cuda.stream(s):
                    for _ in range(3):
                        fn(x, N)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    for _ in range(reps):
                        fn(x, N)
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                best = None
                for _ in range(3):
                    e0.record()
                    g.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    t = e0.elapsed_time(e1) / reps
                    best = t if best is None else min(best, t)
                depth = (N - 1).bit_length()
                alg = {"fused": 2 * N * s_bytes, "tree_fused": 2 * N * s_bytes,
                       "tree_staged": 5 * (N - 1) * s_bytes}.get(name, 5 * (N - 1) * s_bytes)
                row[name] = {"us_per_call": best * 1e3, "busbw_gbs": 2 * (N - 1) / N * s_bytes / (best / 1e3) / 1e9,
                             "hbm_alg_gbs": alg / (best / 1e3) / 1e9,
                             "launches_per_call": {"staged": 2 * (N - 1), "tree_staged": 2 * depth}.get(name, 1)}
                if name == "persistent":
                    assert int(status[0]) == 0, "persistent ring reported a barrier timeout"
                del g
            print(json.dumps(row), flush=True)
            del x
            torch.cuda.empty_cache()


def overlap_bench(ddp, workloads, torch, dev, steps):
    """Backward/communication overlap on the decoder DDP step (N = 8, fp32).

    A synthetic backward walks the layers in reverse: per transformer block two
    bf16 GEMMs of 4096^3 on a compute stream (emulated layer backward), then
    ONE kernel writes the block's gradients on every rank (a fill of the
    block's [N, block numel] slice of the gradient arena: HBM traffic equal to
    the block's gradient bytes, as a weight-gradient GEMM's epilogue would
    write them).  Three timings:
      backward      -- the synthetic backward alone
      serial        -- backward, then ddp_sync_buckets (view fusion) on the same stream
      overlapped    -- backward with a ddp_reducer that syncs each bucket on a comm
                       stream as soon as its gradients are ready
    exposed_comm_ms = overlapped - backward (the communication tail left after overlap)."""
    shapes = workloads.decoder_param_shapes()
    numels = workloads.param_numels(shapes)
    N, total = N_RANKS, sum(numels)
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, MiB, 25 * MiB)
    g = torch.empty((N, total), dtype=torch.float32, device=dev)
    offs = [0]
    for n in numels:
        offs.append(offs[-1] + n)
    views = [[g[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
    A = torch.randn(4096, 4096, dtype=torch.bfloat16, device=dev)
    B = torch.randn(4096, 4096, dtype=torch.bfloat16, device=dev)
    C = torch.empty(4096, 4096, dtype=torch.bfloat16, device=dev)
    # parameters grouped by block, in backward order: lnf, block 23 .. block 0, wpe+wte
    groups = [[len(numels) - 1, len(numels) - 2]]
    for blk in range(23, -1, -1):
        first = 2 + 12 * blk
        groups.append(list(range(first + 11, first - 1, -1)))
    groups.append([1, 0])
    compute, comm = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # the same reducer on a high-priority stream: its CTAs are dispatched
    # ahead of queued backward CTAs whenever an SM frees up
    lo_prio, hi_prio = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") else (0, -1)
    comm_hi = torch.cuda.Stream(device=dev, priority=hi_prio)
    red = ddp.Reducer(views, plan, None, N, ddp.DDP_ALGO_VIEW, comm_stream=comm)
    red_hi = ddp.Reducer(views, plan, None, N, ddp.DDP_ALGO_VIEW, comm_stream=comm_hi)
    sync = ddp.SyncCall(views, plan, None, N, ddp.DDP_ALGO_VIEW)

    # each group's parameters are contiguous in the arena: one [N, span] slice
    spans = [(offs[min(grp)], offs[max(grp) + 1]) for grp in groups]

    def backward(reducer):
        with torch.cuda.stream(compute):
            for gi, grp in enumerate(groups):
                if 0 < gi <= 24:
                    torch.mm(A, B, out=C)
                    torch.mm(C, B, out=C)
                a, b = spans[gi]
                g[:, a:b].fill_(1e-3 * (gi + 1))          # one write-only kernel for the whole block
                if reducer is not None:
                    for p in grp:
                        reducer.mark_ready(p, compute)

    def timed(fn):
        # capture the whole pass (both streams) into a CUDA graph so that the
        # host's per-op launch cost is not what gets measured
        fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=compute):
            fn()
        graph.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = None
        replay_stream = torch.cuda.current_stream()      # graph.replay() runs here
        for _ in range(steps):
            torch.cuda.synchronize()
            ev0.record(replay_stream)
            graph.replay()
            ev1.record(replay_stream)
            torch.cuda.synchronize()
            t = ev0.elapsed_time(ev1)
            best = t if best is None else min(best, t)
        del graph
        return best

    def run_backward():
        backward(None)

    def run_serial():
        backward(None)
        sync(compute)

    def run_overlapped():
        red.prepare()
        backward(red)
        red.finalize(compute)

    def run_overlapped_hi():
        red_hi.prepare()
        backward(red_hi)
        red_hi.finalize(compute)

    t_b = timed(run_backward)
    res = {"backward_ms": t_b,
           "note": "synthetic backward: 2 bf16 GEMMs of 4096^3 per block, then one write-only kernel per block "
                   "for the block's gradients on all ranks, on a compute stream; view-fusion sync; "
                   "each pass captured as one CUDA graph (both streams) and replayed; best of %d; "
                   "max_ctas = CTA cap of the sync kernels (0 = fill the GPU)" % steps, "by_max_ctas": {}}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for cap in (0, sms // 2, sms // 4, sms // 8):
        prev = ddp.ddp_set_max_ctas(cap)
        try:
            t_s, t_o, t_h = timed(run_serial), timed(run_overlapped), timed(run_overlapped_hi)
        finally:
            ddp.ddp_set_max_ctas(prev)
        comm_ms = t_s - t_b
        res["by_max_ctas"][str(cap)] = {"serial_ms": t_s, "overlapped_ms": t_o, "comm_ms": comm_ms,
                                        "exposed_comm_ms": t_o - t_b,
                                        "hidden_fraction": (t_s - t_o) / comm_ms if comm_ms > 0 else None,
                                        "high_priority_comm": {
                                            "overlapped_ms": t_h, "exposed_comm_ms": t_h - t_b,
                                            "hidden_fraction": (t_s - t_h) / comm_ms if comm_ms > 0 else None}}
    # DDP's logging data for one plain (not graph-captured) overlapped pass:
    # every bucket's size and its sync time on the comm stream
    run_overlapped()
    torch.cuda.synchronize()
    times = red.bucket_times()
    res["buckets"] = {"bucket_sizes_bytes": [int(n) * 4 for n in plan[2]],
                      "sync_ms": [round(t, 4) for t in times],
                      "sync_ms_total": sum(times),
                      "note": "per-rank bucket bytes; comm-stream time of each bucket's view sync while the "
                              "synthetic backward runs beside it"}
    red.close()
    red_hi.close()
    del g, views
    torch.cuda.empty_cache()
    return res


def run_cap_sweep(args):
    """Bucket-cap sweep (the pages' 6/12/25/50 MB bucket-size sweep):
    the DDP step for ResNet-50 in bf16 at N = 16 (caps 5, 10, 25, 50 MiB) and
    for the 355M decoder in fp32 at N = 8 (caps 6, 12, 25, 50 MiB), first
    bucket 1 MiB, pack + fused ring + unpack vs the fused view path.  Ten
    steps run back to back per timing, as eager calls and as replays of a
    CUDA graph of one step.  One JSON line per point."""
    import torch
    import gradient_sync_plan_gb300 as ddp
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ddp.lib()
    for model, shapes, N, dtype, caps in (
            ("resnet50", workloads.resnet50_param_shapes(), 16, "bf16", (5, 10, 25, 50)),
            ("decoder355m", workloads.decoder_param_shapes(), 8, "f32", (6, 12, 25, 50))):
        numels = workloads.param_numels(shapes)
        total = sum(numels)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        es = 2 if dtype == "bf16" else 4
        g = torch.empty((N, total), dtype=tdt, device=dev)
        for r in range(N):
            g[r].copy_(workloads.randn_f32(total, r, 1e-2, device=str(dev)).to(tdt))
        offs = [0]
        for n in numels:
            offs.append(offs[-1] + n)
        views = [[g[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
        for cap in caps:
            plan = ddp.ddp_plan_buckets(numels, ddp.BF16 if dtype == "bf16" else ddp.F32, MiB, cap * MiB)
            buckets = [[torch.empty(int(n), dtype=tdt, device=dev) for n in plan[2]] for _ in range(N)]
            row = {"sweep": "bucket cap", "model": model, "ranks": N, "dtype": dtype, "cap_mib": cap,
                   "buckets": int(len(plan[2])), "grad_bytes_per_rank": total * es}
            for name, algo, per_elem in (("pack_fused_unpack", ddp.DDP_ALGO_FUSED, 6), ("view", ddp.DDP_ALGO_VIEW, 2)):
                call = ddp.SyncCall(views, plan, buckets if algo != ddp.DDP_ALGO_VIEW else None, N, algo)
                s = torch.cuda.Stream(device=dev)
                with torch.cuda.stream(s):
                    for _ in range(3):
                        call(s)
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    call(s)
                # steady state: R steps back to back between the events, as a
                # training loop issues them -- eager calls on one stream (each
                # kernel's launch overlaps the previous kernel's tail), and
                # graph replays (each replay starts after the previous one
                # ends); best of 5 each
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                R = 10

                def best_of(run):
                    run()
                    best = None
                    for _ in range(5):
                        torch.cuda.synchronize()
                        e0.record(s)
                        for _r in range(R):
                            run()
                        e1.record(s)
                        torch.cuda.synchronize()
                        t = e0.elapsed_time(e1) / R
                        best = t if best is None else min(best, t)
                    return best

                with torch.cuda.stream(s):
                    t_eager = best_of(lambda: call(s))
                    t_graph = best_of(graph.replay)
                row[name] = {"ms_per_step": t_eager, "hbm_alg_gbs": per_elem * N * total * es / (t_eager / 1e3) / 1e9,
                             "graph_ms_per_step": t_graph,
                             "timing": f"{R} steps back to back on one stream, eager calls (ms_per_step) and "
                                       f"graph replays (graph_ms_per_step), best of 5"}
                del graph
            print(json.dumps(row), flush=True)
            del buckets
            torch.cuda.empty_cache()
        del g, views
        torch.cuda.empty_cache()


def run_profile_view(args):
    """A small DDP step for profiling the fused view kernel: a decoder with
    --profile-layers blocks (d = 1024), N = 8 ranks, fp32, caps 1 / 25 MiB,
    ddp_sync_buckets with the view algorithm, --steps times.  Prints one JSON
    line (not a bench result)."""
    import torch
    import gradient_sync_plan_gb300 as ddp
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    numels = workloads.param_numels(workloads.decoder_param_shapes(n_layer=args.profile_layers))
    N, total = N_RANKS, sum(numels)
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, MiB, 25 * MiB)
    g = torch.empty((N, total), dtype=torch.float32, device=dev)
    for r in range(N):
        g[r].copy_(workloads.randn_f32(total, r, 1e-2, device=str(dev)))
    offs = [0]
    for n in numels:
        offs.append(offs[-1] + n)
    views = [[g[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
    call = ddp.SyncCall(views, plan, None, N, ddp.DDP_ALGO_VIEW)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    print(json.dumps({"profile": "view sync", "layers": args.profile_layers, "params": total, "ranks": N,
                      "buckets": int(len(plan[2])), "ms_per_step": ms,
                      "hbm_alg_gbs": 2 * N * total * 4 / (ms / 1e3) / 1e9}), flush=True)


def run_profile_resnet(args):
    """The ResNet-50 DDP step in bf16 at N = 16 with the 25 MiB cap (first
    bucket 1 MiB), for profiling: --steps times pack + fused ring + unpack,
    then --steps times the fused view sync.  Prints one JSON line (not a
    bench result)."""
    import torch
    import gradient_sync_plan_gb300 as ddp
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    numels = workloads.param_numels(workloads.resnet50_param_shapes())
    N, total = 16, sum(numels)
    plan = ddp.ddp_plan_buckets(numels, ddp.BF16, MiB, 25 * MiB)
    g = torch.empty((N, total), dtype=torch.bfloat16, device=dev)
    for r in range(N):
        g[r].copy_(workloads.randn_f32(total, r, 1e-2, device=str(dev)).to(torch.bfloat16))
    offs = [0]
    for n in numels:
        offs.append(offs[-1] + n)
    views = [[g[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
    buckets = [[torch.empty(int(n), dtype=torch.bfloat16, device=dev) for n in plan[2]] for _ in range(N)]
    out = {"profile": "resnet50 bf16 sync", "params": total, "ranks": N, "buckets": int(len(plan[2]))}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, call in (("pack_fused_unpack", ddp.SyncCall(views, plan, buckets, N, ddp.DDP_ALGO_FUSED)),
                       ("view", ddp.SyncCall(views, plan, None, N, ddp.DDP_ALGO_VIEW))):
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            call()
        e1.record()
        torch.cuda.synchronize()
        out[name + "_ms"] = e0.elapsed_time(e1) / max(1, args.steps)
    print(json.dumps(out), flush=True)


def run_profile_kernels(args):
    """Every kernel family once on one workload larger than L2, for a
    per-kernel ncu DRAM capture: N = 8 ranks x 2^25 fp32 (128 MiB per rank,
    1 GiB over all ranks), in this order -- fused ring (vector, then TMA
    kernel), staged ring, persistent ring, fused tree (vector, then TMA
    kernel), staged tree, no_sync accumulation, pack and unpack of one
    bucket of 4 members per rank, bf16 pack and unpack (one 2^25-element
    member per rank), fused view (one bucket of 4 members per rank; register
    kernel, then TMA kernel).  --steps
    repeats the sequence.  Prints one JSON line (not a bench result)."""
    import torch
    import gradient_sync_plan_gb300 as ddp
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, S = N_RANKS, 1 << 25
    x = torch.empty((N, S), dtype=torch.float32, device=dev)
    for r in range(N):
        x[r].copy_(workloads.randn_f32(S, r, 1e-2, device=str(dev)))
    y = torch.empty_like(x)
    y.copy_(x)
    b16 = torch.empty((N, S), dtype=torch.bfloat16, device=dev)
    bk = torch.empty((N, S), dtype=torch.float32, device=dev)
    members = [S // 4] * 4
    offs = [0, S // 4, S // 2, 3 * S // 4]
    views = [[x[r, o:o + n] for o, n in zip(offs, members)] for r in range(N)]
    status = torch.zeros(2, dtype=torch.int32, device=dev)

    def forced(kind, fn):
        prev = ddp.ddp_set_fused_kernel(kind)
        try:
            fn()
        finally:
            ddp.ddp_set_fused_kernel(prev)

    seq = [("ring_fused_vector", lambda: forced(ddp.DDP_FUSED_VECTOR, lambda: ddp.ring_allreduce_fused(x, N))),
           ("ring_fused_tma", lambda: forced(ddp.DDP_FUSED_TMA, lambda: ddp.ring_allreduce_fused(x, N))),
           ("ring_staged", lambda: ddp.ring_allreduce_staged(x, N)),
           ("ring_persistent", lambda: ddp.ring_allreduce_persistent(x, N, status=status)),
           ("tree_fused_vector", lambda: forced(ddp.DDP_FUSED_VECTOR, lambda: ddp.tree_allreduce_fused(x, N))),
           ("tree_fused_tma", lambda: forced(ddp.DDP_FUSED_TMA, lambda: ddp.tree_allreduce_fused(x, N))),
           ("tree_staged", lambda: ddp.tree_allreduce_staged(x, N)),
           ("accumulate", lambda: ddp.ddp_grad_accumulate(x, y)),
           ("pack", lambda: ddp.ddp_bucket_pack(views, offs, bk)),
           ("unpack", lambda: ddp.ddp_bucket_unpack(views, offs, bk)),
           ("pack_bf16", lambda: ddp.ddp_bucket_pack_bf16([[x[r]] for r in range(N)], [0], b16)),
           ("unpack_bf16", lambda: ddp.ddp_bucket_unpack_bf16([[y[r]] for r in range(N)], [0], b16)),
           ("view_register", lambda: forced(ddp.DDP_FUSED_VECTOR,
                                            lambda: ddp.ddp_bucket_allreduce_view(views, offs, S, N))),
           ("view_tma", lambda: forced(ddp.DDP_FUSED_TMA, lambda: ddp.ddp_bucket_allreduce_view(views, offs, S, N)))]
    out = {"profile": "kernels", "ranks": N, "numel": S}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max(1, args.steps)):
        for name, fn in seq:
            torch.cuda.synchronize()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            out[name + "_ms"] = e0.elapsed_time(e1)
    assert int(status[0].item()) == 0
    print(json.dumps(out), flush=True)


def run_cpu_table(args):
    """The CPU oracle (single-threaded C, this host) on every workload,
    for the comparison table: one JSON line per measurement."""
    import numpy as np
    import oracle
    import workloads
    oracle.build()

    def timed(fn, reps=1):
        best = None
        for _ in range(reps):
            t = time.perf_counter()
            fn()
            dt = time.perf_counter() - t
            best = dt if best is None else min(best, dt)
        return best

    def emit(**kw):
        kw.setdefault("cores", 1)
        kw["host_cores_present"] = host_cores()
        print(json.dumps(kw), flush=True)

    # C1 and C2 and the C5 sweep: one bucket, ring allreduce / N; C1 and C2
    # also through the -fopenmp build of the same source (ranks of a
    # half-step on N threads, same per-element operations)
    for cfg, N, S, reps in (("C1", 4, 1 << 20, 3), ("C2", 8, 1 << 28, 1)):
        x = workloads.rank_vectors(N, S, "randn", std=1.0 if cfg == "C1" else 1e-2).numpy()
        rows = [x[r] for r in range(N)]
        t = timed(lambda: oracle.ring_allreduce(rows, oracle.F32, N), reps)
        emit(config=cfg, ranks=N, bytes_per_rank=S * 4, seconds=t,
             busbw_gbs=2 * (N - 1) / N * S * 4 / t / 1e9)
        try:
            t = timed(lambda: oracle.ring_allreduce_2d_openmp(x, oracle.F32, N), reps)
            emit(config=cfg, build="openmp", cores=min(N, host_cores() or N), ranks=N, bytes_per_rank=S * 4,
                 seconds=t, busbw_gbs=2 * (N - 1) / N * S * 4 / t / 1e9)
        except Exception as e:          # a compiler without OpenMP: no second row
            emit(config=cfg, build="openmp", unavailable=str(e)[:120])
        del x, rows
    for N, kmax in ((8, 16), (64, 14)):
        for k in range(0, kmax + 1, 2):
            S = 1024 << k
            x = workloads.rank_vectors(N, S, "uniform").numpy()
            rows = [x[r] for r in range(N)]
            t = timed(lambda: oracle.ring_allreduce(rows, oracle.F32, N), 3 if S < (1 << 22) else 1)
            emit(config="C5", ranks=N, bytes_per_rank=S * 4, seconds=t,
                 busbw_gbs=2 * (N - 1) / N * S * 4 / t / 1e9)
            del x, rows
    # C3: the decoder DDP step (plan, pack, ring / 8, unpack), and no_sync's accumulation
    numels = workloads.param_numels(workloads.decoder_param_shapes())
    N, total = 8, sum(numels)
    offs = np.cumsum([0] + numels)
    flat = workloads.rank_vectors(N, total, "randn", std=1e-2).numpy()
    grads = [[flat[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
    t = timed(lambda: oracle.ddp_sync(grads, oracle.F32))
    emit(config="C3", step="pack + ring / 8 + unpack, 37 buckets", ranks=N, grad_bytes_per_rank=total * 4, seconds=t)
    t = timed(lambda: oracle.accumulate(flat.reshape(-1), flat.reshape(-1).copy(), oracle.F32))
    emit(config="C3", step="one no_sync accumulation of all gradients, all ranks", ranks=N,
         grad_bytes_per_rank=total * 4, seconds=t)
    del flat, grads
    # C4: ResNet-50 bf16, N = 16, caps 5/10/25/50 MiB
    numels = workloads.param_numels(workloads.resnet50_param_shapes())
    N, total = 16, sum(numels)
    offs = np.cumsum([0] + numels)
    base = workloads.rank_vectors(N, total, "randn", std=1e-2, dtype="bf16").view(torch_int16()).numpy()
    for cap in (5, 10, 25, 50):
        flat = base.view(np.uint16).copy()
        grads = [[flat[r, offs[p]:offs[p + 1]] for p in range(len(numels))] for r in range(N)]
        t = timed(lambda: oracle.ddp_sync(grads, oracle.BF16, MiB, cap * MiB))
        emit(config="C4", cap_mib=cap, ranks=N, grad_bytes_per_rank=total * 2, seconds=t)


def torch_int16():
    import torch
    return torch.int16


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--numel", type=int, default=NUMEL, help="elements per rank (default: the 1 GiB bucket)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of CPU-oracle work")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work to size the per-step sample for")
    ap.add_argument("--cpu-table", action="store_true", help="time the CPU oracle on every config instead")
    ap.add_argument("--profile-view", action="store_true", help="small view-sync run for profiling instead")
    ap.add_argument("--profile-resnet", action="store_true",
                    help="ResNet-50 bf16 N=16 sync (25 MiB cap) for profiling instead")
    ap.add_argument("--profile-kernels", action="store_true",
                    help="every kernel family once on 8 x 128 MiB, for profiling instead")
    ap.add_argument("--profile-layers", type=int, default=2)
    ap.add_argument("--cap-sweep", action="store_true", help="bucket-cap sweep (one JSON line per point) instead")
    ap.add_argument("--sweep", action="store_true", help="message-size sweep (one JSON line per point) instead")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and args.steps >= 10:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    if args.sweep:
        run_sweep(args)
        return
    if args.cap_sweep:
        run_cap_sweep(args)
        return
    if args.profile_view:
        run_profile_view(args)
        return
    if args.profile_resnet:
        run_profile_resnet(args)
        return
    if args.profile_kernels:
        run_profile_kernels(args)
        return
    if args.cpu_table:
        run_cpu_table(args)
        return
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
