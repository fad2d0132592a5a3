#!/usr/bin/env python3
"""Throughput of exact attention (forward + backward) on GB300.

One step is one pass of the whole hot path over one batch of the causal
N=4096, d=128 workload (B=2, H=32, 1% of Q and K rows scaled x20): the
forward kernel, then the three backward stages (prepare, main, finish) --
exactly the launches fattn_fwd + fattn_bwd make.  FLOPs are counted as
4*B*H*N^2*d for the forward, x2.5 for the backward, halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fattn|reference]

With torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (attention over (batch, head) needs no exchange),
the timed region is bracketed by barriers and the max time over ranks is
used.  Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores instead (one
head of the workload per step), on the same metric.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s and fraction of GB300 dense BF16 peak"
DEFAULT_WORKLOAD = "b2h32_n4096_d128_causal_outliers"
KERNEL_SOURCES = {
    "fwd": ("exact_attention_fattn_gb300/csrc/fattn_fwd.cu",),
    "bwd_main": ("exact_attention_fattn_gb300/csrc/fattn_bwd.cu",
                 "exact_attention_fattn_gb300/csrc/fattn_bwd2.cu",
                 "exact_attention_fattn_gb300/csrc/fattn_sched.h",
                 "exact_attention_fattn_gb300/csrc/fattn_sched.cu"),
    "bwd_prepare": ("exact_attention_fattn_gb300/csrc/fattn_bwd_aux.cu",),
    "bwd_finish": ("exact_attention_fattn_gb300/csrc/fattn_bwd_aux.cu",),
}
L2_BYTES = 129 * 10**6


def flop_counts(w):
    base = 4.0 * w.B * w.H * w.N * w.N * w.d * (0.5 if w.causal else 1.0)
    return base, 2.5 * base


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def source_hash(rels):
    """sha256[:16] of a kernel's source files, concatenated, with comments and
    whitespace removed, so that only a change to the code (the kernel or the
    schedule it runs) invalidates a capture."""
    src = ""
    for rel in rels:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            src += f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"\s+", "", src)
    return hashlib.sha256(src.encode("utf-8")).hexdigest()[:16]


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed after the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload:
                    if parts[3] == source_hash(KERNEL_SOURCES[kernel]):
                        return float(parts[2])
                    return None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, time-stamped on the host."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed_region"
        if not inside and self.samples:
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            window = "nearest_to_timed_region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in inside:
            for name, flag in zip(names, s[3][1:]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------- replicas
# Every rank runs an independent replica of the workload (attention over
# (batch, head) needs no exchange); these helpers are the only cross-rank
# steps, and they work with either the nccl (GPU) or the gloo (CPU) backend.

def rank_info():
    """(rank, world size, local rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch of the same workload."""
    return base_seed + 7919 * rank


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(value: float, dist, device=None) -> float:
    """The slowest rank's time defines the step (whole-job timing)."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_replica: float, world: int, seconds: float) -> float:
    """Units processed by all replicas per second."""
    return world * units_per_replica / seconds


def cpu_baseline(w, heads: int):
    """The fp64 oracle, as it stands, on `heads` (b, h) slices of the
    workload: full forward + backward of each slice on the host cores."""
    import oracle
    from exact_attention_fattn_gb300 import workloads as W

    inp = W.make_inputs(w, with_grad=True)
    base, bwd = flop_counts(w)
    per_head = (base + bwd) / (w.B * w.H)
    t0 = time.perf_counter()
    for hflat in range(heads):
        b, h = divmod(hflat, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        sub = {n: inp[n][sl] for n in ("q", "k", "v", "do")}
        oracle.attention_forward(sub["q"], sub["k"], sub["v"], w.causal, w.scale)
        oracle.attention_backward(sub["q"], sub["k"], sub["v"], sub["do"], w.causal, w.scale)
    dt = time.perf_counter() - t0
    return {"value": per_head * heads / dt / 1e12, "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} heads of {w.name}: fp64 forward + backward "
                      f"({dt:.1f} s; BLAS threads at their default)",
            "seconds": dt}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from exact_attention_fattn_gb300 import workloads as W

    inp = W.make_inputs(w, with_grad=True)
    base, bwd = flop_counts(w)
    per_head = (base + bwd) / (w.B * w.H)
    nheads = w.B * w.H

    def step(k):
        b, h = divmod(k % nheads, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        sub = {n: inp[n][sl] for n in ("q", "k", "v", "do")}
        oracle.attention_forward(sub["q"], sub["k"], sub["v"], w.causal, w.scale)
        oracle.attention_backward(sub["q"], sub["k"], sub["v"], sub["do"], w.causal, w.scale)

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(args.warmup + k)
    dt = time.perf_counter() - t0
    value = per_head * args.steps / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = f"one (b, h) head of {w.name} per step, rotating over heads; fp64 forward + backward"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_fattn(args, w):
    import torch

    from exact_attention_fattn_gb300 import attention as A
    from exact_attention_fattn_gb300 import workloads as W

    rank, world, local = rank_info()
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    # replicas only: each rank draws its own batch of the same workload
    inp = W.make_inputs(w, seed=replica_seed(w.seed, rank), with_grad=True)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = A.workspace_for(q)
    sc = w.scale

    def fwd():
        A.fattn_fwd(q, k, v, causal=w.causal, scale=sc, out=o, lse=lse)

    def prep():
        A.fattn_bwd_prepare(o, do, lse, ws)

    def main():
        A.fattn_bwd_main(q, k, v, do, ws, dk, dv, causal=w.causal, scale=sc)

    def finish():
        A.fattn_bwd_finish(ws, dq, scale=sc)

    A.fattn_set_bwd_pair(args.bwd_pair)
    stages = [("fwd", fwd), ("bwd_prepare", prep), ("bwd_main", main), ("bwd_finish", finish)]
    for _ in range(args.warmup):
        for _, fn in stages:
            fn()
    status = A.fattn_check_status(dev)
    if status != 0:
        raise RuntimeError(f"libfattn reported status {status} during warm-up")

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    sampler = ClockSampler(uuid)
    time.sleep(0.3)

    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    start.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        for i, (_, fn) in enumerate(stages):
            fn()
            ev[s][i + 1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier(dist)
    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    step_times = [ev[s][0].elapsed_time(ev[s][len(stages)]) for s in range(args.steps)]
    status = A.fattn_check_status(dev)
    if status != 0:
        raise RuntimeError(f"libfattn reported status {status} in the timed region")
    per_stage = {name: statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1])
                                       for s in range(args.steps))
                 for i, (name, _) in enumerate(stages)}
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)

    # ---- end to end through the public API: pinned host buffers in, results out.
    # Every step copies its inputs host -> device, runs fattn_fwd + fattn_bwd
    # and copies O, L, dQ, dK, dV back.  The steps are pipelined the way a
    # serving loop would drive the library: step k+1's uploads and step k-1's
    # downloads run on their own streams while step k's kernels run, with two
    # device buffer sets (inputs and outputs) ordered by events.
    e2e = None
    if not args.no_e2e:
        host_in = {n: inp[n].pin_memory() for n in ("q", "k", "v", "do")}
        out_names = ("o", "lse", "dq", "dk", "dv")
        host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for n, t in zip(out_names, (o, lse, dq, dk, dv))}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        sets = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)]
        sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set b uploaded
        ev_run = [torch.cuda.Event() for _ in range(2)]    # kernels on set b done
        ev_out = [torch.cuda.Event() for _ in range(2)]    # outputs of set b downloaded

        def e2e_step(i):
            b = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_run[i % 2])          # step i-2 no longer reads set b
                for n in ("q", "k", "v", "do"):
                    b[n].copy_(host_in[n], non_blocking=True)
                ev_in[i % 2].record(s_in)
            stream.wait_event(ev_in[i % 2])
            if i >= 2:
                stream.wait_event(ev_out[i % 2])            # step i-2's outputs are out
            A.fattn_fwd(b["q"], b["k"], b["v"], causal=w.causal, scale=sc, out=b["o"],
                        lse=b["lse"])
            A.fattn_bwd(b["q"], b["k"], b["v"], b["o"], b["do"], b["lse"], causal=w.causal,
                        scale=sc, workspace=ws, dq=b["dq"], dk=b["dk"], dv=b["dv"])
            ev_run[i % 2].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[i % 2])
                for n in out_names:
                    host_out[n].copy_(b[n], non_blocking=True)
                ev_out[i % 2].record(s_out)

        e2e_steps = max(3, min(args.steps, 50))
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        s_in.wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i)
        stream.wait_event(ev_out[(e2e_steps - 1) % 2])
        stream.wait_event(ev_out[(e2e_steps - 2) % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
        base, bwd = flop_counts(w)
        e2e = {"value": whole_job_rate(base + bwd, world, e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": e2e_steps,
               "pipelining": "step k+1's H2D and step k-1's D2H overlap step k's kernels "
                             "(separate streams, two device buffer sets)"}
        if A.fattn_check_status(dev) != 0:
            raise RuntimeError("libfattn reported an error in the end-to-end run")

    # ---- extra rows, timed after the headline metric on the same inputs:
    # the FP8 forward (block quantization of Q, K, V, then the e4m3 forward)
    # and the deterministic backward.
    extras = None
    if not args.no_extras and w.d == 128:
        try:
            extras = measure_extras(args, w, (q, k, v, do), (o, lse), ws, (dq, dk, dv), dev,
                                    stream)
        except Exception as exc:   # the headline line must still be printed
            A.fattn_set_deterministic(False)
            extras = {"error": f"{type(exc).__name__}: {exc}"}
        try:
            extras["sweep"] = measure_sweep(dev)
        except Exception as exc:
            extras["sweep"] = {"error": f"{type(exc).__name__}: {exc}"}


    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return

    peaks = load_peaks()
    base, bwd = flop_counts(w)
    ms_step = total_ms / args.steps
    value = whole_job_rate(base + bwd, world, ms_step * 1e-3) / 1e12
    stage_flops = {"fwd": base, "bwd_main": bwd}
    dominant = max(per_stage, key=per_stage.get)
    dom_ms = per_stage[dominant]
    achieved = stage_flops.get(dominant, 0.0) / (dom_ms * 1e-3) / 1e12
    traffic = load_traffic(dominant, w.name)
    # The timed region lasts steps x ms_per_step (tens of ms at the default
    # step count), far shorter than the seconds-long loop behind the
    # sustained figure, so the burst peak is the denominator; the sustained
    # one only applies to a region of a second or more.
    region_s = total_ms * 1e-3
    peak_key = "bf16_sustained" if region_s >= 1.0 else "bf16"
    peak_kind = "sustained" if peak_key == "bf16_sustained" else "burst"
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks[peak_key],
                "unit": "TFLOP/s", "frac": achieved / peaks[peak_key],
                "traffic": traffic, "kernel": dominant,
                "peak_kind": f"bf16 dense, {peak_kind} ({peaks['source']}); timed region "
                             f"{region_s * 1e3:.1f} ms",
                "frac_of_sustained_peak": achieved / peaks["bf16_sustained"]}
    fwd_tf = base / (per_stage["fwd"] * 1e-3) / 1e12
    roofline_fwd = {"bound": "tensor", "achieved": fwd_tf, "peak": peaks[peak_key],
                    "unit": "TFLOP/s", "frac": fwd_tf / peaks[peak_key],
                    "traffic": load_traffic("fwd", w.name), "kernel": "fwd",
                    "peak_kind": roofline["peak_kind"],
                    "gate": "forward at >= 0.60 of the dense bf16 peak on this workload"}
    bwd_ms = per_stage["bwd_prepare"] + per_stage["bwd_main"] + per_stage["bwd_finish"]
    bwd_tf = bwd / (bwd_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "parallelism": f"replicas x{world}",
                   "bwd_kernel": "cta_pair" if args.bwd_pair else "one_cta_per_tile",
                   "l2": "inputs larger than L2: q, k, v, o, dO take "
                         f"{5 * q.numel() * 2 / 2**20:.0f} MiB > 129 MB L2; no flush"},
        "frac_of_peak": value / world / peaks["bf16"],
        "frac_of_peak_note": f"per-GPU value / {peaks['bf16']} TFLOP/s bf16 dense "
                             f"({peaks['source']} burst)",
        "fwd_tflops": fwd_tf, "fwd_frac_of_peak": fwd_tf / peaks["bf16"],
        "bwd_tflops": bwd_tf,
        "stage_ms": per_stage,
        "step_ms": {"mean": ms_step, "median": statistics.median(step_times),
                    "min": min(step_times)},
        "frac_of_spec_peak": value / world / spec_tflops(dev, clocks),
        "frac_of_spec_peak_note": "per-GPU value / (SMs x 8192 FLOP/clk/SM x max SM clock)",
        "roofline": roofline,
        "roofline_fwd": roofline_fwd,
        "clocks": clocks,
        "gpu_launches": args.steps * len(stages),
        "e2e": e2e,
    }
    if extras is not None:
        line["extras"] = extras
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_heads)
    print(json.dumps(line), flush=True)



def spec_tflops(dev, clocks):
    """SMs x 8192 dense bf16 FLOP per clock per SM x the maximum SM clock."""
    import torch

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    return sms * 8192.0 * float(mhz) * 1e6 / 1e12


# The workloads besides the headline one, timed per call: (name, B, H, N, d,
# causal, value scale, with backward).  The non-causal N = 4096 points use the
# batch and heads of the sweep workload and of the headline workload.
SWEEP = (
    ("tiny_b1h1_n128_d64", 1, 1, 128, 64, False, 1.0, False),
    ("b4h16_n1024_d64", 4, 16, 1024, 64, False, 1.0, True),
    ("b8h16_n512_d128_half", 8, 16, 512, 128, False, 0.5, False),
    ("b8h16_n1024_d128_half", 8, 16, 1024, 128, False, 0.5, False),
    ("b8h16_n2048_d128_half", 8, 16, 2048, 128, False, 0.5, False),
    ("b8h16_n4096_d128", 8, 16, 4096, 128, False, 1.0, True),
    ("b2h32_n4096_d128", 2, 32, 4096, 128, False, 1.0, True),
    ("b1h16_n16384_d128_causal", 1, 16, 16384, 128, True, 1.0, True),
)


def measure_sweep(dev, warmup=5, reps=20):
    """Forward (and backward) TFLOP/s of every workload besides the headline:
    inputs drawn on the device (timing only), 5 warm-up calls, then 20 calls
    each between CUDA events; median and best.  The tiny workload is bound by
    the host's call rate, not by the kernel."""
    import torch

    from exact_attention_fattn_gb300 import attention as A

    g = torch.Generator(device=dev)
    out = []
    for name, B, H, N, d, causal, vs, with_bwd in SWEEP:
        g.manual_seed(2000 + len(out))
        q, k, v, do = (
            (torch.randn((B, H, N, d), generator=g, device=dev) * vs).to(torch.bfloat16)
            for _ in range(4))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        sc = A.default_scale(d)
        fl = 4.0 * B * H * N * N * d * (0.5 if causal else 1.0)

        def per_call(fn):
            for _ in range(warmup):
                fn()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
            torch.cuda.synchronize(dev)
            evs[0].record()
            for i in range(reps):
                fn()
                evs[i + 1].record()
            torch.cuda.synchronize(dev)
            ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(reps)]
            return statistics.median(ms), min(ms)

        fwd_med, fwd_min = per_call(
            lambda: A.fattn_fwd(q, k, v, causal=causal, scale=sc, out=o, lse=lse))
        row = {"workload": name, "fwd_ms_median": fwd_med,
               "fwd_tflops_median": fl / (fwd_med * 1e-3) / 1e12,
               "fwd_tflops_best": fl / (fwd_min * 1e-3) / 1e12}
        if with_bwd:
            ws = A.workspace_for(q)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            bwd_med, bwd_min = per_call(
                lambda: A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=sc, workspace=ws,
                                    dq=dq, dk=dk, dv=dv))
            row.update({"bwd_ms_median": bwd_med,
                        "bwd_tflops_median": 2.5 * fl / (bwd_med * 1e-3) / 1e12,
                        "bwd_tflops_best": 2.5 * fl / (bwd_min * 1e-3) / 1e12})
            del ws, dq, dk, dv
        status = A.fattn_check_status(dev)
        if status != 0:
            raise RuntimeError(f"libfattn reported status {status} on {name}")
        out.append(row)
        del q, k, v, do, o, lse
        torch.cuda.empty_cache()
    return out


def measure_extras(args, w, qkvd, out, ws, grads, dev, stream):
    """Extra rows, timed after the headline metric on the same inputs: the FP8
    forward (block quantization of Q, K, V, also with Q and K rotated for
    incoherent processing, then the e4m3 forward) and the deterministic
    backward."""
    import torch

    from exact_attention_fattn_gb300 import attention as A

    q, k, v, do = qkvd
    o, lse = out
    dq, dk, dv = grads
    sc = w.scale

    def timed(fn, reps):
        for _ in range(3):
            fn()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a0.record(stream)
        for _ in range(reps):
            fn()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        return a0.elapsed_time(a1) / reps

    def graph_timed(fn, reps):
        # Short kernels: the host enqueues more slowly than the GPU runs them,
        # so they are timed from a captured graph of ``reps`` calls.
        fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        cur = torch.cuda.current_stream(dev)
        for _ in range(2):
            g.replay()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a0.record(cur)
        g.replay()
        a1.record(cur)
        torch.cuda.synchronize(dev)
        return a0.elapsed_time(a1) / reps

    q8, sq = A.fattn_quantize_fp8(q)
    k8, sk = A.fattn_quantize_fp8(k)
    v8t, sv = A.fattn_quantize_fp8(v, transposed=True)
    reps = max(3, min(args.steps, 50))
    quant_ms = graph_timed(lambda: (A.fattn_quantize_fp8(q), A.fattn_quantize_fp8(k),
                                    A.fattn_quantize_fp8(v, transposed=True)), 20)
    signs = torch.ones(w.d, dtype=torch.float32, device=dev)
    signs[1::2] = -1.0
    rot_ms = graph_timed(lambda: (A.fattn_quantize_fp8(q, signs=signs),
                                  A.fattn_quantize_fp8(k, signs=signs),
                                  A.fattn_quantize_fp8(v, transposed=True)), 20)
    fp8_ms = timed(lambda: A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=w.causal, scale=sc,
                                           out=o, lse=lse), reps)
    A.fattn_set_deterministic(True)
    try:
        det_ms = timed(lambda: A.fattn_bwd(q, k, v, o, do, lse, causal=w.causal, scale=sc,
                                           workspace=ws, dq=dq, dk=dk, dv=dv), reps)
    finally:
        A.fattn_set_deterministic(False)
    status = A.fattn_check_status(dev)
    if status != 0:
        raise RuntimeError(f"libfattn reported status {status} in the extra measurements")
    base, bwd = flop_counts(w)
    return {"fp8_fwd": {"tflops": base / (fp8_ms * 1e-3) / 1e12, "ms": fp8_ms,
                        "quantize_qkv_ms": quant_ms, "quantize_qkv_rotated_ms": rot_ms,
                        "steps": reps},
            "bwd_deterministic": {"tflops": bwd / (det_ms * 1e-3) / 1e12, "ms": det_ms,
                                  "steps": reps}}

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("fattn", "reference"), default="fattn")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the FP8 forward, deterministic backward and workload sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd-pair", action="store_true",
                    help="time the CTA-pair backward kernel (fattn_set_bwd_pair) instead of the "
                         "default one-CTA-per-tile kernel")
    ap.add_argument("--cpu-heads", type=int, default=32)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)      # at least three untimed warm-up steps
    from exact_attention_fattn_gb300 import workloads as W

    w = W.BY_NAME.get(args.workload)
    if w is None:
        name, _, n = args.workload.partition("@N")
        w = W.BY_NAME[name].with_n(int(n))
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_fattn(args, w)


if __name__ == "__main__":
    main()
