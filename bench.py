#!/usr/bin/env python3
"""Benchmark: exact attention forward TFLOP/s on GB300 (one JSON line).

Workload (default): the Llama-3-8B layer shape B=1, H=32, N=8192, d=128,
causal, bf16 Q/K/V i.i.d. N(0,1) from seed 3, scale 1/sqrt(128).
Metric: 4*B*H*N^2*d / t, halved for causal, in TFLOP/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

ours: W warm-up steps, then exactly K timed steps (one fa_fwd launch each),
  bracketed by a barrier and a device synchronise on both sides, CUDA events
  on the launching stream, max over ranks.  Three resident input sets
  (3 x 256 MiB incl. outputs, > the 129 MB L2) are used in rotation, so a
  step never finds its K/V already in L2 from the step before.  Adds the
  end-to-end number through the host-buffer C-ABI call (pinned host memory,
  copies inside the timed region), the roofline of the kernel, SM clocks
  sampled during the timed region, and the fp64 CPU oracle timed on a
  bounded sample of the same workload.
reference: the fp64 CPU oracle as it stands, on the host cores, each step a
  bounded sample of the same workload (rank 0 only under torchrun).
Under torchrun every rank runs the full workload on its own GPU (weak
scaling, no data-path collective); value = all ranks' FLOPs / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from online_softmax_fa_gb300.inputs import (DECODE_WORKLOADS, WORKLOADS,  # noqa: E402
                                            make_decode, make_workload)

METRIC = ("attn fwd TFLOP/s (4·B·H·N²·d, causal halved) "
          "and % of GB300 BF16 tensor peak")
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCES = ["online_softmax_fa_gb300/csrc/fa_fwd_sm103.cu",
                  "online_softmax_fa_gb300/csrc/sm103_primitives.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fa_fwd_llama_traffic.json")


def workload_config(w, causal, kind="forward"):
    kv = f" (K/V heads {w.kv_heads})" if w.kv_heads != w.H else ""
    return {"workload": f"{w.name} attention {kind} B{w.B} H{w.H}{kv} N{w.N} d{w.d}"
                        + (" causal" if causal else ""),
            "B": w.B, "H": w.H, "H_kv": w.kv_heads, "N": w.N, "d": w.d, "causal": causal,
            "scale": "1/sqrt(d) in fp32", "inputs": f"bf16 i.i.d. N(0,1), seed {w.seed}",
            "l2": "inputs > L2: 3 resident input sets of 256 MiB used in rotation"}


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a host float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of `flops_per_rank`
    (weak scaling), timed by the slowest rank (`max_ms` for all steps)."""
    return world * flops_per_rank * steps / (max_ms * 1e-3) / 1e12


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0) or 0), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 0.0, "fallback"


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per launch from an ncu capture, if taken on this kernel."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_source_digest():
        return None  # the kernel changed since the counters were taken
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle leg
def row_flops(rows: np.ndarray, N: int, d: int, causal: bool) -> float:
    """Nominal FLOPs of the given query rows (4*d per attended key)."""
    if causal:
        return float(4.0 * d * np.sum(rows.astype(np.float64) + 1.0))
    return float(4.0 * d * N * rows.size)


def oracle_sample(w, causal, q, k, v, rows_per_head, nthreads, offset=0, keep=None):
    """Time the fp64 oracle on `rows_per_head` evenly spread rows of every
    head; returns (seconds, nominal FLOPs of those rows).  With a dict as
    `keep`, also leaves the rows and the oracle's O and LSE there."""
    import oracle
    BH = w.B * w.H
    stride = max(1, w.N // rows_per_head)
    base = (np.arange(rows_per_head, dtype=np.int64) * stride + offset) % w.N
    rows = np.broadcast_to(base, (BH, rows_per_head)).copy()
    t0 = time.perf_counter()
    o_ref, l_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=w.scale, rows=rows,
                                        nthreads=nthreads)
    dt = time.perf_counter() - t0
    if keep is not None:
        keep.update(rows=rows, o=o_ref, lse=l_ref)
    return dt, row_flops(rows, w.N, w.d, causal)


# The output contract: O max-abs and mean-abs error, LSE abs error against
# the fp64 oracle (bf16 output, fp32 accumulation).
PARITY_BOUNDS = {"o_max_abs": 2e-2, "o_mean_abs": 2e-3, "lse_max_abs": 1e-3}


def sample_parity(o_gpu, lse_gpu, rows, o_ref, l_ref):
    """Error of the GPU output (O bf16 [B,H,N,d], LSE fp32 [B,H,N], device or
    host tensors) on the oracle's sampled rows [B*H, R]."""
    BH, R = rows.shape
    o = o_gpu.float().cpu().numpy().reshape(BH, -1, o_gpu.shape[-1])
    lse = lse_gpu.float().cpu().numpy().reshape(BH, -1)
    o_s = np.take_along_axis(o, rows[:, :, None], axis=1)
    l_s = np.take_along_axis(lse, rows, axis=1)
    eo = np.abs(o_s - o_ref.reshape(BH, R, -1))
    el = np.abs(l_s - l_ref.reshape(BH, R))
    got = {"o_max_abs": float(eo.max()), "o_mean_abs": float(eo.mean()),
           "lse_max_abs": float(el.max())}
    return {"rows": int(BH * R), **got, "bounds": PARITY_BOUNDS,
            "within_bounds": all(got[key] <= PARITY_BOUNDS[key] for key in got)}


def oracle_inputs(w):
    """Q, K, V in fp64 as [B*H, N, d]; grouped-query K/V heads are repeated
    for the query heads of their group (query head h uses K/V head
    h // (H / H_kv)), so the dense oracle sees the same attention."""
    import oracle
    q, k, v = make_workload(w)
    BH = w.B * w.H
    shp = (BH, w.N, w.d)
    group = w.H // w.kv_heads
    if group > 1:
        k, v = (t.repeat_interleave(group, dim=1) for t in (k, v))
    return tuple(oracle.bf16_bits_to_f64(t.reshape(shp)) for t in (q, k, v))


def host_cpu() -> str:
    """The host CPU as the kernel reports it (model name or CPU part), with
    the machine type and the number of online cores."""
    import platform
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part") and ":" in line:
                    name = line.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    return f"{platform.machine()} {name} x{os.cpu_count()}".strip()


def cpu_baseline(w, causal, target_s=15.0, gpu_out=None):
    """The oracle timed on a bounded sample of the workload's rows; with the
    GPU's (O, LSE) of the same inputs, also their error on those rows."""
    import oracle
    qf, kf, vf = oracle_inputs(w)
    nth = oracle.default_threads()
    dt, _ = oracle_sample(w, causal, qf, kf, vf, 8, nth)  # calibration
    per_row = dt / 8
    rph = int(min(w.N, max(8, target_s / max(per_row, 1e-6))))
    ref = {}
    dt, fl = oracle_sample(w, causal, qf, kf, vf, rph, nth, keep=ref)
    out = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
           "cpu": host_cpu(),
           "sample": f"{rph} evenly spaced query rows in each of the {w.B * w.H} heads "
                     f"({rph * w.B * w.H} rows, {dt:.1f} s); fp64, S and P materialised "
                     f"over all N keys per row; FLOPs counted as 4*d per attended key"}
    if gpu_out is not None:
        out["parity"] = sample_parity(*gpu_out, ref["rows"], ref["o"], ref["lse"])
    return out


def run_reference(args, w, causal):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    qf, kf, vf = oracle_inputs(w)
    nth = oracle.default_threads()
    dt, _ = oracle_sample(w, causal, qf, kf, vf, 8, nth)
    per_row = dt / 8
    budget_s = 120.0
    total_steps = max(1, args.steps + args.warmup)
    rph = int(min(w.N, max(1, budget_s / total_steps / max(per_row, 1e-6))))
    for i in range(args.warmup):
        oracle_sample(w, causal, qf, kf, vf, rph, nth, offset=i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = oracle_sample(w, causal, qf, kf, vf, rph, nth, offset=args.warmup + i)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = (f"each step: {rph} evenly spaced query rows (offset by the step index) in each "
              f"of the {w.B * w.H} heads; fp64 oracle, S and P materialised")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(w, causal),
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
                            "cpu": host_cpu(),
                            "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ our arm
def run_ours(args, w, causal):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from online_softmax_fa_gb300 import fa
    from online_softmax_fa_gb300.build import build_library
    build_library()  # no-op when up to date; raises if nvcc fails
    fa.load_library()

    q, k, v = make_workload(w)
    B, H, N, d = w.B, w.H, w.N, w.d
    gqa = w.kv_heads != w.H
    step = fa.fa_fwd_gqa if gqa else fa.fa_fwd
    sets = []
    for _ in range(3):
        sets.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(q, device=dev),
                     torch.empty((B, H, N), dtype=torch.float32, device=dev)))
    stream = torch.cuda.current_stream()
    flops = w.flops(causal)

    for i in range(args.warmup):
        qd, kd, vd, od, ld = sets[i % 3]
        step(qd, kd, vd, od, ld, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    if fa.fa_device_error() != 0:
        raise RuntimeError("device status set during warm-up")

    props = torch.cuda.get_device_properties(dev)
    gpu_uuid = None
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        gpu_uuid = s if s.startswith("GPU-") else "GPU-" + s
    sampler = ClockSampler(gpu_uuid)
    time.sleep(0.5)  # let the sampler start
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        qd, kd, vd, od, ld = sets[i % 3]
        starts[i].record(stream)
        step(qd, kd, vd, od, ld, causal=causal, scale=w.scale)
        ends[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    status = fa.fa_device_error()
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed region")
    total_ms = e0.elapsed_time(e1)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kern_ms = statistics.fmean(launch_ms)
    total_ms_max = max_over_ranks(total_ms, ws)
    value = aggregate_tflops(flops, args.steps, total_ms_max, ws)

    # end to end through the host-buffer entry point: H2D of Q, K, V from
    # pinned memory, the kernel, D2H of O and LSE -- every step
    e2e_steps = max(3, min(args.steps, 30))
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    if gqa:
        wsp = torch.empty(fa.fa_fwd_host_gqa_workspace_bytes(B, H, w.kv_heads, N, d),
                          dtype=torch.uint8, device=dev)
        host_step = fa.fa_fwd_host_gqa
    else:
        wsp = torch.empty(fa.fa_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                          device=dev)
        host_step = fa.fa_fwd_host
    for _ in range(2):
        host_step(qh, kh, vh, oh, lh, wsp, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    barrier(ws)
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        host_step(qh, kh, vh, oh, lh, wsp, causal=causal, scale=w.scale)
    x1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    if fa.fa_device_error() != 0:
        raise RuntimeError("device status set during the end-to-end leg")
    e2e_ms = max_over_ranks(x0.elapsed_time(x1), ws)
    e2e_value = aggregate_tflops(flops, e2e_steps, e2e_ms, ws)
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = q.numel() * 2 + B * H * N * 4

    if rank != 0:
        return
    peak, peak_sust, peak_kind = load_peaks()
    achieved = flops / (kern_ms * 1e-3) / 1e12
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w, causal),
        "pct_of_nominal_bf16_peak": 100.0 * value / ws / NOMINAL_BF16_TFLOPS,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"bf16_tflops (burst) of {peak_kind}",
                     "traffic": recorded_traffic() if w.name == "llama" else None,
                     "kernel": f"fa_fwd_kernel<{d},{str(causal).lower()}>",
                     "kernel_ms": kern_ms,
                     # per-launch CUDA-event durations of the same timed launches
                     "kernel_ms_median": statistics.median(launch_ms),
                     "kernel_ms_min": min(launch_ms), "launches_timed": len(launch_ms)},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": e2e_ms / e2e_steps,
                "api": ("fa_fwd_host_gqa" if gqa else "fa_fwd_host")
                       + " (C ABI, pinned host buffers)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if ws == 1 and not args.no_secondary:
        out["secondary"] = secondary_legs(dev, fa, peak, peak_kind)
    if ws == 1 and not args.no_cpu_baseline:
        # the timed launches' output (every set holds the same inputs)
        out["cpu_baseline"] = cpu_baseline(w, causal, gpu_out=(sets[0][3], sets[0][4]))
    print(json.dumps(out), flush=True)


# ------------------------------------------------------- secondary legs
def time_device(step, n, warmup, steps, stream):
    """Runs step(i) `warmup` times, then times `steps` calls with CUDA events
    on `stream` (synchronised on both sides).  Returns (mean ms per call
    over the whole timed region, per-call ms list)."""
    import torch
    for i in range(warmup):
        step(i % n)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        step(i % n)
        ends[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, [a.elapsed_time(b) for a, b in zip(starts, ends)]


def secondary_legs(dev, fa, peak, peak_kind):
    """The other rows of the hot path, measured in the same process after
    the headline leg, a few steps each: the backward pass on the llama
    workload, the grouped-query forward (device and host buffers), the
    d = 256 forward, decoding against a K/V cache, the latency-bound small
    workloads, and the oracle on the small workloads (one thread and all)."""
    import torch
    import oracle
    from online_softmax_fa_gb300.inputs import make_grad
    stream = torch.cuda.current_stream()
    out = {}
    status = []

    def fwd_leg(name, steps, e2e_steps=0, keep=None):
        w = WORKLOADS[name]
        causal = w.causal[-1]
        q, k, v = make_workload(w)
        gqa = w.kv_heads != w.H
        f = fa.fa_fwd_gqa if gqa else fa.fa_fwd
        sets = [(q.to(dev), k.to(dev), v.to(dev)) for _ in range(3)]
        outs = [(torch.empty_like(sets[0][0]),
                 torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev))
                for _ in range(3)]

        def step(i):
            f(*sets[i], o=outs[i][0], lse=outs[i][1], causal=causal, scale=w.scale)
        ms, per = time_device(step, 3, 5, steps, stream)
        status.append(fa.fa_device_error())
        tf = w.flops(causal) / (ms * 1e-3) / 1e12
        leg = {"workload": workload_config(w, causal)["workload"], "value": tf,
               "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
               "kernel_ms_median": statistics.median(per),
               "roofline": {"bound": "tensor", "achieved": tf, "peak": peak,
                            "frac": tf / peak, "peak_source": f"bf16_tflops of {peak_kind}"}}
        if keep is not None:
            keep["gpu"] = (outs[0][0].cpu(), outs[0][1].cpu())
        del sets, outs
        if e2e_steps:
            host = fa.fa_fwd_host_gqa if gqa else fa.fa_fwd_host
            wbytes = (fa.fa_fwd_host_gqa_workspace_bytes(w.B, w.H, w.kv_heads, w.N, w.d)
                      if gqa else fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.N, w.d))
            wsp = torch.empty(wbytes, dtype=torch.uint8, device=dev)
            qh, kh, vh = (t.pin_memory() for t in (q, k, v))
            oh = torch.empty_like(q).pin_memory()
            lh = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
            ms_h, _ = time_device(lambda i: host(qh, kh, vh, oh, lh, wsp, causal=causal,
                                                 scale=w.scale), 1, 2, e2e_steps, stream)
            status.append(fa.fa_device_error())
            leg["e2e"] = {"value": w.flops(causal) / (ms_h * 1e-3) / 1e12, "unit": "TFLOP/s",
                          "ms_per_step": ms_h, "steps": e2e_steps,
                          "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2,
                          "d2h_bytes_per_step": q.numel() * 2 + w.B * w.H * w.N * 4,
                          "api": ("fa_fwd_host_gqa" if gqa else "fa_fwd_host")}
        return leg

    out["gqa_forward"] = fwd_leg("llama_gqa", 100, e2e_steps=10)
    out["d256_forward"] = fwd_leg("d256", 100)
    # the other two full-size configurations, each with the oracle timed on
    # a bounded sample of its rows (the batch workload: 16 rows per head;
    # the long one: its parity sample, 512 seeded rows per head and the edge
    # rows, all of which attend to up to 32771 keys)
    for name, rph in (("batch", 16), ("long", 0)):
        w = WORKLOADS[name]
        causal = w.causal[-1]
        kept = {}
        leg = fwd_leg(name, 50 if name == "batch" else 20, keep=kept)
        qf, kf, vf = oracle_inputs(w)
        nth = oracle.default_threads()
        ref = {}
        if rph:
            dt, fl = oracle_sample(w, causal, qf, kf, vf, rph, nth, keep=ref)
            what = f"{rph} evenly spaced rows in each of the {w.B * w.H} heads"
        else:
            from online_softmax_fa_gb300.inputs import sample_rows
            rows = sample_rows(w.N, w.B * w.H, w.sampled_rows, seed=w.seed)
            t0 = time.perf_counter()
            o_ref, l_ref = oracle.attention_fwd(qf, kf, vf, causal=causal, scale=w.scale,
                                                rows=rows, nthreads=nth)
            dt = time.perf_counter() - t0
            ref.update(rows=rows, o=o_ref, lse=l_ref)
            fl = row_flops(rows, w.N, w.d, causal)
            what = f"the parity sample: {rows.shape[1]} rows in each of the {w.B * w.H} heads"
        leg["oracle"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "seconds": dt,
                         "cores": nth, "sample": what,
                         "parity": sample_parity(*kept["gpu"], ref["rows"], ref["o"],
                                                 ref["lse"])}
        out[f"{name}_forward"] = leg
        del qf, kf, vf

    # backward (5 nominal N x N x d products) on the llama workload and at
    # head dimension 256
    def bwd_leg(name, steps):
        w = WORKLOADS[name]
        q, k, v = (t.to(dev) for t in make_workload(w))
        do = make_grad(w.B, w.H, w.N, w.d, w.seed).to(dev)
        o, lse = fa.fa_fwd(q, k, v, causal=True, scale=w.scale)
        grads = [tuple(torch.empty_like(q) for _ in range(3)) for _ in range(2)]
        wsb = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                          device=dev)

        def bstep(i):
            fa.fa_bwd(q, k, v, o, lse, do, *grads[i], workspace=wsb, causal=True,
                      scale=w.scale)
        ms, per = time_device(bstep, 2, 3, steps, stream)
        status.append(fa.fa_device_error())
        tf = 2.5 * w.flops(True) / (ms * 1e-3) / 1e12
        return {"workload": f"{name} attention backward B{w.B} H{w.H} N{w.N} d{w.d} causal",
                "metric": "TFLOP/s over 10*B*H*N^2*d, causal halved",
                "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
                "kernel_ms_median": statistics.median(per), "launches_per_step": 3,
                "roofline": {"bound": "tensor", "achieved": tf, "peak": peak,
                             "frac": tf / peak, "peak_source": f"bf16_tflops of {peak_kind}"}}

    out["backward"] = bwd_leg("llama", 100)
    out["d256_backward"] = bwd_leg("d256", 20)

    # decoding: one new query row per head against an 8192-position cache
    wd = DECODE_WORKLOADS["decode"]
    qd, kd, vd = make_decode(wd.B, wd.H, wd.kv_heads, wd.N, wd.d, wd.seed)
    need = fa.fa_decode_workspace_bytes(wd.B, wd.H, wd.kv_heads, wd.N, wd.d)
    dsets = [(qd.to(dev), kd.to(dev), vd.to(dev), torch.empty(need, dtype=torch.uint8,
                                                             device=dev)) for _ in range(3)]
    dout = (torch.empty_like(dsets[0][0]),
            torch.empty((wd.B, wd.H), dtype=torch.float32, device=dev))
    ms, per = time_device(lambda i: fa.fa_decode(*dsets[i][:3], workspace=dsets[i][3],
                                                 o=dout[0], lse=dout[1], scale=wd.scale),
                          3, 10, 200, stream)
    status.append(fa.fa_device_error())
    nbytes = decode_bytes(wd)
    hbm, hkind = load_hbm_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["decode"] = {"workload": f"decode B{wd.B} H{wd.H} (K/V heads {wd.kv_heads}) "
                                 f"N{wd.N} d{wd.d}, one query row per head",
                     "value": gbs, "unit": "GB/s", "ms_per_step": ms, "steps": 200,
                     "launches_per_step": 2,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm,
                                  "frac": gbs / hbm, "peak_source": f"hbm_gbs of {hkind}",
                                  "algorithmic_bytes": nbytes}}
    del dsets

    # latency-bound small workloads: per-call device time, and the oracle
    # on the same inputs (all host threads, and one thread for the tiniest)
    small = {}
    for name, causal in (("tiny", False), ("late", False), ("late", True)):
        w = WORKLOADS[name]
        qc, kc, vc = make_workload(w)
        qg, kg, vg = (t.to(dev) for t in (qc, kc, vc))
        og = torch.empty_like(qg)
        lg = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        ms, per = time_device(lambda i: fa.fa_fwd(qg, kg, vg, o=og, lse=lg, causal=causal,
                                                  scale=w.scale), 1, 20, 200, stream)
        status.append(fa.fa_device_error())
        med = statistics.median(per)
        # the device time without the host's submission cost: 20 calls
        # captured in a CUDA graph, the graph replayed
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(20):
                fa.fa_fwd(qg, kg, vg, o=og, lse=lg, causal=causal, scale=w.scale)
        ms_graph, _ = time_device(lambda i: graph.replay(), 1, 3, 10, stream)
        status.append(fa.fa_device_error())
        del graph
        nth = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.attention_fwd(qc, kc, vc, causal=causal, scale=w.scale, nthreads=nth)
        t_all = time.perf_counter() - t0
        key = f"{name}_{'causal' if causal else 'noncausal'}"
        small[key] = {"workload": workload_config(w, causal)["workload"],
                      "us_per_call_median": med * 1e3, "us_per_call_mean": ms * 1e3,
                      "tflops_at_median": w.flops(causal) / (med * 1e-3) / 1e12,
                      "us_per_call_graph": ms_graph / 20 * 1e3,
                      "tflops_graph": w.flops(causal) / (ms_graph / 20 * 1e-3) / 1e12,
                      "oracle_s": t_all, "oracle_threads": nth}
        if name == "tiny":
            t0 = time.perf_counter()
            oracle.attention_fwd(qc, kc, vc, causal=causal, scale=w.scale, nthreads=1)
            small[key]["oracle_s_one_thread"] = time.perf_counter() - t0
    out["small"] = small
    if any(st != 0 for st in status):
        raise RuntimeError("device status set during a secondary leg")
    return out


def load_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ------------------------------------------------------------ decode leg
def decode_bytes(w) -> int:
    """Algorithmic HBM bytes of one decoding step: K and V read once per K/V
    head, q read, O and LSE written.  The partial softmax states the split
    kernel hands to the merge kernel (about 1 MB here) are not counted: they
    are the implementation's, not the problem's."""
    kv = 2 * w.B * w.kv_heads * w.N * w.d * 2
    qo = 2 * w.B * w.H * w.d * 2
    return kv + qo + w.B * w.H * 4


def run_decode(args, w):
    import torch
    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from online_softmax_fa_gb300 import fa
    from online_softmax_fa_gb300.build import build_library
    build_library()
    fa.load_library()
    q, k, v = make_decode(w.B, w.H, w.kv_heads, w.N, w.d, w.seed)
    need = fa.fa_decode_workspace_bytes(w.B, w.H, w.kv_heads, w.N, w.d)
    sets = [(q.to(dev), k.to(dev), v.to(dev),
             torch.empty(need, dtype=torch.uint8, device=dev),
             torch.empty_like(q, device=dev),
             torch.empty((w.B, w.H), dtype=torch.float32, device=dev)) for _ in range(3)]
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        qd, kd, vd, wk, od, ld = sets[i % 3]
        fa.fa_decode(qd, kd, vd, wk, od, ld, scale=w.scale)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        qd, kd, vd, wk, od, ld = sets[i % 3]
        fa.fa_decode(qd, kd, vd, wk, od, ld, scale=w.scale)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws_)
    if fa.fa_device_error() != 0:
        raise RuntimeError("device status set during the decode leg")
    ms = max_over_ranks(e0.elapsed_time(e1), ws_) / args.steps
    if rank != 0:
        return
    nbytes = decode_bytes(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    flops = 4.0 * w.B * w.H * w.N * w.d
    hbm, kind = load_hbm_peak()
    out = {"metric": "attn decode TFLOP/s (4·B·H·N·d) at one query row per head",
           "value": ws_ * flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": ws_,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"decode B{w.B} H{w.H} (K/V heads {w.kv_heads}) "
                                  f"N{w.N} d{w.d}, one query row per head",
                      "l2": "inputs > L2: 3 resident K/V caches of 537 MB in rotation"},
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                        "frac": gbs / hbm, "peak_source": f"hbm_gbs of {kind}",
                        "traffic": None, "algorithmic_bytes": nbytes},
           "gpu_launches": 2 * args.steps}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------- backward leg
def run_backward(args, w, causal):
    """fa_bwd on the workload: TFLOP/s over the nominal backward FLOPs,
    10*B*H*N^2*d (five N x N x d products: S, dP, dV, dK, dQ), halved when
    causal.  The kernels recompute S and dP once more for dQ (seven
    products); the metric counts the nominal five."""
    import torch
    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from online_softmax_fa_gb300 import fa
    from online_softmax_fa_gb300.build import build_library
    from online_softmax_fa_gb300.inputs import make_grad
    build_library()
    fa.load_library()
    q, k, v = make_workload(w)
    do = make_grad(w.B, w.H, w.N, w.d, w.seed)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    gqa = bool(w.H_kv) and w.H_kv != w.H
    fwd = fa.fa_fwd_gqa if gqa else fa.fa_fwd
    bwd = fa.fa_bwd_gqa if gqa else fa.fa_bwd
    o, lse = fwd(qd, kd, vd, causal=causal, scale=w.scale)
    grads = [(torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd))
             for _ in range(2)]
    wsb = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                      device=dev)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        dq, dk, dv = grads[i % 2]
        bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, wsb, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        dq, dk, dv = grads[i % 2]
        bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, wsb, causal=causal, scale=w.scale)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws_)
    if fa.fa_device_error() != 0:
        raise RuntimeError("device status set during the backward leg")
    ms = max_over_ranks(e0.elapsed_time(e1), ws_) / args.steps
    if rank != 0:
        return
    flops = 2.5 * w.flops(causal)
    peak, _, peak_kind = load_peaks()
    value = ws_ * flops / (ms * 1e-3) / 1e12
    out = {"metric": "attn bwd TFLOP/s (10·B·H·N²·d, causal halved)", "value": value,
           "unit": "TFLOP/s", "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": workload_config(w, causal, "backward"),
           "roofline": {"bound": "tensor", "achieved": value / ws_, "peak": peak,
                        "unit": "TFLOP/s", "frac": value / ws_ / peak,
                        "peak_source": f"bf16_tflops (burst) of {peak_kind}",
                        "traffic": None, "kernel": "pre + dkdv + dq (three launches)"},
           "gpu_launches": 3 * args.steps}
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(DECODE_WORKLOADS),
                    default="llama")
    ap.add_argument("--causal", choices=["auto", "0", "1"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other hot-path legs (backward, GQA, d = 256, decoding, "
                         "small workloads) that a one-GPU run adds to its line")
    ap.add_argument("--backward", action="store_true",
                    help="time fa_bwd (gradients) instead of the forward pass")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.workload in DECODE_WORKLOADS:
        run_decode(args, DECODE_WORKLOADS[args.workload])
        return
    w = WORKLOADS[args.workload]
    causal = w.causal[-1] if args.causal == "auto" else args.causal == "1"
    ws, rank, local = dist_env()
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.backward:
            run_backward(args, w, causal)
        elif args.impl == "reference":
            run_reference(args, w, causal)
        else:
            run_ours(args, w, causal)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
