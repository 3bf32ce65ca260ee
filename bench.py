#!/usr/bin/env python3
"""Benchmark: direct conv2d forward (and the fused stencil) on one or more GPUs.

Workload of the headline line: the 3-layer upscaling-style net on one
1280x720 single-channel fp32 image (conv 5x5 1->32 + ReLU, conv 3x3 32->32
+ ReLU, conv 3x3 32->4), NHWC, synthetic seeded data and He-normal weights.
A step is one forward pass of the three layers; `value` is conv GFLOP/s
(2*N*H*W*Cin*Cout*R*S per layer), device-timed with CUDA events per step,
with L2 flushed between steps (a 256 MiB write, then a 256 MiB read of a
clean buffer, both outside the timed events: see L2Flush).
The line also carries Mpixel/s, a per-workload breakdown of all five
workloads, the roofline of the dominant kernel, the oracle's CPU timing,
an end-to-end number through host buffers, SM clocks during the timed
region and the number of kernel launches.

--impl reference times the fp64 CPU oracle on the machine's host cores on a
strip of the same workload (the same metric and unit).
Multi-GPU: one independent replica per rank (the path has no exchange).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv GFLOP/s and output Mpixel/s per config; % of FP32/HBM roofline"
WORKLOAD = "3-layer upscaling net, 1x1280x720 fp32 (5x5 1->32 ReLU, 3x3 32->32 ReLU, 3x3 32->4)"
L2_FLUSH_BYTES = 256 << 20
FP32_LANES_PER_SM = 128          # FP32 FMA lanes per Blackwell SM (4 schedulers x 32)


# --only cases: (workload id, layer index; None = the stencil pipeline)
ONLY_CASES = {
    "1": (1, 0), "2": (2, 0), "3-L1": (3, 0), "3-L2": (3, 1), "3-L3": (3, 2), "4": (4, 0), "5": (5, None),
    "4-tc": (4, 0), "3-L2-tc": (3, 1), "3-L3-tc": (3, 2),
    "4-bf16": (4, 0), "3-L2-bf16": (3, 1), "3-L3-bf16": (3, 2), "3-L23-fused": (3, 1),
    "4-x3": (4, 0), "3-L2-x3": (3, 1), "3-L3-x3": (3, 2),
    "S1": (4, "repack"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-per-config", action="store_true", help="skip the five-workload breakdown")
    ap.add_argument("--no-autotune", action="store_true", help="default tile configurations (no first-call tuning)")
    ap.add_argument("--only", choices=sorted(ONLY_CASES),
                    help="launch one workload's kernel warmup+steps times and exit (for ncu captures)")
    ap.add_argument("--candidate", type=int, default=None,
                    help="with --only on a 3x3 FP32 layer: that tile configuration of the autotuner's list")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device=None):
    """The largest of the ranks' values (the job's step time is its slowest
    rank's); `device` holds the reduction tensor (the GPU for NCCL, None =
    CPU for gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput: every rank processes units_per_rank per step of
    ms milliseconds (weak scaling, replicas)."""
    return world * units_per_rank / (ms * 1e-3)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return None


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_sources(L):
    """Source files that define the kernel a conv layer runs on (for the
    profile-staleness hash)."""
    c = "stencil_conv2d_fwd_gb300/csrc/"
    if L.cin == 1:
        return [c + "conv_c1.cu", c + "common.cuh"]
    if max(L.r, L.s) == 3:   # the TMA-staged kernels and the dispatch that picks them
        return [c + "conv_tma.cuh", c + "conv_tma_k3.cu", c + "common.cuh", c + "conv_general_k3.cu",
                c + "conv_general_k3n.cu", c + "conv_narrow.cuh", c + "conv_narrow_k3.cu", c + "conv_small.cu"]
    return [c + "conv_general.cuh", c + "common.cuh", c + f"conv_general_k{max(L.r, L.s)}.cu"]


def profiled_traffic(kernel_key: str, src_hash: str):
    """DRAM bytes per launch recorded from an ncu capture under profiles/, or
    None when absent or taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        for line in open(path):
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                if parts[1] == src_hash:
                    return float(parts[2])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# The GPU arm
# --------------------------------------------------------------------------


def conv_flops(n, h, w, L):
    return 2 * n * h * w * L.cin * L.cout * L.r * L.s


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import synthetic as S
    import stencil_conv2d_fwd_gb300 as sc

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    sc.load()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)
    n_sm = props.multi_processor_count
    peaks = measured_peaks() or {}
    sm_max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    fp32_peak_tflops = n_sm * FP32_LANES_PER_SM * 2 * sm_max_mhz * 1e6 / 1e12
    hbm_gbs = float(peaks.get("hbm_gbs", 6800.0))
    hbm_src = "measured" if "hbm_gbs" in peaks else "fallback"

    wl = S.config(3)
    N, H, W = wl.n, wl.h, wl.w
    layers = wl.layers
    flops_layer = [conv_flops(N, H, W, L) for L in layers]
    flops_step = sum(flops_layer)

    xd = torch.from_numpy(wl.x).to(dev)  # Cin = 1: NCHW == NHWC
    wds = [torch.from_numpy(L.w).to(dev) for L in layers]
    bds = [torch.from_numpy(L.b).to(dev) for L in layers]
    acts = [torch.empty(N * H * W * L.cout, device=dev) for L in layers]
    flush = L2Flush(torch, dev)

    def step(ev=None):
        src = xd
        for li, L in enumerate(layers):
            if ev is not None:
                ev[li][0].record(stream)
            rc = sc.conv2d_fwd(src, wds[li], bds[li], acts[li], N, H, W, L.cin, L.cout, L.r, L.s,
                               sc.SC_NHWC, L.act, stream)
            if rc != 0:
                raise RuntimeError(f"conv2d_fwd layer {li + 1}: {sc.sc_status_string(rc)}")
            if ev is not None:
                ev[li][1].record(stream)
            src = acts[li]

    # first-call autotuning of the tile configurations: the first warm-up
    # step times the candidates of each layer shape (outside the timed region)
    if not args.no_autotune:
        sc.sc_set_autotune(1)
    for _ in range(args.warmup):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    st = sc.sc_last_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {sc.sc_status_string(st)}")
    tuned = {}
    for li, L in enumerate(layers):
        names = sc.sc_autotune_candidates(L.cin, L.cout, L.r, L.s)
        c = sc.sc_autotune_lookup(N, H, W, L.cin, L.cout, L.r, L.s, L.act, True)
        tuned[f"layer {li + 1}"] = names[c] if 0 <= c < len(names) else "default (not tuned)"

    K = args.steps
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in layers] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        flush(float(k))                # evict L2: outside the per-step events
        step(ev[k])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    st = sc.sc_last_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {sc.sc_status_string(st)}")

    layer_ms = [[ev[k][li][0].elapsed_time(ev[k][li][1]) for k in range(K)] for li in range(len(layers))]
    step_ms = [ev[k][0][0].elapsed_time(ev[k][-1][1]) for k in range(K)]
    ms_step = max_over_ranks(sum(step_ms) / K, world, dev)
    value = job_rate(world, flops_step, ms_step) / 1e9
    mpix = job_rate(world, N * H * W, ms_step) / 1e6

    # dominant kernel: the layer with the largest mean time
    means = [sum(v) / K for v in layer_ms]
    dom = max(range(len(layers)), key=lambda i: means[i])
    Ld = layers[dom]
    dom_bytes = 4 * (N * H * W * (Ld.cin + Ld.cout) + Ld.w.size + Ld.b.size)
    achieved_tflops = flops_layer[dom] / (means[dom] * 1e-3) / 1e12
    key = f"conv_{Ld.cin}x{Ld.cout}_{Ld.r}x{Ld.s}_{W}x{H}"
    traffic = profiled_traffic(key, kernel_source_hash(kernel_sources(Ld)))
    roofline = {
        "kernel": f"conv2d_fwd layer {dom + 1} ({Ld.cin}->{Ld.cout}, {Ld.r}x{Ld.s}, {W}x{H})",
        "bound": "alu",
        "achieved": round(achieved_tflops, 3),
        "peak": round(fp32_peak_tflops, 2),
        "unit": "TFLOP/s",
        "frac": round(achieved_tflops / fp32_peak_tflops, 4),
        "traffic": traffic,
        "algorithmic_bytes": dom_bytes,
        "peak_note": (f"FP32 FFMA: {n_sm} SMs x {FP32_LANES_PER_SM} lanes x 2 FLOP x {sm_max_mhz:.0f} MHz "
                      "(max SM clock of MEASURED_PEAKS.json)"),
        "layer_ms": [round(m, 4) for m in means],
    }

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64; He-normal weights)",
        "config": {"workload": WORKLOAD, "layout": "NHWC", "flops_per_step": flops_step,
                   "l2": L2Flush.DESCRIPTION,
                   "parallelism": f"replicas x{world}"},
        "mpixel_per_s": round(mpix, 2),
        "wall_s_timed_region": round(wall, 4),
        "roofline": roofline,
        "clocks": clk,
        "gpu_launches": K * len(layers),
        "autotune": tuned if not args.no_autotune else "off",
    }

    # ---- end to end through the C-ABI call that takes host buffers
    # (conv2d_chain_fwd_host: pinned host image in, the three layers, host
    # output back), its copies inside the timed region
    x_host = torch.from_numpy(wl.x.copy()).pin_memory()
    y_host = torch.empty(N * H * W * layers[-1].cout, dtype=torch.float32).pin_memory()
    chain = [(wds[li], bds[li], L.cout, L.r, L.s, L.act) for li, L in enumerate(layers)]
    e2e_ms = []
    for k in range(args.warmup + K):
        flush(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rc = sc.conv2d_chain_fwd_host(x_host, y_host, N, H, W, layers[0].cin, chain, stream)
        if rc != 0:
            raise RuntimeError(f"conv2d_chain_fwd_host: {sc.sc_status_string(rc)}")
        e1.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_step = max_over_ranks(sum(e2e_ms) / K, world, dev)
    result["e2e"] = {"value": round(job_rate(world, flops_step, e2e_step) / 1e9, 2), "unit": "GFLOP/s",
                     "ms_per_step": round(e2e_step, 4), "api": "conv2d_chain_fwd_host (pinned host buffers)",
                     "h2d_bytes_per_step": x_host.numel() * 4, "d2h_bytes_per_step": y_host.numel() * 4}

    # ---- the five workloads, one line each inside the JSON
    if not args.no_per_config:
        result["per_config"] = per_config(sc, S, dev, stream, flush, fp32_peak_tflops, hbm_gbs, hbm_src)

    # ---- measured FP32 FMA rate and HBM copy bandwidth (context for the peaks)
    result["ffma_probe_tflops"] = ffma_probe(sc, dev, stream, n_sm)
    result["hbm_probe_gbs"] = hbm_probe(dev, stream)

    # ---- oracle on the host cores (rank 0 only)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, min_seconds=10.0)
        if not args.no_per_config:
            result["cpu_baseline"]["per_config"] = oracle_per_config(S)

    if "per_config" in result:
        # compact per-workload summary, last in the line: [ms mean, roofline frac, kernel ms, frac]
        result["per_config_summary"] = per_config_summary(result["per_config"])

    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def per_config_summary(pc):
    """{short name: [ms mean, roofline fraction]} of every timed entry of
    per_config, followed where measured by [kernel ms, roofline fraction]
    from time_in_graph and, for workloads 1 and 2, by the graph per-launch
    time and the launch floor in us."""
    tags = (("replayed as a CUDA graph", "graph"), ("split-TF32 tensor cores", "x3 net"),
            ("tcgen05 split TF32", "x3"), ("tcgen05 TF32", "tf32"), ("tcgen05 BF16", "bf16"))
    out = {}
    for name, e in pc.items():
        if name.startswith("_") or "ms_mean" not in e:
            continue
        short = name.split(":")[0] if ":" in name else name.split(" (")[0]
        for pat, tag in tags:
            if pat in name:
                short += " " + tag
                break
        v = [e["ms_mean"], e.get("roofline_frac")]
        if "ms_kernel" in e:
            v += [e["ms_kernel"], e["roofline_frac_kernel"]]
        if "graph_ms_per_launch" in e:
            v += [e["graph_ms_per_launch"], e.get("launch_floor_us")]
        out[short] = v
    return out


class L2Flush:
    """Evicts L2 (129 MB) between timed steps, outside the timed events.

    A write of a 256 MiB buffer alone leaves L2 full of dirty lines, and the
    next kernel then pays for writing them back to HBM (for the 4096x4096
    stencil that doubles its DRAM traffic).  So the write is followed by a
    read of a second 256 MiB buffer that is never written: the write-backs
    happen during that read, and the timed kernel starts from an L2 that
    holds none of its data and nothing dirty."""
    DESCRIPTION = ("flushed between steps: 256 MiB write, then a 256 MiB read of a clean buffer "
                   "(write-backs outside the timed events)")

    def __init__(self, torch, dev):
        self.wr = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
        self.rd = torch.zeros(L2_FLUSH_BYTES // 4, device=dev)

    def __call__(self, v):
        self.wr.fill_(v)
        self.rd.sum()


def time_events(fn, stream, flush, reps=40, warm=3):
    """(mean, min, median) of `reps` timed calls in ms, `flush` before each.

    CUDA-event timestamps on this GPU advance in steps of about 1.02 us, so a
    median of a few tens of microseconds sits on that grid; the mean over
    many calls does not, and is the figure the fractions are taken from."""
    import torch
    for _ in range(warm):
        flush(0.0)
        fn()
    ts = []
    for k in range(reps):
        flush(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return sum(ts) / len(ts), min(ts), statistics.median(ts)


def time_graph(fn, stream, launches=100, reps=5):
    """Per-launch time of `launches` back-to-back calls captured in one CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)
        torch.cuda.current_stream().synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(launches):
                fn(s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / launches)
    return min(ts)


def time_in_graph(fn, flush, stream, n=20, reps=3):
    """Per-call device time of fn(s) with L2 flushed before every call, in ms:
    one CUDA graph of n (flush, call) pairs against one of the n flushes
    alone, each replayed and timed with events; the difference over n.

    A start/end event pair around one call adds about 4 us on this GPU (a
    kernel that does nothing measures 4.7 us that way and 0.56 us a launch
    in a graph), so for the kernels of a few tens of microseconds the
    per-call event time overstates the kernel by 10-15%; this measure
    leaves the pair out while keeping the flush before every call."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graphs = []
    with torch.cuda.stream(s):
        fn(s)
        flush(0.0)
        torch.cuda.current_stream().synchronize()
        for with_fn in (True, False):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    flush(float(i))
                    if with_fn:
                        fn(s)
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(s)
    t = []
    for g in graphs:
        g.replay()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        t.append(best)
    return (t[0] - t[1]) / n


def per_config(sc, S, dev, stream, flush, fp32_tflops, hbm_gbs, hbm_src):
    import numpy as np
    import torch
    out = {}

    def no_flush(_v):
        pass

    def conv_entry(name, n, h, w, L, xin_nhwc, graph=False, warm=False):
        xd = torch.from_numpy(np.ascontiguousarray(xin_nhwc)).to(dev)
        wd = torch.from_numpy(L.w).to(dev)
        bd = torch.from_numpy(L.b).to(dev)
        yd = torch.empty(n * h * w * L.cout, device=dev)

        def call(s=None):
            rc = sc.conv2d_fwd(xd, wd, bd, yd, n, h, w, L.cin, L.cout, L.r, L.s, sc.SC_NHWC, L.act,
                               s if s is not None else stream)
            if rc != 0:
                raise RuntimeError(sc.sc_status_string(rc))
        med, mn, mdn = time_events(call, stream, flush)
        names = sc.sc_autotune_candidates(L.cin, L.cout, L.r, L.s)
        choice = sc.sc_autotune_lookup(n, h, w, L.cin, L.cout, L.r, L.s, L.act, True)
        flops = conv_flops(n, h, w, L)
        byts = 4 * (n * h * w * (L.cin + L.cout) + L.w.size + L.b.size)
        t_roof = max(flops / (fp32_tflops * 1e12), byts / (hbm_gbs * 1e9))
        bound = "alu" if flops / (fp32_tflops * 1e12) >= byts / (hbm_gbs * 1e9) else "hbm"
        e = {"ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
             "gflops": round(flops / (med * 1e-3) / 1e9, 2),
             "mpixel_per_s": round(n * h * w / (med * 1e-3) / 1e6, 2),
             "roofline_bound": bound, "roofline_us": round(t_roof * 1e6, 3),
             "roofline_frac": round(t_roof / (med * 1e-3), 4),
             "tile_config": names[choice] if 0 <= choice < len(names) else "default"}
        kern = time_in_graph(call, flush, stream)
        e["ms_kernel"] = round(kern, 5)
        e["roofline_frac_kernel"] = round(t_roof / (kern * 1e-3), 4)
        if graph:
            per = time_graph(call, stream)
            e["graph_ms_per_launch"] = round(per, 5)
            e["graph_roofline_frac"] = round(t_roof / (per * 1e-3), 4)
            e["launch_floor_us"] = floor_us
            e["graph_per_launch_vs_floor"] = round(per * 1e3 / floor_us, 3)
        if warm:   # back to back without the L2 flush (inputs partly L2-resident)
            wmed, _, _ = time_events(call, stream, no_flush)
            e["ms_mean_warm_l2"] = round(wmed, 5)
        out[name] = e
        return yd

    # the launch floor: a kernel that does nothing (one CTA of 128 threads per
    # SM), replayed back to back from the same CUDA-graph harness
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count

    def empty(s=None):
        sc.check(sc.sc_empty_kernel(n_sm, 128, s if s is not None else stream))
    floor_us = round(time_graph(empty, stream) * 1e3, 3)
    out["launch_floor"] = {"us_per_launch": floor_us,
                           "note": f"empty kernel, {n_sm} CTAs x 128 threads, 100 launches in one CUDA graph"}

    c1 = S.config(1)
    conv_entry("1: 64x64 1->1 3x3", 1, 64, 64, c1.layers[0], c1.x[0, 0], graph=True)
    c2 = S.config(2)
    conv_entry("2: 128x128 16->16 3x3", 1, 128, 128, c2.layers[0], c2.x.transpose(0, 2, 3, 1), graph=True)
    c3 = S.config(3)
    # layers of the net, each timed alone with its real input (the previous layer's output)
    prev = c3.x[0, 0]
    for li, L in enumerate(c3.layers):
        yd = conv_entry(f"3-L{li + 1}: 1280x720 {L.cin}->{L.cout} {L.r}x{L.s}", 1, 720, 1280, L, prev, warm=True)
        prev = yd.view(720, 1280, L.cout).cpu().numpy()
    c4 = S.config(4)
    conv_entry("4: N=32 56x56 64->64 3x3", 32, 56, 56, c4.layers[0], c4.x.transpose(0, 2, 3, 1), warm=True)

    # S1, the activation repack NCHW -> NHWC at workload 4's size (what
    # conv2d_fwd with SC_NCHW runs before the convolution): pure bandwidth
    rp_src = torch.from_numpy(np.ascontiguousarray(c4.x)).to(dev)
    rp_dst = torch.empty_like(rp_src)
    n4, c4c, h4, w4 = c4.x.shape

    def repack(s=None):
        sc.check(sc.sc_repack(rp_src, rp_dst, n4, c4c, h4, w4, sc.SC_NCHW, sc.SC_NHWC,
                              s if s is not None else stream))
    med, mn, mdn = time_events(repack, stream, flush)
    byts = 2 * 4 * rp_src.numel()
    out["S1: repack NCHW->NHWC N=32 64x56x56"] = {
        "ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
        "gbytes_per_s": round(byts / (med * 1e-3) / 1e9, 1),
        "roofline_bound": "hbm", "roofline_us": round(byts / (hbm_gbs * 1e9) * 1e6, 3),
        "roofline_frac": round(byts / (hbm_gbs * 1e9) / (med * 1e-3), 4),
        "note": "read and write of the 25.7 MB activation once each"}
    kern = time_in_graph(repack, flush, stream)
    out["S1: repack NCHW->NHWC N=32 64x56x56"].update(
        {"ms_kernel": round(kern, 5), "roofline_frac_kernel": round(byts / (hbm_gbs * 1e9) / (kern * 1e-3), 4)})

    # the FFMA net (the headline pass) captured once into a CUDA graph and
    # replayed: the same three kernels without the host's launch gaps between
    # the layers (L2 flushed before every replay, outside the events)
    n_px3 = 720 * 1280
    g_in = torch.from_numpy(np.ascontiguousarray(c3.x[0, 0])).to(dev)
    g_w = [(torch.from_numpy(L.w).to(dev), torch.from_numpy(L.b).to(dev)) for L in c3.layers]
    g_act = [g_in] + [torch.empty(n_px3 * L.cout, device=dev) for L in c3.layers]

    def net_calls(st_):
        for li, L in enumerate(c3.layers):
            rc = sc.conv2d_fwd(g_act[li], *g_w[li], g_act[li + 1], 1, 720, 1280, L.cin, L.cout, L.r, L.s,
                               sc.SC_NHWC, L.act, st_)
            if rc != 0:
                raise RuntimeError(sc.sc_status_string(rc))
    net_calls(stream)   # first calls (tensor maps, opt-ins) outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        net_calls(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    gmed, gmn, gmdn = time_events(lambda: graph.replay(), stream, flush)
    out["3: 3-layer net replayed as a CUDA graph"] = {
        "ms_mean": round(gmed, 5), "ms_median": round(gmdn, 5), "ms_min": round(gmn, 5),
        "gflops": round(sum(conv_flops(1, 720, 1280, L) for L in c3.layers) / (gmed * 1e-3) / 1e9, 2),
        "note": "the headline pass's three FFMA kernels without host launch gaps"}

    # tensor-core (tcgen05) variants, reported separately, each against the
    # TF32 tensor peak and HBM:
    #  * conv2d_fwd_tc: TF32 operands, its own tolerance (5e-3 * sum|x*w|);
    #  * conv2d_fwd_tc_x3: split TF32 (three TF32 products per product), the
    #    fp32 tolerance (1e-5 * sum|x*w|); its tensor work is 3x the FLOPs.
    peaks = measured_peaks() or {}
    tf32_tflops = float(peaks.get("bf16_tflops", 1900.0)) * 1.1 / 2.25
    variants = (("tcgen05 TF32", sc.conv2d_fwd_tc, 1, "5e-3 * sum|x*w| (TF32 operands)"),
                ("tcgen05 split TF32", sc.conv2d_fwd_tc_x3, 3,
                 "1e-5 * sum|x*w| (fp32 bound; x = hi + lo, w = hi + lo, three TF32 products)"))
    for vname, entry, work, tol in variants:
        for cname, cid, li in (("4", 4, 0), ("3-L2", 3, 1), ("3-L3", 3, 2)):
            wl = S.config(cid)
            L = wl.layers[li]
            xin = wl.x if li == 0 else np.maximum(S.uniform(77, 0, (wl.n, L.cin, wl.h, wl.w), -1, 1), 0)
            xd = torch.from_numpy(np.ascontiguousarray(xin.transpose(0, 2, 3, 1)).astype(np.float32)).to(dev)
            wd, bd = torch.from_numpy(L.w).to(dev), torch.from_numpy(L.b).to(dev)
            yd = torch.empty(wl.n * wl.h * wl.w * L.cout, device=dev)

            def call_tc(s=None):
                rc = entry(xd, wd, bd, yd, wl.n, wl.h, wl.w, L.cin, L.cout, L.r, L.s, L.act,
                           s if s is not None else stream)
                if rc != 0:
                    raise RuntimeError(sc.sc_status_string(rc))
            med, mn, mdn = time_events(call_tc, stream, flush)
            flops = conv_flops(wl.n, wl.h, wl.w, L)
            byts = 4 * (wl.n * wl.h * wl.w * (L.cin + L.cout) + L.w.size + L.b.size)
            t_c, t_m = work * flops / (tf32_tflops * 1e12), byts / (hbm_gbs * 1e9)
            out[f"{cname} ({vname})"] = {
                "ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
                "gflops": round(flops / (med * 1e-3) / 1e9, 2),
                "mpixel_per_s": round(wl.n * wl.h * wl.w / (med * 1e-3) / 1e6, 2),
                "roofline_bound": "tensor" if t_c >= t_m else "hbm",
                "roofline_us": round(max(t_c, t_m) * 1e6, 3),
                "roofline_frac": round(max(t_c, t_m) / (med * 1e-3), 4),
                "tolerance": tol,
                "tensor_flops_per_fp32_flop": work,
                "tf32_peak_tflops": round(tf32_tflops, 1)}
            kern = time_in_graph(call_tc, flush, stream)
            out[f"{cname} ({vname})"].update({"ms_kernel": round(kern, 5),
                                              "roofline_frac_kernel": round(max(t_c, t_m) / (kern * 1e-3), 4)})

    # bf16 activation storage with BF16 tensor-core operands (conv2d_fwd_tc_bf16):
    # x and y bf16 in HBM (the synthetic input rounded to bf16), fp32 filters and
    # bias; roofline against the measured BF16 peak and HBM
    bf16_tflops = float(peaks.get("bf16_tflops", 1900.0))
    for name, cid, li in (("4 (tcgen05 BF16, bf16 x/y)", 4, 0), ("3-L2 (tcgen05 BF16, bf16 x/y)", 3, 1),
                          ("3-L3 (tcgen05 BF16, bf16 x/y)", 3, 2)):
        wl = S.config(cid)
        L = wl.layers[li]
        xin = wl.x if li == 0 else np.maximum(S.uniform(77, 0, (wl.n, L.cin, wl.h, wl.w), -1, 1), 0)
        xd = torch.from_numpy(np.ascontiguousarray(xin.transpose(0, 2, 3, 1)).astype(np.float32)).to(dev)
        xd = xd.to(torch.bfloat16)
        wd, bd = torch.from_numpy(L.w).to(dev), torch.from_numpy(L.b).to(dev)
        yd = torch.empty(wl.n * wl.h * wl.w * L.cout, dtype=torch.bfloat16, device=dev)

        def call_bf(s=None):
            rc = sc.conv2d_fwd_tc_bf16(xd, wd, bd, yd, wl.n, wl.h, wl.w, L.cin, L.cout, L.r, L.s, L.act,
                                       sc.SC_BF16, s if s is not None else stream)
            if rc != 0:
                raise RuntimeError(sc.sc_status_string(rc))
        med, mn, mdn = time_events(call_bf, stream, flush)
        flops = conv_flops(wl.n, wl.h, wl.w, L)
        byts = 2 * wl.n * wl.h * wl.w * (L.cin + L.cout) + 4 * (L.w.size + L.b.size)
        t_c, t_m = flops / (bf16_tflops * 1e12), byts / (hbm_gbs * 1e9)
        out[name] = {"ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
                     "gflops": round(flops / (med * 1e-3) / 1e9, 2),
                     "mpixel_per_s": round(wl.n * wl.h * wl.w / (med * 1e-3) / 1e6, 2),
                     "roofline_bound": "tensor" if t_c >= t_m else "hbm",
                     "roofline_us": round(max(t_c, t_m) * 1e6, 3),
                     "roofline_frac": round(max(t_c, t_m) / (med * 1e-3), 4),
                     "tolerance": "5e-3 * sum|x*w| + 2^-8 |y| (bf16 operands and storage)",
                     "bf16_peak_tflops": round(bf16_tflops, 1)}
        kern = time_in_graph(call_bf, flush, stream)
        out[name].update({"ms_kernel": round(kern, 5),
                          "roofline_frac_kernel": round(max(t_c, t_m) / (kern * 1e-3), 4)})

    # layer fusion (f2): layers 2 and 3 of the net in one tensor-core pass,
    # the 32-channel intermediate kept on chip (TF32 operands)
    wl = S.config(3)
    L2, L3 = wl.layers[1], wl.layers[2]
    xin = np.maximum(S.uniform(77, 0, (wl.n, L2.cin, wl.h, wl.w), -1, 1), 0)
    xd = torch.from_numpy(np.ascontiguousarray(xin.transpose(0, 2, 3, 1)).astype(np.float32)).to(dev)
    w2d, b2d = torch.from_numpy(L2.w).to(dev), torch.from_numpy(L2.b).to(dev)
    w3d, b3d = torch.from_numpy(L3.w).to(dev), torch.from_numpy(L3.b).to(dev)
    yd = torch.empty(wl.n * wl.h * wl.w * L3.cout, device=dev)

    def call_fused(s=None):
        rc = sc.conv2d_fwd_tc_fused2(xd, w2d, b2d, w3d, b3d, yd, wl.n, wl.h, wl.w, L2.cin, L2.cout, L3.cout,
                                     L2.act, L3.act, s if s is not None else stream)
        if rc != 0:
            raise RuntimeError(sc.sc_status_string(rc))
    med, mn, mdn = time_events(call_fused, stream, flush)
    flops = conv_flops(wl.n, wl.h, wl.w, L2) + conv_flops(wl.n, wl.h, wl.w, L3)
    byts = 4 * (wl.n * wl.h * wl.w * (L2.cin + L3.cout) + L2.w.size + L2.b.size + L3.w.size + L3.b.size)
    t_c, t_m = flops / (tf32_tflops * 1e12), byts / (hbm_gbs * 1e9)
    out["3-L2+3-L3 fused (tcgen05 TF32)"] = {
        "ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
        "gflops": round(flops / (med * 1e-3) / 1e9, 2),
        "mpixel_per_s": round(wl.n * wl.h * wl.w / (med * 1e-3) / 1e6, 2),
        "roofline_bound": "tensor" if t_c >= t_m else "hbm",
        "roofline_us": round(max(t_c, t_m) * 1e6, 3),
        "roofline_frac": round(max(t_c, t_m) / (med * 1e-3), 4),
        "note": "FLOP and bytes are the two layers' algorithmic counts; the intermediate never reaches HBM"}

    # the whole 3-layer net with its two 32-channel-input layers on the
    # split-TF32 tensor-core path, which meets the same fp32 bound
    # (1e-5 * sum|x*w|); layer 1 (one input channel) stays on conv2d_fwd.
    # Reported separately; the headline value is the FFMA path.
    wl = S.config(3)
    L1, L2, L3 = wl.layers
    n_px = wl.n * wl.h * wl.w
    x0 = torch.from_numpy(np.ascontiguousarray(wl.x.transpose(0, 2, 3, 1))).to(dev)
    wds = [(torch.from_numpy(L.w).to(dev), torch.from_numpy(L.b).to(dev)) for L in (L1, L2, L3)]
    a1 = torch.empty(n_px * L1.cout, device=dev)
    a2 = torch.empty(n_px * L2.cout, device=dev)
    a3 = torch.empty(n_px * L3.cout, device=dev)

    def call_net_x3(s=None):
        st_ = s if s is not None else stream
        for rc in (sc.conv2d_fwd(x0, *wds[0], a1, wl.n, wl.h, wl.w, L1.cin, L1.cout, L1.r, L1.s, sc.SC_NHWC, L1.act,
                                 st_),
                   sc.conv2d_fwd_tc_x3(a1, *wds[1], a2, wl.n, wl.h, wl.w, L2.cin, L2.cout, L2.r, L2.s, L2.act, st_),
                   sc.conv2d_fwd_tc_x3(a2, *wds[2], a3, wl.n, wl.h, wl.w, L3.cin, L3.cout, L3.r, L3.s, L3.act, st_)):
            if rc != 0:
                raise RuntimeError(sc.sc_status_string(rc))
    med, mn, mdn = time_events(call_net_x3, stream, flush)
    flops = sum(conv_flops(wl.n, wl.h, wl.w, L) for L in (L1, L2, L3))
    out["3: 3-layer net, layers 2 and 3 on split-TF32 tensor cores"] = {
        "ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
        "gflops": round(flops / (med * 1e-3) / 1e9, 2),
        "mpixel_per_s": round(n_px / (med * 1e-3) / 1e6, 2),
        "tolerance": "1e-5 * sum|x*w| per layer (the fp32 bound of every layer)",
        "note": "layer 1 on the FFMA kernel; same FLOP count as the headline pass"}

    c5 = S.config(5)
    ind = torch.from_numpy(c5.img).to(dev)
    outd = torch.empty_like(ind)

    def pipe(s=None):
        rc = sc.stencil_pipeline_fwd(ind, outd, c5.h, c5.w, s if s is not None else stream)
        if rc != 0:
            raise RuntimeError(sc.sc_status_string(rc))
    med, mn, mdn = time_events(pipe, stream, flush)
    wmed, _, _ = time_events(pipe, stream, no_flush)
    byts = 8 * c5.h * c5.w
    t_roof = byts / (hbm_gbs * 1e9)
    out["5: 4096x4096 fused blur/unsharp"] = {
        "ms_mean": round(med, 5), "ms_median": round(mdn, 5), "ms_min": round(mn, 5),
        "mpixel_per_s": round(c5.h * c5.w / (med * 1e-3) / 1e6, 2),
        "gbytes_per_s": round(byts / (med * 1e-3) / 1e9, 1),
        "roofline_bound": "hbm", "roofline_us": round(t_roof * 1e6, 3),
        "roofline_frac": round(t_roof / (med * 1e-3), 4),
        "ms_mean_warm_l2": round(wmed, 5)}
    kern = time_in_graph(pipe, flush, stream)
    out["5: 4096x4096 fused blur/unsharp"].update(
        {"ms_kernel": round(kern, 5), "roofline_frac_kernel": round(t_roof / (kern * 1e-3), 4)})
    out["_peaks"] = {"fp32_tflops": round(fp32_tflops, 2), "hbm_gbs": hbm_gbs, "hbm_source": hbm_src,
                     "fp32_source": "nominal: SMs x 128 FP32 lanes x 2 x max SM clock"}
    return out


def hbm_probe(dev, stream, nbytes=1 << 30, reps=5):
    """Device-to-device copy of nbytes (2 x nbytes of HBM traffic per copy;
    buffers 8x the L2), best of reps: context for the measured HBM peak."""
    import torch
    src = torch.ones(nbytes // 4, device=dev)
    dst = torch.empty_like(src)
    dst.copy_(src)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(src)
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del src, dst
    return round(2 * nbytes / (best * 1e-3) / 1e9, 1)


def ffma_probe(sc, dev, stream, n_sm):
    import torch
    blocks, iters = n_sm * 8, 4096
    sink = torch.empty(blocks * 256, device=dev)
    for _ in range(2):
        sc.check(sc.sc_measure_ffma_peak(sink, blocks, iters, stream))
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sc.check(sc.sc_measure_ffma_peak(sink, blocks, iters, stream))
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return round(blocks * 256 * iters * 16 * 2 / (best * 1e-3) / 1e12, 2)


# --------------------------------------------------------------------------
# CPU oracle timing (our arm's cpu_baseline, and the reference arm)
# --------------------------------------------------------------------------


def oracle_net_pass(oracle, wl, rows):
    """The oracle's forward pass of the net over a strip of `rows` image rows
    (the strip treated as a rows x 1280 image: the same per-pixel work)."""
    x = wl.x[:, :, :rows, :]
    for L in wl.layers:
        y, _ = oracle.conv2d_nchw(x, L.w, L.b, L.act, with_scale=False)
        x = y.astype("float32")
    return wl.n * rows * wl.w


def cpu_baseline(wl, min_seconds=10.0, rows=None):
    import oracle
    cores = oracle.set_threads(0)
    rows = rows or wl.h
    flops_px = sum(2 * L.cin * L.cout * L.r * L.s for L in wl.layers)
    t0 = time.perf_counter()
    px = 0
    passes = 0
    while True:
        px += oracle_net_pass(oracle, wl, rows)
        passes += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(px * flops_px / dt / 1e9, 3), "unit": "GFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} pass(es) of the 3-layer net over {rows} of 720 rows x 1280 (fp64 C oracle, "
                      f"OpenMP), {dt:.1f} s"}


def oracle_per_config(S, min_seconds=0.5):
    """The oracle on every workload, on the machine's host cores: all OpenMP
    threads for every workload and one thread for workloads 1, 2 and 5, each
    on a bounded sample (whole images for 1 and 2, one image of the batch
    for 4, a row strip for 3 and 5), repeated for at least min_seconds.
    Output Mpixel/s (and GFLOP/s for the convolutions)."""
    import oracle
    cores = oracle.set_threads(0)

    def timed(fn):
        n, t0 = 0, time.perf_counter()
        while True:
            px = fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                return n * px / dt, n, dt

    def conv_sample(wl, images=None):
        x = wl.x if images is None else wl.x[:images]
        L = wl.layers[0]

        def fn():
            oracle.conv2d_nchw(x, L.w, L.b, L.act, with_scale=False)
            return x.shape[0] * wl.h * wl.w
        return fn, 2 * L.cin * L.cout * L.r * L.s

    w3 = S.config(3)
    w5 = S.config(5)
    strip5 = 64
    cases = {
        "1": (*conv_sample(S.config(1)), "the 64x64 image", True),
        "2": (*conv_sample(S.config(2)), "the 128x128 image", True),
        "3": (lambda: oracle_net_pass(oracle, w3, 16), sum(2 * L.cin * L.cout * L.r * L.s for L in w3.layers),
              "a 16-row strip of the 3-layer net", False),
        "4": (*conv_sample(S.config(4), images=1), "one 56x56 image of the 32", False),
        "5": (lambda: (oracle.stencil_pipeline(w5.img, rows=(0, strip5)), strip5 * w5.w)[1], None,
              f"a {strip5}-row strip of the 4096x4096 image", True),
    }
    out = {}
    for name, (fn, flops_px, sample, single) in cases.items():
        runs = [(cores, "openmp")] + ([(1, "1 thread")] if single else [])
        ent = {"sample": sample}
        for threads, tag in runs:
            oracle.set_threads(threads)
            px_s, n, dt = timed(fn)
            r = {"mpixel_per_s": round(px_s / 1e6, 4), "threads": threads, "calls": n, "seconds": round(dt, 2)}
            if flops_px:
                r["gflops"] = round(px_s * flops_px / 1e9, 3)
            ent[tag] = r
        oracle.set_threads(cores)
        out[name] = ent
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    import synthetic as S
    import oracle
    wl = S.config(3)
    cores = oracle.set_threads(0)
    rows = 90                               # one eighth of the image per step
    flops_px = sum(2 * L.cin * L.cout * L.r * L.s for L in wl.layers)
    for _ in range(args.warmup):
        oracle_net_pass(oracle, wl, rows)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        px = oracle_net_pass(oracle, wl, rows)
        ts.append(time.perf_counter() - t0)
    ms = 1e3 * sum(ts) / len(ts)
    value = px * flops_px / (ms * 1e-3) / 1e9
    sample = f"a {rows}-row strip (of 720) x 1280 of the 3-layer net per step, fp64 C oracle on {cores} threads"
    print(json.dumps({
        "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64; He-normal weights)",
        "config": {"workload": WORKLOAD, "layout": "NCHW (oracle)", "sample_rows": rows},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_only(args, local):
    """One workload's kernel, launched warmup + steps times on real inputs
    (the layer's input is the previous layer's output), for profilers."""
    import numpy as np
    import torch

    import synthetic as S
    import stencil_conv2d_fwd_gb300 as sc

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    sc.load()
    cid, li = ONLY_CASES[args.only]
    wl = S.config(cid)
    if li == "repack":   # S1: the NCHW -> NHWC repack of the workload's input
        src = torch.from_numpy(np.ascontiguousarray(wl.x)).to(dev)
        dst = torch.empty_like(src)
        n_, c_, h_, w_ = wl.x.shape
        launch = lambda: sc.sc_repack(src, dst, n_, c_, h_, w_, sc.SC_NCHW, sc.SC_NHWC)
    elif li is None:
        ind = torch.from_numpy(wl.img).to(dev)
        outd = torch.empty_like(ind)
        launch = lambda: sc.stencil_pipeline_fwd(ind, outd, wl.h, wl.w)
    else:
        N, H, W = wl.n, wl.h, wl.w
        x = torch.from_numpy(np.ascontiguousarray(wl.x.transpose(0, 2, 3, 1))).to(dev)
        for k in range(li + 1):   # earlier layers produce this layer's input
            L = wl.layers[k]
            wd, bd = torch.from_numpy(L.w).to(dev), torch.from_numpy(L.b).to(dev)
            y = torch.empty(N * H * W * L.cout, device=dev)
            if k < li:
                sc.check(sc.conv2d_fwd(x, wd, bd, y, N, H, W, L.cin, L.cout, L.r, L.s, sc.SC_NHWC, L.act))
                x = y
        if args.only.endswith("-tc"):   # the tensor-core (TF32) variant
            launch = lambda: sc.conv2d_fwd_tc(x, wd, bd, y, N, H, W, L.cin, L.cout, L.r, L.s, L.act)
        elif args.only.endswith("-x3"):   # the split-TF32 tensor-core variant
            launch = lambda: sc.conv2d_fwd_tc_x3(x, wd, bd, y, N, H, W, L.cin, L.cout, L.r, L.s, L.act)
        elif args.only == "3-L23-fused":   # layers 2 and 3 fused on the tensor cores
            L3 = wl.layers[2]
            w3d, b3d = torch.from_numpy(L3.w).to(dev), torch.from_numpy(L3.b).to(dev)
            y3 = torch.empty(N * H * W * L3.cout, device=dev)
            launch = lambda: sc.conv2d_fwd_tc_fused2(x, wd, bd, w3d, b3d, y3, N, H, W, L.cin, L.cout, L3.cout,
                                                     L.act, L3.act)
        elif args.only.endswith("-bf16"):   # bf16 storage, BF16 tensor-core operands
            xb = x.to(torch.bfloat16)
            yb = torch.empty(N * H * W * L.cout, dtype=torch.bfloat16, device=dev)
            launch = lambda: sc.conv2d_fwd_tc_bf16(xb, wd, bd, yb, N, H, W, L.cin, L.cout, L.r, L.s, L.act,
                                                   sc.SC_BF16)
        elif args.candidate is not None:   # one tile configuration of the autotuner's list
            launch = lambda: sc.sc_test_conv_candidate(x, wd, bd, y, N, H, W, L.cin, L.cout, L.r, L.s, L.act,
                                                       args.candidate)
        else:
            launch = lambda: sc.conv2d_fwd(x, wd, bd, y, N, H, W, L.cin, L.cout, L.r, L.s, sc.SC_NHWC, L.act)
    for _ in range(args.warmup + args.steps):
        sc.check(launch())
    torch.cuda.synchronize()
    sc.check(sc.sc_last_device_status())
    print(f"only {args.only}: {args.warmup + args.steps} launches ok")


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.only:
        run_only(args, local)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
