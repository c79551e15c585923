#!/usr/bin/env python
"""Throughput of the NVFP4 projection on GB300 -- one JSON line on stdout (rank 0).

Workload (the decode case the metric is quoted on): M = 1 W4A16 NVFP4 linear on the two
decode shapes (K=5120, N=17408) and (K=17408, N=5120), y bf16, synthetic seeded data.
One step = one call of each shape.  Metric: algorithmic GB/s = (packed nibbles + E4M3
scales + x + y + global scale) bytes / time.  Inputs stay resident in HBM; the weights
rotate over several copies (> 2x L2 in total) so every call streams from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the reference arm) on a bounded
sample of the same workload.  Under torchrun with N > 1 every rank runs an independent
replica ("replicas only": the projection needs no exchange); value = all ranks' bytes
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 linear: GB/s (M≤16) & TFLOP/s (M≥512), % of GB300 roofline"
DECODE = ("decode_a", "decode_b")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "gemv_w4a16_decode_traffic.txt")


FP4_NOMINAL_TFLOPS = 13500.0  # dense FP4 tensor peak of a GB300 (nominal, not measured)



# set from --static-weights: the decode/verify calls pass NVFP4_STATIC_WEIGHTS
STATIC_W = False

def max_over_ranks(ms: float, dist, device: str) -> float:
    """The job's duration: the largest of the ranks' timed regions (every rank leaves the
    region through a barrier, so the slowest replica ends it).  `dist` is None for one
    process; `device` is where the collective's tensor lives ("cuda" for NCCL, "cpu" for
    gloo)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_step: int, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: the bytes every replica streamed over the job's duration."""
    return bytes_per_step * steps * world / (ms * 1e-3) / 1e9


def algo_bytes(M, K, N, y_bytes=2):
    return N * K // 2 + N * K // 16 + M * K * 2 + M * N * y_bytes + 4


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# ---- clocks during the timed region ------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [p.strip() for p in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---- our arm -----------------------------------------------------------------------------

class DecodeSetup:
    """Quantized weights (several copies), x and y for the two decode shapes."""

    def __init__(self, nv, torch, copies: int):
        from synth import WORKLOADS, workload_inputs
        self.shapes = []
        for name in DECODE:
            wl = WORKLOADS[name]
            x, w = workload_inputs(name)
            packed, _, swz, g = nv.quantize_weight(w.cuda())
            del w
            cps = [(packed, swz)] + [(packed.clone(), swz.clone()) for _ in range(copies - 1)]
            ys = [torch.empty(1, wl.N, dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
            ws = torch.zeros(nv.nvfp4_workspace_bytes(1, 1, wl.K, wl.N), dtype=torch.uint8,
                             device="cuda")
            self.shapes.append(dict(name=name, M=1, K=wl.K, N=wl.N, x=x.cuda(), x_host=x,
                                    g=g, copies=cps, ys=ys, ws=ws))
        torch.cuda.synchronize()
        self.copies = copies
        self.bytes_per_step = sum(algo_bytes(s["M"], s["K"], s["N"]) for s in self.shapes)
        self.bytes_per_launch = [algo_bytes(s["M"], s["K"], s["N"]) for s in self.shapes]


def hold_stream(torch, cycles: int = 200_000):
    """About 0.1 ms of device-side sleep on the current stream (nothing else runs)."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(cycles)


def capture(torch, fn, nsteps):
    """CUDA graph of nsteps calls of fn(step_index)."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(nsteps):  # warm the path outside the capture
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(nsteps):
            fn(i)
    torch.cuda.synchronize()
    return g


def run_ours(args, rank, world, dist):
    import torch

    import nvfp4_weight_quantized_quantize_gb300 as nv
    from nvfp4_weight_quantized_quantize_gb300 import build_lib

    build_lib.build()
    nv.load()
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    setup = DecodeSetup(nv, torch, args.copies)
    S = setup.shapes

    def step(i, events=None):
        c = i % setup.copies
        for j, s in enumerate(S):
            if events is not None:
                events[2 * j].record()
            nv.nvfp4_linear(s["x"], s["copies"][c][0], s["copies"][c][1], s["g"], s["ys"][c],
                            workspace=s["ws"], static_weights=STATIC_W)
            if events is not None:
                events[2 * j + 1].record()

    # timed region: every one of the K steps runs as a CUDA-graph replay of the production
    # path (a graph of G steps replayed K // G times, then a graph of the K % G remaining
    # steps), so each launch runs back to back with its programmatic-launch overlap
    G = min(args.steps, 256)
    reps, tail = divmod(args.steps, G)
    graph = capture(torch, step, G)
    graph_tail = capture(torch, lambda i: step(reps * G + i), tail) if tail else None

    for i in range(max(args.warmup, 3)):
        step(i)
    graph.replay()
    if graph_tail:
        graph_tail.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, dev)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.4)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # a short device-side sleep keeps the stream busy while the host enqueues the start
    # event and the graph launches, so the region starts with the graph already queued
    # (the graph launch latency of the host is not device time); nothing of the step runs
    # before t0
    hold_stream(torch)
    t0.record()
    for _ in range(reps):
        graph.replay()
    if graph_tail:
        graph_tail.replay()
    t1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    ms = t0.elapsed_time(t1)
    ms_local = ms
    ms = max_over_ranks(ms, dist, "cuda")
    value = job_gbps(setup.bytes_per_step, args.steps, world, ms)

    # per-launch durations of eager launches bracketed by CUDA events, outside the timed
    # region (events between launches break the programmatic-launch overlap, so these
    # read longer than the launches of the graph)
    EV = 8
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(S))] for _ in range(EV)]
    for i in range(EV):
        step(i, ev[i])
    torch.cuda.synchronize()
    launch_ms = [e[2 * j].elapsed_time(e[2 * j + 1]) for e in ev for j in range(len(S))]

    # end to end: host x -> device, both calls, y -> host, every step
    e2e = run_e2e(torch, nv, setup, args)

    out = None
    if rank == 0:
        pk, pk_src = peaks()
        # a step is nothing but launches of the GEMV kernel, so the kernel's average launch
        # duration is the timed region / launches; the launches run back to back (each may
        # start its prologue under the previous one's tail).  Eager launches bracketed by
        # events are reported beside it.
        eager_launch_s = statistics.mean(launch_ms) * 1e-3
        avg_launch_s = ms_local * 1e-3 / (args.steps * len(S))
        achieved = statistics.mean(setup.bytes_per_launch) / avg_launch_s / 1e9
        traffic = read_traffic()
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) x, N(0,0.02) W with 0.1% x20 outliers)",
            "config": {"workload": "decode M=1 W4A16 NVFP4: (K=5120,N=17408) + "
                                   "(K=17408,N=5120), y bf16",
                       "operands": "e2m1 weights + e4m3 per-16 scales + fp32 global, bf16 x, "
                                   "fp32 accumulate",
                       "static_weights": STATIC_W,
                       "bytes_per_step": setup.bytes_per_step,
                       "l2": "inputs larger than L2: %d rotating weight copies (%.0f MB)"
                             % (setup.copies, setup.bytes_per_step * setup.copies / 1e6),
                       "parallelism": "replicas only (dp%d)" % world,
                       "timing": "every timed step a CUDA-graph replay: a graph of %d steps "
                                 "replayed %d times%s, queued behind a device-side sleep "
                                 "so that the region starts with the graph in the queue"
                                 % (G, reps, (" + a graph of the %d remaining steps" % tail)
                                    if tail else "")},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / pk["hbm_gbs"], 4),
                         "traffic": traffic, "peak_source": pk_src,
                         "kernel": "gemv_m1_pipe_kernel",
                         "launch_us": round(avg_launch_s * 1e6, 2),
                         "launch_timing": "timed region (CUDA-graph replays) / launches",
                         "eager_launch_us": round(eager_launch_s * 1e6, 2)},
            "e2e": e2e,
            "gpu_launches": len(S) * args.steps,
            "clocks": clocks,
        }
        if args.rows:
            # the secondary rows run after the headline is measured; a failure among them
            # is reported in the line instead of costing the line
            try:
                out["rows"] = measure_rows(torch, nv, setup)
            except Exception as exc:
                out["rows_error"] = "%s: %s" % (type(exc).__name__, exc)
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return out


def run_e2e(torch, nv, setup, args):
    S = setup.shapes
    # the step's inputs (both projections' x) sit in one pinned host buffer and go over in
    # one copy; both outputs come back in one copy
    ks = [s["K"] for s in S]
    ns = [s["N"] for s in S]
    xh = torch.cat([s["x_host"].reshape(-1) for s in S]).pin_memory()
    yh = torch.empty(sum(ns), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty(sum(ks), dtype=torch.bfloat16, device="cuda")
    yd = torch.empty(sum(ns), dtype=torch.bfloat16, device="cuda")
    xv = [xd[sum(ks[:j]):sum(ks[:j + 1])].view(1, -1) for j in range(len(S))]
    yv = [yd[sum(ns[:j]):sum(ns[:j + 1])].view(1, -1) for j in range(len(S))]

    def step(i):
        c = i % setup.copies
        xd.copy_(xh, non_blocking=True)
        for j, s in enumerate(S):
            nv.nvfp4_linear(xv[j], s["copies"][c][0], s["copies"][c][1], s["g"], yv[j],
                            workspace=s["ws"], static_weights=STATIC_W)
        yh.copy_(yd, non_blocking=True)

    # at least 256 steps (a region of several ms), queued behind a device-side sleep like
    # the headline's region, so that host launch jitter does not enter the figure
    n = min(max(args.steps, 256), 2048)
    G = min(n, 32)
    while n % G:
        G -= 1
    graph = capture(torch, step, G)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    hold_stream(torch)
    t0.record()
    for _ in range(n // G):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    h2d = xh.numel() * 2
    d2h = yh.numel() * 2
    return {"value": round(setup.bytes_per_step * n / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n}


def time_graph(torch, fn, nsteps, reps):
    g = capture(torch, fn, nsteps)
    g.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / (nsteps * reps)  # ms per call


def measure_rows(torch, nv, setup):
    """Per-row throughput of the other hot-path steps (outside the timed region)."""
    from synth import WORKLOADS, random_x, workload_inputs
    rows = {}
    # a1 quantize (fp32 weights) and a2 repack, decode_a shape
    s = setup.shapes[0]
    _, w = workload_inputs("decode_a")
    wd = w.cuda()
    N, K = wd.shape
    packed = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(N, K // 16, dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.nvfp4_workspace_bytes(0, N, K), dtype=torch.uint8, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_quantize(wd, packed, scales, g, ws), 4, 5)
    qbytes = N * K * 4 + N * K // 2 + N * K // 16 + 4
    rows["a1_quantize_fp32_17408x5120"] = {"GB/s": round(qbytes / ms / 1e6, 1),
                                           "us": round(ms * 1e3, 1)}
    swz = torch.empty(nv.nvfp4_repack_bytes(N, K), dtype=torch.uint8, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_repack(scales, K, swz), 8, 5)
    rows["a2_repack_17408x5120"] = {"GB/s": round(2 * N * K / 16 / ms / 1e6, 1),
                                    "us": round(ms * 1e3, 1)}
    del wd
    # FP8 (E4M3, block-128) checkpoint -> BF16 -> NVFP4 on the same shape; 3 rotating
    # copies of the FP8 input (267 MB > L2)
    from synth import random_fp8_block128
    q8, s8 = random_fp8_block128(N, K, 1)
    q8d = [torch.from_numpy(q8).cuda() for _ in range(3)]
    s8d = torch.from_numpy(s8).cuda()
    ms = time_graph(torch, lambda i: nv.nvfp4_quantize_fp8_block128(q8d[i % 3], s8d, packed,
                                                                    scales, g, ws), 6, 5)
    fb = N * K + s8.size * 4 + N * K // 2 + N * K // 16 + 4
    rows["f3_fp8_block128_to_nvfp4_17408x5120"] = {"GB/s": round(fb / ms / 1e6, 1),
                                                   "us": round(ms * 1e3, 1)}
    del q8d
    for sh in setup.shapes:
        ms = time_graph(torch, lambda i, sh=sh: nv.nvfp4_linear(
            sh["x"], sh["copies"][i % setup.copies][0], sh["copies"][i % setup.copies][1],
            sh["g"], sh["ys"][i % setup.copies], workspace=sh["ws"], static_weights=STATIC_W),
            4 * setup.copies, 50)
        b = algo_bytes(1, sh["K"], sh["N"])
        rows["a3_decode_%s_K%d_N%d" % (sh["name"], sh["K"], sh["N"])] = {
            "GB/s": round(b / ms / 1e6, 1), "us": round(ms * 1e3, 2)}
    # a4 verify M=7 (W quantized on the GPU; 3 copies of the large shape)
    for name in ("verify_a", "verify_b"):
        wl = WORKLOADS[name]
        x, w = workload_inputs(name)
        p, _, z, gg = nv.quantize_weight(w.cuda())
        del w
        ncp = 3 if wl.N > 10000 else 12
        cps = [(p, z)] + [(p.clone(), z.clone()) for _ in range(ncp - 1)]
        xd = x.cuda()
        y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
        wsv = torch.zeros(nv.nvfp4_workspace_bytes(1, wl.M, wl.K, wl.N), dtype=torch.uint8,
                          device="cuda")
        ms = time_graph(torch, lambda i: nv.nvfp4_linear(xd, cps[i % ncp][0], cps[i % ncp][1],
                                                         gg, y, workspace=wsv,
                                                         static_weights=STATIC_W), 2 * ncp, 20)
        b = algo_bytes(wl.M, wl.K, wl.N)
        rows["a4_verify_%s_M7_K%d_N%d" % (name, wl.K, wl.N)] = {
            "GB/s": round(b / ms / 1e6, 1), "us": round(ms * 1e3, 2)}
        del cps, p, z
    # W4A4 at decode (decode_a weights, 4 copies): a static activation scale quantizes x
    # inside the GEMV; a dynamic one runs the amax and quantize passes first
    sh = setup.shapes[0]
    wsa = torch.zeros(nv.nvfp4_workspace_bytes(1, 1, sh["K"], sh["N"], nv.NVFP4_W4A4),
                      dtype=torch.uint8, device="cuda")
    gxs = torch.tensor([0.004], dtype=torch.float32, device="cuda")
    for tag, gxa in (("static_fused", gxs), ("dynamic", None)):
        ms = time_graph(torch, lambda i, gxa=gxa: nv.nvfp4_linear(
            sh["x"], sh["copies"][i % setup.copies][0], sh["copies"][i % setup.copies][1],
            sh["g"], sh["ys"][i % setup.copies], mode="w4a4", x_global_scale=gxa,
            workspace=wsa, static_weights=STATIC_W), 4 * setup.copies, 50)
        b = algo_bytes(1, sh["K"], sh["N"])
        rows["f2_w4a4_%s_M1_K%d_N%d" % (tag, sh["K"], sh["N"])] = {
            "GB/s": round(b / ms / 1e6, 1), "us": round(ms * 1e3, 2)}
    # the small-M curve: M = 1 .. 16 on the verify_a weights (K 5120, N 34816; 3 copies)
    wl = WORKLOADS["verify_a"]
    _, w = workload_inputs("verify_a")
    p, _, z, gg = nv.quantize_weight(w.cuda())
    del w
    cps = [(p, z)] + [(p.clone(), z.clone()) for _ in range(2)]
    curve = {}
    for m in range(1, 17):
        xd = random_x(m, wl.K, 40 + m).cuda()
        y = torch.empty(m, wl.N, dtype=torch.bfloat16, device="cuda")
        wsv = torch.zeros(nv.nvfp4_workspace_bytes(1, m, wl.K, wl.N), dtype=torch.uint8,
                          device="cuda")
        ms = time_graph(torch, lambda i: nv.nvfp4_linear(xd, cps[i % 3][0], cps[i % 3][1], gg,
                                                         y, workspace=wsv,
                                                         static_weights=STATIC_W), 6, 10)
        curve["M%d" % m] = round(algo_bytes(m, wl.K, wl.N) / ms / 1e6, 1)
    rows["f4_small_m_curve_K%d_N%d_GBps" % (wl.K, wl.N)] = curve
    del cps, p, z
    # a wide output (an lm-head-sized N = 151936, K 5120) at M = 1: one 438 MB copy > L2;
    # weights drawn on the device (same N(0, 0.02) recipe, device generator)
    Nw, Kw = 151936, 5120
    gen = torch.Generator(device="cuda").manual_seed(9)
    w = torch.randn(Nw, Kw, generator=gen, device="cuda", dtype=torch.float32) * 0.02
    p, _, z, gg = nv.quantize_weight(w)
    del w
    xd = random_x(1, Kw, 9).cuda()
    y = torch.empty(1, Nw, dtype=torch.bfloat16, device="cuda")
    wsv = torch.zeros(nv.nvfp4_workspace_bytes(1, 1, Kw, Nw), dtype=torch.uint8, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_linear(xd, p, z, gg, y, workspace=wsv,
                                                     static_weights=STATIC_W), 4, 10)
    b = algo_bytes(1, Kw, Nw)
    rows["f4_wide_n_M1_K%d_N%d" % (Kw, Nw)] = {"GB/s": round(b / ms / 1e6, 1),
                                               "us": round(ms * 1e3, 2)}
    del p, z
    # a5 prefill M=512 W4A16 on the tensor cores (2 weight copies, inputs > L2)
    pk, _ = peaks()
    for name in ("prefill_a", "prefill_b"):
        wl = WORKLOADS[name]
        x, w = workload_inputs(name)
        p, _, z, gg = nv.quantize_weight(w.cuda())
        del w
        cps = [(p, z), (p.clone(), z.clone())]
        xd = x.cuda()
        y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
        wsv = torch.zeros(nv.nvfp4_workspace_bytes(1, wl.M, wl.K, wl.N), dtype=torch.uint8,
                          device="cuda")
        ms = time_graph(torch, lambda i: nv.nvfp4_linear(xd, cps[i % 2][0], cps[i % 2][1],
                                                         gg, y, workspace=wsv), 4, 5)
        tf = 2.0 * wl.M * wl.N * wl.K / (ms * 1e-3) / 1e12
        rows["a5_prefill_%s_M%d_K%d_N%d" % (name, wl.M, wl.K, wl.N)] = {
            "TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 1),
            "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4)}
        del cps, p, z
    # the fused MLP activation on a 512-token chunk: silu(gate) * up -> NVFP4 from the
    # gate/up output [512, 34816] (5 rotating copies, 178 MB > L2), dynamic and static g;
    # then the down projection on those NVFP4 activations (K 17408, N 5120, 3 weight
    # copies, 150 MB)
    from synth import random_gate_up
    Mf, If = 512, 17408
    gus = [random_gate_up(Mf, If, 50).cuda()]
    gus += [gus[0].clone() for _ in range(4)]
    hq = torch.empty(Mf, If // 2, dtype=torch.uint8, device="cuda")
    hs = torch.empty((Mf + 127) // 128 * 128 * ((If // 16 + 3) // 4 * 4), dtype=torch.uint8,
                     device="cuda")
    hg = torch.empty(1, dtype=torch.float32, device="cuda")
    hws = torch.empty(nv.nvfp4_workspace_bytes(0, Mf, If), dtype=torch.uint8, device="cuda")
    hb = Mf * 2 * If * 2 + Mf * If // 2 + Mf * If // 16 + 4
    ms = time_graph(torch, lambda i: nv.nvfp4_silu_mul_quantize(gus[i % 5], hq, hs, hg,
                                                                workspace=hws), 10, 5)
    rows["f1_silu_mul_quant_dynamic_%dx%d" % (Mf, If)] = {"GB/s": round(hb / ms / 1e6, 1),
                                                          "us": round(ms * 1e3, 1)}
    gstat = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    hg2 = torch.empty(1, dtype=torch.float32, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_silu_mul_quantize(gus[i % 5], hq, hs, hg2, gstat),
                    10, 5)
    rows["f1_silu_mul_quant_static_%dx%d" % (Mf, If)] = {"GB/s": round(hb / ms / 1e6, 1),
                                                         "us": round(ms * 1e3, 1)}
    del gus
    nv.nvfp4_silu_mul_quantize(random_gate_up(Mf, If, 51).cuda(), hq, hs, hg, workspace=hws)
    wl = WORKLOADS["prefill_b"]
    _, w = workload_inputs("prefill_b")
    p, _, z, gg = nv.quantize_weight(w.cuda())
    del w
    cps = [(p, z)] + [(p.clone(), z.clone()) for _ in range(2)]
    y = torch.empty(Mf, wl.N, dtype=torch.bfloat16, device="cuda")
    wsv = torch.zeros(nv.nvfp4_workspace_bytes(1, Mf, If, wl.N, nv.NVFP4_W4A4),
                      dtype=torch.uint8, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_linear_nvfp4_x(hq, hs, hg, cps[i % 3][0],
                                                             cps[i % 3][1], gg, y, wsv), 6, 5)
    tf = 2.0 * Mf * wl.N * If / (ms * 1e-3) / 1e12
    rows["f1_down_proj_nvfp4_x_M%d_K%d_N%d" % (Mf, If, wl.N)] = {
        "TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 1),
        "frac_fp4_nominal": round(tf / FP4_NOMINAL_TFLOPS, 4)}
    del cps, p, z
    # f1 fused: the gate/up projection of a 512-token chunk (K 5120 -> 2 x 17408, the
    # prefill_a weights as [gate; up]) with silu(gate) * up quantized to NVFP4 in the GEMM's
    # epilogue (static scale), against the two-kernel chain it replaces (the GEMM writing
    # bf16 gu, then the activation quantizer)
    wl = WORKLOADS["prefill_a"]
    x, w = workload_inputs("prefill_a")
    p, _, z, gg = nv.quantize_weight(w.cuda())
    del w
    cps = [(p, z), (p.clone(), z.clone())]
    xd = x.cuda()
    If = wl.N // 2
    hq2 = torch.empty(wl.M, If // 2, dtype=torch.uint8, device="cuda")
    hs2 = torch.empty((wl.M + 127) // 128 * 128 * ((If // 16 + 3) // 4 * 4), dtype=torch.uint8,
                      device="cuda")
    wsf = torch.zeros(nv.nvfp4_workspace_bytes(2, wl.M, wl.K, If), dtype=torch.uint8,
                      device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_linear_silu_mul_quantize(
        xd, cps[i % 2][0], cps[i % 2][1], gg, gstat, hq2, hs2, wsf), 4, 5)
    tf = 2.0 * wl.M * wl.N * wl.K / (ms * 1e-3) / 1e12
    rows["f1_gate_up_silu_quant_fused_M%d_K%d_I%d" % (wl.M, wl.K, If)] = {
        "TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 1),
        "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4)}
    gu2 = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    wsg = torch.zeros(nv.nvfp4_workspace_bytes(1, wl.M, wl.K, wl.N), dtype=torch.uint8,
                      device="cuda")

    def chain(i):
        nv.nvfp4_linear(xd, cps[i % 2][0], cps[i % 2][1], gg, gu2, workspace=wsg)
        nv.nvfp4_silu_mul_quantize(gu2, hq2, hs2, hg2, gstat)

    ms = time_graph(torch, chain, 4, 5)
    rows["f1_gate_up_then_silu_quant_two_kernels_M%d_K%d_I%d" % (wl.M, wl.K, If)] = {
        "us": round(ms * 1e3, 1)}
    del cps, p, z, gu2
    # a6 activation quantization (bf16 x 2048 x 5120) and a7 the W4A4 block-scaled GEMM
    # (the call quantizes x itself, so its time includes a6)
    wl = WORKLOADS["w4a4"]
    x, w = workload_inputs("w4a4")
    xd = x.cuda()
    xq = torch.empty(wl.M, wl.K // 2, dtype=torch.uint8, device="cuda")
    xs = torch.empty(wl.M, wl.K // 16, dtype=torch.uint8, device="cuda")
    gxd = torch.empty(1, dtype=torch.float32, device="cuda")
    wsq = torch.empty(nv.nvfp4_workspace_bytes(0, wl.M, wl.K), dtype=torch.uint8, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_quantize(xd, xq, xs, gxd, wsq), 8, 5)
    qb = wl.M * wl.K * 2 + wl.M * wl.K // 2 + wl.M * wl.K // 16 + 4
    rows["a6_act_quant_bf16_%dx%d" % (wl.M, wl.K)] = {"GB/s": round(qb / ms / 1e6, 1),
                                                      "us": round(ms * 1e3, 1)}
    p, _, z, gg = nv.quantize_weight(w.cuda())
    del w
    cps = [(p, z), (p.clone(), z.clone())]
    y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    wsv = torch.zeros(nv.nvfp4_workspace_bytes(1, wl.M, wl.K, wl.N, nv.NVFP4_W4A4),
                      dtype=torch.uint8, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_linear(xd, cps[i % 2][0], cps[i % 2][1], gg, y,
                                                     mode="w4a4", workspace=wsv), 4, 5)
    tf = 2.0 * wl.M * wl.N * wl.K / (ms * 1e-3) / 1e12
    rows["a7_w4a4_M%d_K%d_N%d_incl_act_quant" % (wl.M, wl.K, wl.N)] = {
        "TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 1),
        "frac_fp4_nominal": round(tf / FP4_NOMINAL_TFLOPS, 4)}
    # f2: the same call with a static activation scale (one quantization pass inside the
    # GEMM, no amax pass and no grid barrier)
    gx4 = torch.tensor([0.002], dtype=torch.float32, device="cuda")
    ms = time_graph(torch, lambda i: nv.nvfp4_linear(xd, cps[i % 2][0], cps[i % 2][1], gg, y,
                                                     mode="w4a4", x_global_scale=gx4,
                                                     workspace=wsv), 4, 5)
    tf = 2.0 * wl.M * wl.N * wl.K / (ms * 1e-3) / 1e12
    rows["f2_w4a4_static_scale_M%d_K%d_N%d_incl_act_quant" % (wl.M, wl.K, wl.N)] = {
        "TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 1),
        "frac_fp4_nominal": round(tf / FP4_NOMINAL_TFLOPS, 4)}
    del cps, p, z
    torch.cuda.synchronize()
    return rows


def read_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current source of the GEMV kernel (else null)."""
    try:
        txt = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    src = open(os.path.join(ROOT, "nvfp4_weight_quantized_quantize_gb300", "csrc",
                            "gemv.cu"), "rb").read()
    digest = hashlib.sha256(src).hexdigest()[:16]
    fields = dict(ln.split(":", 1) for ln in txt.splitlines() if ":" in ln)
    if fields.get("gemv_source_sha256_16", "").strip() != digest:
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


# ---- the CPU oracle (cpu_baseline leg and the reference arm) ------------------------------

def oracle_decode_inputs():
    import oracle
    from synth import workload_inputs
    out = []
    for name in DECODE:
        x, w = workload_inputs(name)
        wq, ws, gw = oracle.quantize(w.numpy())
        out.append((x, wq, ws, gw))
    return out


def oracle_slab(data, frac: float):
    """One timed unit of the oracle: the first `frac` of each decode shape's output rows
    (a contiguous slab of W rows, all M = 1 outputs of it), through the oracle's linear,
    which spreads the rows over every host thread.  Returns (run, algorithmic bytes)."""
    slabs = []
    for x, wq, ws, gw in data:
        n = max(1, min(wq.shape[0], int(round(wq.shape[0] * frac))))
        slabs.append((x, wq[:n], ws[:n], gw, n))
    nbytes = sum(algo_bytes(1, x.shape[1], n) for x, _, _, _, n in slabs)

    def run():
        for x, wq, ws, gw, _ in slabs:
            oracle_linear(x, wq, ws, gw)

    return run, nbytes, [n for *_, n in slabs]


def oracle_linear(x, wq, ws, gw):
    import oracle
    return oracle.linear_w4a16(x, wq, ws, gw)


def cpu_baseline(seconds: float = 10.0):
    import oracle
    data = oracle_decode_inputs()
    run, nbytes, _ = oracle_slab(data, 1.0)
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": round(nbytes * reps / el / 1e9, 3), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d full passes over both decode shapes (M=1, all N outputs, fp64)"
                      % reps}


def run_reference(args, rank, world, budget_s: float = 90.0):
    """The reference arm: the CPU oracle on the host cores.  A step is one pass over the
    same workload (both decode shapes, M = 1); where --steps full passes would take longer
    than budget_s, every step takes the same contiguous slab of each shape's rows, sized to
    the budget (at least 64 rows per host thread, so every thread has work)."""
    if rank != 0:
        return None
    import oracle
    data = oracle_decode_inputs()
    probe, _, _ = oracle_slab(data, 1.0)
    t0 = time.perf_counter()
    probe()
    full_s = time.perf_counter() - t0
    frac = min(1.0, budget_s / max(1e-9, full_s * (args.steps + args.warmup)))
    min_rows = 64 * oracle.num_threads()
    frac = max(frac, min(1.0, min_rows / min(wq.shape[0] for _, wq, _, _ in data)))
    run, nbytes, rows = oracle_slab(data, frac)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    if frac >= 1.0:
        sample = "every step one full pass over both decode shapes (M=1, all N outputs, fp64)"
    else:
        sample = ("every step the first %d and %d output rows of the two decode shapes (a "
                  "contiguous slab of W rows; the bytes of those rows: nibbles, scales, x, "
                  "y)" % tuple(rows))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode M=1 W4A16 NVFP4: (K=5120,N=17408) + "
                                   "(K=17408,N=5120), y bf16", "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.num_threads(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_one_workload(name: str, calls: int = 3):
    """A few nvfp4_linear calls on one workload and nothing else: the command that ncu
    captures a single kernel from (no timing, no JSON line)."""
    import torch

    import nvfp4_weight_quantized_quantize_gb300 as nv
    from nvfp4_weight_quantized_quantize_gb300 import build_lib
    from synth import WORKLOADS, workload_inputs

    build_lib.build()
    nv.load()
    if name == "fp8_requant":
        # FP8 block-128 -> NVFP4 on the decode_a shape (17408 x 5120)
        from synth import random_fp8_block128
        q8, s8 = random_fp8_block128(17408, 5120, 1)
        q8d, s8d = torch.from_numpy(q8).cuda(), torch.from_numpy(s8).cuda()
        packed = torch.empty(17408, 2560, dtype=torch.uint8, device="cuda")
        scales = torch.empty(17408, 320, dtype=torch.uint8, device="cuda")
        g = torch.empty(1, dtype=torch.float32, device="cuda")
        ws = torch.empty(nv.nvfp4_workspace_bytes(0, 17408, 5120), dtype=torch.uint8,
                         device="cuda")
        for _ in range(calls):
            nv.nvfp4_quantize_fp8_block128(q8d, s8d, packed, scales, g, ws)
        torch.cuda.synchronize()
        print("ran %d calls of %s" % (calls, name), flush=True)
        return
    if name == "mlp_act":
        # the 512-token MLP chunk: silu(gate) * up -> NVFP4 (dynamic g), then the down
        # projection (K 17408, N 5120) on those activations
        from synth import random_gate_up
        M, I, N = 512, 17408, 5120
        gu = random_gate_up(M, I, 50).cuda()
        hq = torch.empty(M, I // 2, dtype=torch.uint8, device="cuda")
        hs = torch.empty((M + 127) // 128 * 128 * ((I // 16 + 3) // 4 * 4), dtype=torch.uint8,
                         device="cuda")
        hg = torch.empty(1, dtype=torch.float32, device="cuda")
        hws = torch.empty(nv.nvfp4_workspace_bytes(0, M, I), dtype=torch.uint8, device="cuda")
        _, w = workload_inputs("prefill_b")
        packed, _, swz, g = nv.quantize_weight(w.cuda())
        del w
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, I, N, nv.NVFP4_W4A4),
                           dtype=torch.uint8, device="cuda")
        for _ in range(calls):
            nv.nvfp4_silu_mul_quantize(gu, hq, hs, hg, workspace=hws)
            nv.nvfp4_linear_nvfp4_x(hq, hs, hg, packed, swz, g, y, work)
        torch.cuda.synchronize()
        assert nv.nvfp4_workspace_error(work) == 0
        print("ran %d calls of %s" % (calls, name), flush=True)
        return
    if name.startswith("verify_a_m"):
        # the M = 9..16 end of the f4 curve: M tokens against the verify_a weights
        from synth import random_x
        M = int(name[len("verify_a_m"):])
        wl = WORKLOADS["verify_a"]
        _, w = workload_inputs("verify_a")
        packed, _, swz, g = nv.quantize_weight(w.cuda())
        del w
        xd = random_x(M, wl.K, seed=M).cuda()
        y = torch.empty(M, wl.N, dtype=torch.bfloat16, device="cuda")
        work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, wl.K, wl.N), dtype=torch.uint8,
                           device="cuda")
        for _ in range(calls):
            nv.nvfp4_linear(xd, packed, swz, g, y, workspace=work)
        torch.cuda.synchronize()
        assert nv.nvfp4_workspace_error(work) == 0
        print("ran %d calls of %s" % (calls, name), flush=True)
        return
    wl = WORKLOADS[name]
    x, w = workload_inputs(name)
    packed, _, swz, g = nv.quantize_weight(w.cuda())
    del w
    mode = nv.NVFP4_W4A4 if wl.w4a4 else nv.NVFP4_W4A16
    xd = x.cuda()
    y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, wl.M, wl.K, wl.N, mode), dtype=torch.uint8,
                       device="cuda")
    for _ in range(calls):
        nv.nvfp4_linear(xd, packed, swz, g, y, mode="w4a4" if wl.w4a4 else "w4a16",
                        workspace=work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    print("ran %d calls of %s" % (calls, name), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=256)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=4)
    ap.add_argument("--static-weights", type=int, default=1,
                    help="1 (default): the decode and verify calls declare their weights "
                         "static (NVFP4_STATIC_WEIGHTS: nothing in flight writes them), so "
                         "each launch streams them before the previous launch has ended")
    ap.add_argument("--rows", type=int, default=1, help="also measure the other rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only-workload", default=None,
                    help="run a few calls of one workload and exit (for ncu captures): a "
                         "workload name, fp8_requant, mlp_act or verify_a_m<M> (M tokens on "
                         "the verify_a weights)")
    args = ap.parse_args()
    global STATIC_W
    STATIC_W = bool(args.static_weights)
    if args.only_workload:
        run_one_workload(args.only_workload)
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
        out = run_ours(args, rank, world, dist)
        if dist:
            dist.destroy_process_group()
    if out is not None and rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
