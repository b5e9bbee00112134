"""Benchmark of the block-quantized weight x Q8 activation matmul on GB300.

One JSON line on rank 0.  The headline workload is the Q8_0 x Q8_0 decode
matvec of an 8B-class FFN gate (N = 12288 rows, K = 4096, one token): a step
quantizes the token's activation (Q8_0) and streams the whole weight matrix
through the matvec, and `value` is weight bytes per second over exactly K timed
steps.  The same run measures, as extra keys, the other workloads (Q4_0
4864x896, the Q4_K_M decoder-layer set, Q2_K 12288x4096, the Q4_0 prefill at
M = 128/512/2048), the dominant kernel against the HBM roofline, the
end-to-end path from pinned host memory, and the CPU oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qmm|reference]

Under torchrun each rank runs its own copy of the workload on its own GPU (the
matvec shards along independent output rows, so ranks need no collective);
`value` is the bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "quant matvec weight-stream GB/s (M=1) & prefill int8 TOPS, % of roofline"
HEADLINE = "q8_0_matvec_12288x4096"
L2_BYTES = 129 * 10**6
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILE_FILE = os.path.join(ROOT, "profiles", "matvec_q8_0_12288x4096.txt")
MATVEC_SOURCES = ["block_quantized_weight_q8_gb300/csrc/matvec.cu", "block_quantized_weight_q8_gb300/csrc/qmm_device.cuh"]


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment; (0, 0, 1) without it."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """The maximum of x over ranks (x itself on one rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_per_rank: float, world: int, device=None):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    t = reduce_max(seconds_per_rank, world, device)
    return units_per_rank * world / t, t


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms while the benchmark runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [s for (t, s) in self.samples if any(a - 0.05 <= t <= b + 0.05 for a, b in self.windows)]
        pool = inside if len(inside) >= 3 else [s for (_, s) in self.samples]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in pool:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(pool), "in_timed_regions": len(inside) >= 3}


# ------------------------------------------------------------------ helpers
def act_of(wtype):
    return "q8_0" if wtype in ("q4_0", "q8_0", "q4_1", "q5_0", "q5_1") else "q8_K"


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def matvec_source_hash():
    h = hashlib.sha256()
    for p in MATVEC_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    try:
        text = open(PROFILE_FILE).read()
    except OSError:
        return None, "no profile summary"
    m_hash = re.search(r"kernel source hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram bytes per launch:\s*([0-9]+)", text)
    if not (m_hash and m_bytes):
        return None, "profile summary incomplete"
    if m_hash.group(1) != matvec_source_hash():
        return None, "kernel changed since the ncu capture"
    return int(m_bytes.group(1)), "ncu capture"


class Timer:
    """CUDA events on a stream, bracketed by barrier + synchronize."""

    def __init__(self, torch, stream, world, clocks):
        self.torch, self.stream, self.world, self.clocks = torch, stream, world, clocks

    def run(self, fn, iters: int) -> float:
        torch = self.torch
        barrier(self.world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        w0 = time.time()
        e0.record(self.stream)
        for i in range(iters):
            fn(i)
        e1.record(self.stream)
        torch.cuda.synchronize()
        w1 = time.time()
        barrier(self.world)
        if self.clocks is not None:
            self.clocks.mark(w0, w1)
        return e0.elapsed_time(e1) / 1000.0  # seconds


def timed_regions(timer, region, world, device, min_seconds: float):
    """Times region() (one bracketed timed region each) repeatedly until at least min_seconds of
    device time is timed; every rank runs the same number of regions.  Returns (seconds, regions)."""
    first = timer.run(region, 1)
    want = int(np.ceil(min_seconds / max(first, 1e-7)))
    regions = max(1, min(100000, int(reduce_max(want, world, device))))
    secs = sum(timer.run(region, 1) for _ in range(regions))
    return secs, regions


def make_graph(torch, stream, body, count: int):
    """Capture `count` calls of body(i) into one CUDA graph on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(count):
            body(i)
    return g


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, rank, local_rank, world):
    import torch

    import block_quantized_weight_q8_gb300 as qmm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    init_dist(world, "nccl")
    qmm.build()
    qmm.load()
    peaks = load_peaks()
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    stream = torch.cuda.Stream(device=dev)
    timer = Timer(torch, stream, world, clocks)
    out = {}

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def quantized_weights(wtype, N, K, seed, stream_id=0, jitter=False):
        w = to_dev(workloads.weights_f32(N, K, seed, stream=stream_id, row_jitter=jitter))
        W = torch.empty(N * qmm.qmm_row_bytes(wtype, K), dtype=torch.uint8, device=dev)
        qmm.quantize(wtype, w, W, N, K, stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        del w
        return W

    def copies_for(nbytes):
        return max(2, int(np.ceil(2.5 * L2_BYTES / nbytes)))

    # ---------------- headline: Q8_0 decode step (quantize + matvec)
    cfg = workloads.WORKLOADS[HEADLINE]
    N, K = cfg["N"], cfg["K"]
    W0 = quantized_weights("q8_0", N, K, cfg["seed"])
    wbytes = W0.numel()
    C = copies_for(wbytes)
    Ws = [W0] + [W0.clone() for _ in range(C - 1)]
    x = to_dev(workloads.activations_f32(1, K, cfg["seed"]))
    xrb = qmm.qmm_row_bytes("q8_0", K)
    xq = torch.empty(xrb, dtype=torch.uint8, device=dev)
    y = torch.empty(N, dtype=torch.float32, device=dev)
    sh = stream.cuda_stream

    def step(i):
        qmm.qmm_linear_q8_0(Ws[i % C], x, xq, xrb, y, 1, N, K, stream=sh)

    # One timed region is exactly --steps steps: a CUDA graph of G = min(steps, 64) calls replayed
    # steps // G times, then a graph of the remaining steps % G calls.
    G = min(args.steps, 64)
    full, rest = divmod(args.steps, G)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
        graph = make_graph(torch, stream, step, G)
        graph_rest = make_graph(torch, stream, lambda i: step(full * G + i), rest) if rest else None
    torch.cuda.synchronize()

    def region(_):
        for _ in range(full):
            graph.replay()
        if graph_rest is not None:
            graph_rest.replay()

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // G)):  # at least one full replay of each graph
            graph.replay()
        if graph_rest is not None:
            graph_rest.replay()
        secs, regions = timed_regions(timer, region, world, dev, args.min_timed_s)
    value, tmax = aggregate(wbytes * args.steps * regions, secs, world, dev)
    ms_per_step = tmax / (args.steps * regions) * 1e3
    launches = 1 * args.steps  # per timed region: the step is one kernel (it quantizes x, then multiplies)

    # the step's kernel is the dominant (only) kernel: roofline from the step's own timing.
    # Algorithmic bytes per launch: W, the f32 x, the quantized row stored once, y.
    step_s = secs / (args.steps * regions)
    algo_bytes = wbytes + 4 * K + xrb + 4 * N
    achieved = algo_bytes / step_s / 1e9

    # the multiply alone on an already-quantized row (public qmm_matvec_q8_0), for reference
    def mv(i):
        qmm.qmm_matvec_q8_0(Ws[i % C], xq, y, N, K, stream=sh)

    with torch.cuda.stream(stream):
        mv_graph = make_graph(torch, stream, mv, 64)
        mv_graph.replay()
        mv_secs, mv_regions = timed_regions(timer, lambda i: mv_graph.replay(), 1, dev, args.min_timed_s)
    mv_launch_s = mv_secs / (mv_regions * 64)
    traffic, traffic_src = profiled_traffic()
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": "matvec_kernel<Q8_0, super-unit, fused quantize>",
                "algorithmic_bytes_per_launch": algo_bytes,
                "launch_us": round(step_s * 1e6, 3),
                "matvec_only_us": round(mv_launch_s * 1e6, 3),
                "matvec_only_GB/s": round((wbytes + xrb + 4 * N) / mv_launch_s / 1e9, 1),
                "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs: a copy kernel, read+write)" % peaks["source"],
                "traffic_source": traffic_src}

    # ---------------- end to end: pinned host x -> device, linear, y -> pinned host
    x_host = torch.from_numpy(workloads.activations_f32(1, K, cfg["seed"] + 7)).pin_memory()
    y_host = torch.empty(N, dtype=torch.float32).pin_memory()
    x_dev = torch.empty(K, dtype=torch.float32, device=dev)

    def e2e_step(i):
        # one C-ABI call with host buffers: x_host -> device, quantize + multiply, y -> y_host
        qmm.qmm_linear_host("q8_0", Ws[i % C], x_host, x_dev, xq, xrb, y, y_host, 1, N, K, stream=sh)

    e2e_steps = min(args.steps, 2000)
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        e2e_secs, e2e_regions = timed_regions(timer, lambda _: [e2e_step(i) for i in range(e2e_steps)], world, dev,
                                              args.min_timed_s)
    e2e_value, _ = aggregate(wbytes * e2e_steps * e2e_regions, e2e_secs, world, dev)
    e2e = {"value": round(e2e_value / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": 4 * K,
           "d2h_bytes_per_step": 4 * N, "steps": e2e_steps, "timed_regions": e2e_regions,
           "note": "qmm_linear_host per step, eager calls through the binding: x (16 KB) read from pinned host "
                   "memory by the quantize kernel over the host link, the multiply, y (48 KB) written by it into "
                   "pinned host memory; both transfers inside the timed region, one stream"}
    del Ws, W0

    # ---------------- other workloads
    extra = {}
    if not args.headline_only:
        extra = other_workloads(args, torch, qmm, dev, stream, timer, peaks, world, quantized_weights, copies_for)

    clock_info = clocks.summary() if clocks else None
    if clocks:
        clocks.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value / 1e9, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "timed_regions": regions,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded N(0,0.02) weights quantized on the GPU; N(0,1) activation with 1% x20)",
            "config": {"workload": HEADLINE, "wtype": "q8_0", "M": 1, "N": N, "K": K, "weight_bytes": wbytes,
                       "step": "qmm_linear_q8_0: one kernel per token (each CTA quantizes x to Q8_0, then the "
                               "matvec), chained launches, CUDA graph",
                       "timing": "each timed region is exactly `steps` steps, bracketed by barrier + synchronize "
                                 "and CUDA events on the launching stream; regions repeat until at least %.0f ms "
                                 "is timed (%d regions); value and ms_per_step over all of them" % (
                                     args.min_timed_s * 1e3, regions),
                       "l2": "weights rotate over %d resident copies (%.0f MB > 2x the 129 MB L2)" % (
                           C, C * wbytes / 1e6),
                       "parallelism": "replicas: each rank streams its own weights" if world > 1 else "1 GPU"},
            "roofline": roofline,
            "gpu_launches": launches,
            "gpu_launches_all_regions": launches * regions,
            "e2e": e2e,
            "clocks": clock_info,
            "configs": extra,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)


def other_workloads(args, torch, qmm, dev, stream, timer, peaks, world, quantized_weights, copies_for):
    res = {}
    sh = stream.cuda_stream
    hbm = peaks["hbm_gbs"]
    steps = max(16, min(args.steps, 512))
    graph_steps = 16

    def timed_graph(body, n_body):
        with torch.cuda.stream(stream):
            for i in range(2):
                body(i)
            g = make_graph(torch, stream, body, n_body)
            g.replay()
            reps = max(2, steps // n_body)
            secs = timer.run(lambda i: g.replay(), reps)
        return secs / (reps * n_body)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # single matvecs
    for name in ("q4_0_matvec_4864x896", "q2_K_matvec_12288x4096", "q4_1_matvec_12288x4096",
                 "q5_0_matvec_12288x4096", "q5_1_matvec_12288x4096", "q5_K_matvec_12288x4096"):
        cfg = workloads.WORKLOADS[name]
        wtype, N, K = cfg["wtype"], cfg["N"], cfg["K"]
        W0 = quantized_weights(wtype, N, K, cfg["seed"])
        C = copies_for(W0.numel())
        Ws = [W0] + [W0.clone() for _ in range(C - 1)]
        act = act_of(wtype)
        x = to_dev(workloads.activations_f32(1, K, cfg["seed"]))
        xrb = qmm.qmm_row_bytes(act, K)
        xq = torch.empty(xrb, dtype=torch.uint8, device=dev)
        y = torch.empty(N, dtype=torch.float32, device=dev)

        def step(i):
            qmm.linear(wtype, Ws[i % C], x, xq, xrb, y, 1, N, K, stream=sh)

        def mv(i):
            qmm.matvec(wtype, Ws[i % C], xq, y, N, K, stream=sh)

        t_step = timed_graph(step, graph_steps)
        t_mv = timed_graph(mv, graph_steps)
        wb = W0.numel()
        res[name] = {"step_us": round(t_step * 1e6, 3), "GB/s": round(wb / t_step / 1e9, 1),
                     "matvec_us": round(t_mv * 1e6, 3), "matvec_GB/s": round(wb / t_mv / 1e9, 1),
                     "frac_hbm": round(wb / t_mv / 1e9 / hbm, 4), "weight_bytes": wb, "copies": C}
        del Ws, W0

    # the decoder-layer set: quantize(x_h) shared by Wq Wk Wv W_gate W_up; Wo and W_down on their own inputs
    cfg = workloads.WORKLOADS["q4_K_M_layer_4096"]
    mats = []
    for i, (label, wtype, N, K) in enumerate(cfg["matrices"]):
        mats.append((label, wtype, N, K, quantized_weights(wtype, N, K, cfg["seed"], stream_id=i, jitter=True)))
    layer_bytes = sum(m[4].numel() for m in mats)
    C = max(2, int(np.ceil(2.5 * 129e6 / layer_bytes)))
    sets = [mats] + [[(a, b, c, d, W.clone()) for (a, b, c, d, W) in mats] for _ in range(C - 1)]
    xh = to_dev(workloads.activations_f32(1, 4096, cfg["seed"]))
    xo = to_dev(workloads.activations_f32(1, 4096, cfg["seed"] + 1))
    xd = to_dev(workloads.activations_f32(1, 12288, cfg["seed"] + 2))
    qh = torch.empty(qmm.qmm_row_bytes("q8_K", 4096), dtype=torch.uint8, device=dev)
    qo = torch.empty_like(qh)
    qd = torch.empty(qmm.qmm_row_bytes("q8_K", 12288), dtype=torch.uint8, device=dev)
    outs = {m[0]: torch.empty(m[2], dtype=torch.float32, device=dev) for m in mats}

    def layer(i):
        s = sets[i % C]
        qmm.qmm_quantize_q8_K(xh, qh, 1, 4096, stream=sh)
        for (label, wtype, N, K, W) in s:
            if label in ("Wq", "Wk", "Wv", "W_gate", "W_up"):
                qmm.matvec(wtype, W, qh, outs[label], N, K, stream=sh)
        qmm.qmm_quantize_q8_K(xo, qo, 1, 4096, stream=sh)
        qmm.matvec("q4_K", s[3][4], qo, outs["Wo"], 4096, 4096, stream=sh)
        qmm.qmm_quantize_q8_K(xd, qd, 1, 12288, stream=sh)
        qmm.matvec("q6_K", s[6][4], qd, outs["W_down"], 4096, 12288, stream=sh)

    # the same layer through qmm_linear_*: each multiply quantizes its own input row in-kernel
    scratch = torch.empty(qmm.qmm_row_bytes("q8_K", 12288), dtype=torch.uint8, device=dev)
    xin = {"Wq": xh, "Wk": xh, "Wv": xh, "W_gate": xh, "W_up": xh, "Wo": xo, "W_down": xd}

    def layer_linear(i):
        for (label, wtype, N, K, W) in sets[i % C]:
            qmm.linear(wtype, W, xin[label], scratch, scratch.numel(), outs[label], 1, N, K, stream=sh)

    # the same layer with the projections that read one row grouped: Q, K, V in one launch, gate and up
    # in another (qmm_linear_group), Wo and W_down on their own
    by = {m[0]: i for i, m in enumerate(mats)}

    def layer_group(i):
        s = sets[i % C]
        for names, xin_ in ((("Wq", "Wk", "Wv"), xh), (("Wo",), xo), (("W_gate", "W_up"), xh), (("W_down",), xd)):
            ms = [s[by[n]] for n in names]
            K = ms[0][3]
            qmm.qmm_linear_group(ms[0][1], [m[4] for m in ms], [m[2] for m in ms], xin_, scratch, scratch.numel(),
                                 [outs[n] for n in names], 1, K, stream=sh)

    # the same four launches with each group's RMSNorm inside it: h = rmsnorm(x) ; qa = quantize(h)
    # feeding Q, K, V (and gate, up) from one launch, as the layer's data flow reads
    gam = to_dev(np.random.default_rng(cfg["seed"]).uniform(0.5, 1.5, size=4096).astype(np.float32))

    def layer_norm(i):
        s = sets[i % C]
        for names, xin_, normed in ((("Wq", "Wk", "Wv"), xh, True), (("Wo",), xo, False),
                                    (("W_gate", "W_up"), xh, True), (("W_down",), xd, False)):
            ms = [s[by[n]] for n in names]
            K = ms[0][3]
            if normed:
                qmm.qmm_linear_norm(ms[0][1], [m[4] for m in ms], [m[2] for m in ms], xin_, gam, 1e-6, scratch,
                                    scratch.numel(), [outs[n] for n in names], 1, K, stream=sh)
            else:
                qmm.qmm_linear_group(ms[0][1], [m[4] for m in ms], [m[2] for m in ms], xin_, scratch,
                                     scratch.numel(), [outs[n] for n in names], 1, K, stream=sh)

    t_layer = timed_graph(layer, 8)
    t_lin = timed_graph(layer_linear, 8)
    t_grp = timed_graph(layer_group, 8)
    t_nrm = timed_graph(layer_norm, 8)
    res["q4_K_M_layer_4096"] = {"layer_us": round(t_layer * 1e6, 3), "GB/s": round(layer_bytes / t_layer / 1e9, 1),
                                "frac_hbm": round(layer_bytes / t_layer / 1e9 / hbm, 4), "weight_bytes": layer_bytes,
                                "equiv_tok_s_36_layers_matmuls_only": round(1.0 / (36 * t_layer), 1),
                                "launches_per_layer": 10, "copies": C,
                                "how": "3 shared qmm_quantize_q8_K + 7 qmm_matvec",
                                "linear_layer_us": round(t_lin * 1e6, 3),
                                "linear_GB/s": round(layer_bytes / t_lin / 1e9, 1),
                                "linear_launches_per_layer": 7,
                                "group_layer_us": round(t_grp * 1e6, 3),
                                "group_GB/s": round(layer_bytes / t_grp / 1e9, 1),
                                "group_frac_hbm": round(layer_bytes / t_grp / 1e9 / hbm, 4),
                                "group_launches_per_layer": 4,
                                "group_equiv_tok_s_36_layers_matmuls_only": round(1.0 / (36 * t_grp), 1),
                                "group_with_rmsnorm_layer_us": round(t_nrm * 1e6, 3),
                                "group_with_rmsnorm_GB/s": round(layer_bytes / t_nrm / 1e9, 1),
                                "group_with_rmsnorm_note": "QKV and gate+up launches also RMSNorm their row"}
    del sets, mats

    # the Q8 KV cache of one decode-attention layer: quantize the query heads, score every cached
    # position against them, and sum the V rows under the attention weights (the softmax between the
    # two is not part of the library: its output is an input here).  Enough copies of the caches
    # that a replay cycle streams more than L2 holds.
    cfg = workloads.WORKLOADS["q8_kv_cache_32x8x4096x128"]
    Hq, Hkv, P, hd = cfg["Hq"], cfg["Hkv"], cfg["P"], cfg["hd"]
    q, k, v, w = workloads.kv_inputs(Hq, Hkv, P, hd, cfg["seed"])
    rb = qmm.qmm_kv_row_bytes(hd)
    kc = torch.empty(P * Hkv * rb, dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    with torch.cuda.stream(stream):
        qmm.qmm_kv_quantize(to_dev(k), kc, P * Hkv, hd, stream=sh)
        qmm.qmm_kv_quantize(to_dev(v), vc, P * Hkv, hd, stream=sh)
    stream.synchronize()
    cache_bytes = 2 * kc.numel()
    C = max(2, int(np.ceil(2.5 * 129e6 / cache_bytes)))
    kcs = [kc] + [kc.clone() for _ in range(C - 1)]
    vcs = [vc] + [vc.clone() for _ in range(C - 1)]
    qx, wd = to_dev(q), to_dev(w)
    q8 = torch.empty(Hq * rb, dtype=torch.uint8, device=dev)
    scores = torch.empty(Hq, P, dtype=torch.float32, device=dev)
    out = torch.empty(Hq, hd, dtype=torch.float32, device=dev)
    sbk = qmm.qmm_kv_wsum_scratch_bytes(Hq, P, hd)
    kscratch = torch.empty(sbk, dtype=torch.uint8, device=dev)
    scale = float(1.0 / np.sqrt(hd))

    def attn(i):
        qmm.qmm_kv_quantize(qx, q8, Hq, hd, stream=sh)
        qmm.qmm_kv_scores(q8, kcs[i % C], scores, Hq, Hkv, P, hd, scale, stream=sh)
        qmm.qmm_kv_wsum(wd, vcs[i % C], out, kscratch, sbk, Hq, Hkv, P, hd, stream=sh)

    t_attn = timed_graph(attn, 8)
    t_sc = timed_graph(lambda i: qmm.qmm_kv_scores(q8, kcs[i % C], scores, Hq, Hkv, P, hd, scale, stream=sh), 8)
    t_ws = timed_graph(lambda i: qmm.qmm_kv_wsum(wd, vcs[i % C], out, kscratch, sbk, Hq, Hkv, P, hd, stream=sh), 8)
    res["q8_kv_cache_32x8x4096x128"] = {
        "us": round(t_attn * 1e6, 3), "cache_bytes": cache_bytes, "cache_GB/s": round(cache_bytes / t_attn / 1e9, 1),
        "frac_hbm": round(cache_bytes / t_attn / 1e9 / hbm, 4), "launches": 4, "copies": C,
        "scores_us": round(t_sc * 1e6, 3), "scores_K_GB/s": round(kc.numel() / t_sc / 1e9, 1),
        "wsum_us": round(t_ws * 1e6, 3), "wsum_V_GB/s": round(vc.numel() / t_ws / 1e9, 1),
        "how": "qmm_kv_quantize (32 query heads) + qmm_kv_scores + qmm_kv_wsum (2 launches)"}
    del kcs, vcs

    # prefill
    cfg = workloads.WORKLOADS["q4_0_prefill_512x12288x4096"]
    N, K = cfg["N"], cfg["K"]
    W = quantized_weights("q4_0", N, K, cfg["seed"])
    # weight copies rotate so that each launch finds its W in HBM, not in the 129 MB L2
    Cw = copies_for(W.numel())
    Wr = [W] + [W.clone() for _ in range(Cw - 1)]
    pre = {"weights": "%d rotating copies of W per timing (%.0f MB)" % (Cw, Cw * W.numel() / 1e6)}
    for M in cfg["M_sweep"]:
        x = to_dev(workloads.activations_f32(M, K, cfg["seed"] + M))
        xrb = qmm.qmm_row_bytes("q8_0", K)
        xq = torch.empty(M * xrb, dtype=torch.uint8, device=dev)
        Y = torch.empty(M, N, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            qmm.qmm_quantize_q8_0(x, xq, M, K, stream=sh)

        def mm(i):
            qmm.qmm_matmul_q4_0(Wr[i % Cw], xq, Y, M, N, K, stream=sh)

        t = timed_graph(mm, Cw)
        ops = 2.0 * M * N * K
        tops = ops / t / 1e12
        pre["M=%d" % M] = {"us": round(t * 1e6, 2), "int8_equiv_TOPS": round(tops, 2),
                           "frac_bf16_dense_peak": round(tops / peaks["bf16_tflops"], 4),
                           "frac_hbm_weight_stream": round(W.numel() / t / 1e9 / hbm, 4)}
    # the other 32-value weight formats on the same prefill kernel
    M = 512
    x = to_dev(workloads.activations_f32(M, K, cfg["seed"] + M))
    xq = torch.empty(M * qmm.qmm_row_bytes("q8_0", K), dtype=torch.uint8, device=dev)
    Y = torch.empty(M, N, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        qmm.qmm_quantize_q8_0(x, xq, M, K, stream=sh)
    del Wr
    for wtype in ("q8_0", "q4_1", "q5_0", "q5_1"):
        W8 = quantized_weights(wtype, N, K, cfg["seed"])
        C8 = copies_for(W8.numel())
        W8r = [W8] + [W8.clone() for _ in range(C8 - 1)]
        t = timed_graph(lambda i: qmm.matmul(wtype, W8r[i % C8], xq, Y, M, N, K, stream=sh), C8)
        tops = 2.0 * M * N * K / t / 1e12
        pre["%s_weights_M=512" % wtype] = {"us": round(t * 1e6, 2), "int8_equiv_TOPS": round(tops, 2),
                                           "frac_bf16_dense_peak": round(tops / peaks["bf16_tflops"], 4),
                                           "frac_hbm_weight_stream": round(W8.numel() / t / 1e9 / hbm, 4)}
        del W8, W8r
    del x, xq, Y
    # the K-quant prefill at the decoder layer's shapes (M = 512): W_gate/W_up (Q4_K), W_down (Q6_K),
    # and the Q2_K matrix
    kq = {}
    for wtype, Nk, Kk in (("q4_K", 12288, 4096), ("q6_K", 4096, 12288), ("q2_K", 12288, 4096), ("q5_K", 12288, 4096)):
        M = 512
        Wk = quantized_weights(wtype, Nk, Kk, cfg["seed"])
        xk = to_dev(workloads.activations_f32(M, Kk, cfg["seed"] + 3))
        xqk = torch.empty(M * qmm.qmm_row_bytes("q8_K", Kk), dtype=torch.uint8, device=dev)
        Yk = torch.empty(M, Nk, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            qmm.qmm_quantize_q8_K(xk, xqk, M, Kk, stream=sh)
        Ck = copies_for(Wk.numel())
        Wkr = [Wk] + [Wk.clone() for _ in range(Ck - 1)]
        tk = timed_graph(lambda i: qmm.matmul(wtype, Wkr[i % Ck], xqk, Yk, M, Nk, Kk, stream=sh), Ck)
        tops = 2.0 * M * Nk * Kk / tk / 1e12
        kq["%s_%dx%dx%d" % (wtype, M, Nk, Kk)] = {"us": round(tk * 1e6, 2), "int8_equiv_TOPS": round(tops, 2),
                                                  "frac_bf16_dense_peak": round(tops / peaks["bf16_tflops"], 4),
                                                  "frac_hbm_weight_stream": round(Wk.numel() / tk / 1e9 / hbm, 4)}
        del Wk, Wkr, xk, xqk, Yk
    pre["k_quants_M=512"] = kq

    # context: the GPU's own int8 and fp16 GEMMs (cuBLAS through torch) on the M=512 shape
    try:
        M = 512
        a8 = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev)
        b8 = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev).t()
        ah = torch.randn(M, K, dtype=torch.float16, device=dev)
        bh = torch.randn(K, N, dtype=torch.float16, device=dev)
        t8 = timed_graph(lambda i: torch._int_mm(a8, b8), 2)
        t16 = timed_graph(lambda i: torch.matmul(ah, bh), 2)
        pre["context_cublas_M=512"] = {"int8_TOPS": round(2.0 * M * N * K / t8 / 1e12, 1),
                                       "fp16_TFLOPS": round(2.0 * M * N * K / t16 / 1e12, 1),
                                       "note": "torch._int_mm / fp16 matmul on the same shape: the int8 tensor "
                                               "path of this GPU, and the fp16 path the prefill kernel uses"}
        del a8, b8, ah, bh
    except Exception as ex:  # context only
        pre["context_cublas_M=512"] = {"error": str(ex)[:120]}
    res["q4_0_prefill_12288x4096"] = pre
    return res


# ------------------------------------------------------------------ CPU baseline (the oracle)
def cpu_sample(nthreads: int, target_s: float):
    """Time the oracle on the headline workload: quantize the token and run the matvec over as many
    whole repetitions as fill about target_s seconds.  Returns (GB/s, seconds, reps, rows)."""
    import oracle

    cfg = workloads.WORKLOADS[HEADLINE]
    N, K = cfg["N"], cfg["K"]
    w = workloads.weights_f32(N, K, cfg["seed"])
    W = oracle.quantize("q8_0", w)
    x = workloads.activations_f32(1, K, cfg["seed"])
    t0 = time.perf_counter()
    xq = oracle.quantize("q8_0", x)
    oracle.matmul("q8_0", W, xq, 1, N, K, nthreads=nthreads)
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        xq = oracle.quantize("q8_0", x)
        oracle.matmul("q8_0", W, xq, 1, N, K, nthreads=nthreads)
    secs = time.perf_counter() - t0
    return W.size * reps / secs / 1e9, secs, reps, N


def cpu_baseline(args):
    nthreads = os.cpu_count() or 1
    gbs, secs, reps, rows = cpu_sample(nthreads, args.cpu_seconds)
    # the same on one thread, a shorter sample: the rows split over threads is bit-identical, so this
    # is the single-core rate of the same computation
    gbs1, secs1, reps1, _ = cpu_sample(1, max(1.0, args.cpu_seconds / 3))
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": "%d full steps of the %s workload (quantize + %d-row matvec), %.1f s, rows split over %d "
                      "threads" % (reps, HEADLINE, rows, secs, nthreads),
            "one_thread": {"value": round(gbs1, 3), "unit": "GB/s", "sample": "%d full steps, %.1f s" % (reps1, secs1)},
            "cpu": cpu_model()}


def oracle_table(args):
    """The CPU oracle on every configuration of the benchmark workloads, on one thread and on all of
    the host's threads (rows split evenly, bit-identical results): the median of 5 timed runs of a
    quantize + multiply step, with the CPU model.  The prefill runs on a bounded sample of its
    tokens (all rows, all of K), reported as GOP/s; everything else runs whole."""
    import oracle

    nthreads = os.cpu_count() or 1

    def median_time(fn, reps=5):
        fn()  # warm-up (page-in, caches)
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return float(np.median(ts))

    rows = {}
    for name in ("q4_0_matvec_4864x896", "q8_0_matvec_12288x4096", "q2_K_matvec_12288x4096"):
        cfg = workloads.WORKLOADS[name]
        wt, N, K = cfg["wtype"], cfg["N"], cfg["K"]
        W = oracle.quantize(wt, workloads.weights_f32(N, K, cfg["seed"]))
        x = workloads.activations_f32(1, K, cfg["seed"])
        act = act_of(wt)
        res = {"weight_bytes": int(W.size)}
        for nt in (1, nthreads):
            t = median_time(lambda: oracle.matmul(wt, W, oracle.quantize(act, x), 1, N, K, nthreads=nt))
            res["ms_%dt" % nt] = round(t * 1e3, 3)
            res["GB/s_%dt" % nt] = round(W.size / t / 1e9, 2)
        rows[name] = res
    # the decoder-layer set: three quantized rows, seven matrices
    cfg = workloads.WORKLOADS["q4_K_M_layer_4096"]
    mats = []
    for i, (label, wt, N, K) in enumerate(cfg["matrices"]):
        mats.append((label, wt, N, K, oracle.quantize(wt, workloads.weights_f32(N, K, cfg["seed"], stream=i,
                                                                                  row_jitter=True))))
    xh = workloads.activations_f32(1, 4096, cfg["seed"])
    xo = workloads.activations_f32(1, 4096, cfg["seed"] + 1)
    xd = workloads.activations_f32(1, 12288, cfg["seed"] + 2)
    layer_bytes = sum(m[4].size for m in mats)

    def layer(nt):
        qh, qo, qd = oracle.quantize("q8_K", xh), oracle.quantize("q8_K", xo), oracle.quantize("q8_K", xd)
        for (label, wt, N, K, W) in mats:
            xq = qd if label == "W_down" else (qo if label == "Wo" else qh)
            oracle.matmul(wt, W, xq, 1, N, K, nthreads=nt)

    res = {"weight_bytes": int(layer_bytes)}
    for nt in (1, nthreads):
        t = median_time(lambda: layer(nt))
        res["ms_%dt" % nt] = round(t * 1e3, 3)
        res["GB/s_%dt" % nt] = round(layer_bytes / t / 1e9, 2)
    rows["q4_K_M_layer_4096"] = res
    # the prefill: a bounded sample of tokens against all rows, as GOP/s (the work is linear in M)
    cfg = workloads.WORKLOADS["q4_0_prefill_512x12288x4096"]
    N, K = cfg["N"], cfg["K"]
    W = oracle.quantize("q4_0", workloads.weights_f32(N, K, cfg["seed"]))
    res = {}
    for nt, Ms in ((1, 2), (nthreads, 16)):
        x = workloads.activations_f32(Ms, K, cfg["seed"] + 512)
        t = median_time(lambda: oracle.matmul("q4_0", W, oracle.quantize("q8_0", x), Ms, N, K, nthreads=nt))
        gops = 2.0 * Ms * N * K / t / 1e9
        res["GOP/s_%dt" % nt] = round(gops, 2)
        res["sample_%dt" % nt] = "%d tokens x %d rows x K=%d" % (Ms, N, K)
        for M in cfg["M_sweep"]:
            res["est_ms_M=%d_%dt" % (M, nt)] = round(2.0 * M * N * K / (gops * 1e9) * 1e3, 1)
    rows["q4_0_prefill_12288x4096"] = res
    line = {"oracle_table": rows, "threads": nthreads, "cpu": cpu_model(), "median_of": 5,
            "note": "oracle = quantize + multiply, scalar C (-O2 -ffp-contract=off), rows split over threads"}
    print(json.dumps(line), flush=True)


def cpu_model() -> str:
    """The host CPU's model name as the OS reports it (or the machine type)."""
    arm = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
                if key in ("cpu implementer", "cpu part") and key not in arm:
                    arm[key] = line.split(":", 1)[1].strip()
    except OSError:
        pass
    if arm:  # Arm cores report their implementer and part numbers (0x41 / 0xd4f: Neoverse V2)
        return "Arm implementer %s part %s" % (arm.get("cpu implementer", "?"), arm.get("cpu part", "?"))
    import platform
    return platform.machine() or "unknown"


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, timed on the host cores, same metric and workload."""
    if rank != 0:
        return
    import oracle

    nthreads = os.cpu_count() or 1
    cfg = workloads.WORKLOADS[HEADLINE]
    N, K = cfg["N"], cfg["K"]
    W = oracle.quantize("q8_0", workloads.weights_f32(N, K, cfg["seed"]))
    x = workloads.activations_f32(1, K, cfg["seed"])
    rb = W.shape[1]
    # each step: a bounded sample of the workload (the first `rows` rows), sized so the run ends in minutes
    t0 = time.perf_counter()
    oracle.matmul("q8_0", W, oracle.quantize("q8_0", x), 1, N, K, nthreads=nthreads)
    full = time.perf_counter() - t0
    budget = 60.0 / max(1, args.steps + args.warmup)
    rows = int(min(N, max(64, N * budget / max(full, 1e-4))))
    Ws = np.ascontiguousarray(W[:rows])
    for _ in range(args.warmup):
        oracle.matmul("q8_0", Ws, oracle.quantize("q8_0", x), 1, rows, K, nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul("q8_0", Ws, oracle.quantize("q8_0", x), 1, rows, K, nthreads=nthreads)
    secs = time.perf_counter() - t0
    value = rows * rb * args.steps / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded)",
            "config": {"workload": HEADLINE, "wtype": "q8_0", "M": 1, "N": N, "K": K, "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": "%d of %d rows per step, rows split over %d threads" % (rows, N, nthreads)},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["qmm", "reference"], default="qmm")
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the CPU oracle on every configuration (1 and all threads, median of 5) and exit")
    ap.add_argument("--min-timed-s", type=float, default=0.05,
                    help="repeat the timed region of --steps steps until this much device time is timed")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, local_rank, world = dist_env()
    if args.oracle_table:
        if rank == 0:
            oracle_table(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, local_rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
