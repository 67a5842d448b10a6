"""Benchmark of the weight-only quantized GEMV hot path on GB300.

One step = one decode step through L layers, each layer running the three
batch-1 GEMVs of the headline metric on its own weights:
  W8: int8, group-128 fp32 scales, K = N = 4096, fp32 x / y
  W3: 3-bit, per-column fp16 scale and zero, K = N = 4096, fp16 x / y
  W4: 4-bit act-order (g_idx), group-128 fp16 scales and 4-bit zeros,
      K = 4096, N = 11008, fp16 x / y.  At weight-load time (outside every
      timed region) wq4_actorder_prepare sorts each layer's rows by group
      once; the step runs wq4_gemm_sorted on the sorted copy, which computes
      the same y.  The online act-order kernel (wq4_gemm with g_idx) is timed
      beside it and reported in the config.
The L layers' weights live in distinct device buffers (L * 47 MB > 3x the
L2 cache), so every GEMV streams its weights from HBM.  The kernels of a step
are captured in one CUDA graph and chained with programmatic dependent launch;
the roofline kernel's average launch duration is timed with CUDA events
around a chain of its 16 launches (one per layer, PDL-chained as in the step);
a second replay of the step with an event pair around each W4 launch gives its
isolated duration (events break the launch chain), reported beside it.

value = algorithmic bytes (packed weights + scales + zeros + g_idx + x + y)
of all GEMVs of all steps / device time of the timed steps, in GB/s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs its own replica (weak scaling); rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (% of roofline), W3/W4/W8 GEMV K=N=4096, M=1"
LAYERS = 16
WORKLOAD = ("decode step through 16 layers, each: W8 g128 GEMV 4096x4096 (fp32) + W3 per-column GEMV "
            "4096x4096 (fp16) + W4 act-order g128 GEMV 4096x11008 (fp16), M=1")
FALLBACK_HBM_GBS = 6800.0
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of each kernel of the
# step, from one ncu capture of this script's own command; None until the kernel
# as it is now has been captured (a capture of an older version does not count).
TRAFFIC_BYTES = {"w8": 17338624, "w3": 6337280, "w4": 23494656}
KERNEL_NAMES = {
    "w8": "k8_gemv_kernel<1> (W8 g128 GEMV 4096x4096, fp32 x)",
    "w3": "k3_gemv_kernel<1> (W3 per-column GEMV 4096x4096, fp16 x)",
    "w4": "k4t_gemv_kernel<f16, zeros, perm> (W4 act-order GEMV 4096x11008 on group-sorted rows, mma.sync)",
}


def alg_bytes_w8(M=1, K=4096, N=4096, g=128):
    return K * N + (K // g) * N * 4 + M * K * 4 + M * N * 4


def alg_bytes_w3(M=1, K=4096, N=4096):
    return (3 * K // 32) * N * 4 + N * 2 * 2 + M * K * 2 + M * N * 2


def alg_bytes_w4g(M=1, K=4096, N=11008, g=128):
    G = K // g
    return (K // 8) * N * 4 + G * N * 2 + G * (N // 8) * 4 + K * 4 + M * K * 2 + M * N * 2


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(v: float, world: int, device) -> float:
    """Largest value of v over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_bytes: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed / the slowest rank's time."""
    return step_bytes * steps * world / (max_ms * 1e-3) / 1e9


def measured_bf16_peak():
    """Dense bf16 tensor peak (burst), TFLOP/s: the fp16/bf16 MMA rate the exact
    integer product of the W8A8 path runs at."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for ln in (self.out or "").splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ inputs ----

def make_layer_inputs(layer: int):
    """Seeded inputs of one layer (numpy).  Layer l uses seeds 1000*l + {1, 2, 3}."""
    import synthetic as syn
    base = 1000 * layer
    return (syn.make_wq8(seed=base + 1), syn.make_wq3(seed=base + 2), syn.make_wq4_actorder(seed=base + 3))


def to_dev(a, dev):
    import numpy as np
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


class Layer:
    def __init__(self, d8, d3, d4, dev):
        import torch

        import gemm_dequant_gemv_gb300 as wq
        self.w8 = {k: to_dev(d8[k], dev) for k in ("x", "w", "scales")}
        self.w3 = {k: to_dev(d3[k], dev) for k in ("x", "mat", "scales", "zeros")}
        self.w4 = {k: to_dev(d4[k], dev) for k in ("x", "qweight", "scales", "qzeros", "g_idx")}
        # weight-load-time transform of the act-order layer: rows sorted by group, once
        self.qw_sorted = torch.empty_like(self.w4["qweight"])
        self.perm = torch.empty_like(self.w4["g_idx"])
        wq.wq4_actorder_prepare(self.w4["qweight"], self.w4["g_idx"], 4096, 11008, 128, self.qw_sorted, self.perm)
        self.y8 = torch.empty((1, 4096), dtype=torch.float32, device=dev)
        self.y3 = torch.empty((1, 4096), dtype=torch.float16, device=dev)
        self.y4 = torch.empty((1, 11008), dtype=torch.float16, device=dev)

    def run_w8(self, wq, flags, stream):
        t = self.w8
        wq.wq8_gemv(t["x"], t["w"], t["scales"], self.y8, 1, 4096, 4096, 128, flags=flags, stream=stream)

    def run_w3(self, wq, flags, stream):
        t = self.w3
        wq.wq3_gemv(t["x"], t["mat"], t["scales"], t["zeros"], self.y3, 1, 4096, 4096, flags=flags, stream=stream)

    def run_w4(self, wq, flags, stream):
        t = self.w4
        wq.wq4_gemm_sorted(t["x"], self.qw_sorted, t["scales"], t["qzeros"], self.perm, self.y4, 1, 4096, 11008,
                           128, wq.WQ_F16, flags=flags, stream=stream)

    def run_w4_online(self, wq, flags, stream):
        t = self.w4
        wq.wq4_gemm(t["x"], t["qweight"], t["scales"], t["qzeros"], t["g_idx"], self.y4, 1, 4096, 11008, 128,
                    wq.WQ_F16, flags=flags, stream=stream)


def pack_io(layers, dev):
    """Make every layer's x (and every y) a view into one device buffer, so that a
    step's inputs reach the device in one copy and its results come back in one.
    Views start on 256-byte boundaries (the kernels' tensor maps want 16)."""
    import torch

    def pack(get, put):
        ts = [get(L, j) for L in layers for j in range(3)]
        offs, o = [], 0
        for t in ts:
            offs.append(o)
            o += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.zeros(o, dtype=torch.uint8, device=dev)
        i = 0
        for L in layers:
            for j in range(3):
                t = ts[i]
                v = buf[offs[i]:offs[i] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                v.copy_(t)
                put(L, j, v)
                i += 1
        return buf

    xkeys = ("w8", "w3", "w4")
    xbuf = pack(lambda L, j: getattr(L, xkeys[j])["x"], lambda L, j, v: getattr(L, xkeys[j]).__setitem__("x", v))
    ykeys = ("y8", "y3", "y4")
    ybuf = pack(lambda L, j: getattr(L, ykeys[j]), lambda L, j, v: setattr(L, ykeys[j], v))
    return xbuf, ybuf


# -------------------------------------------------------------- our arm ----

def run_ours(args, rank, world, dev):
    import numpy as np
    import torch

    import gemm_dequant_gemv_gb300 as wq

    torch.cuda.set_device(dev)
    # every layer gets its own device copy of the seeded weights: distinct buffers, so the
    # step's weights (L x 47 MB) exceed the L2 cache and each GEMV streams from HBM
    inputs = make_layer_inputs(rank)
    layers = [Layer(*inputs, dev) for _ in range(LAYERS)]
    xbuf, ybuf = pack_io(layers, dev)
    step_bytes = LAYERS * (alg_bytes_w8() + alg_bytes_w3() + alg_bytes_w4g())
    stream = torch.cuda.Stream(device=dev)
    s = stream.cuda_stream
    PDL = wq.WQ_FLAG_PDL

    # one step as a CUDA graph: per layer W4, W8, W3, chained with PDL
    def step(evs=None):
        for i, L in enumerate(layers):
            if evs is not None:
                evs[i][0].record(stream)
            L.run_w4(wq, PDL, s)
            if evs is not None:
                evs[i][1].record(stream)
            L.run_w8(wq, PDL, s)
            L.run_w3(wq, PDL, s)

    with torch.cuda.stream(stream):
        step()  # eager warm-up of every kernel instance before capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        step()
    # the same step with an event pair around each W4 launch: per-launch duration of the roofline kernel
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(LAYERS)]
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream, capture_error_mode="relaxed"):
        step(ev)
    with torch.cuda.stream(stream):  # CUDAGraph.replay() launches on the current stream
        for _ in range(max(3, args.warmup)):
            graph.replay()
        graph_ev.replay()
    torch.cuda.synchronize(dev)

    gpu_id = torch.cuda.get_device_properties(dev).uuid
    gpu_id = f"GPU-{gpu_id}" if gpu_id and not str(gpu_id).startswith("GPU-") else str(gpu_id)
    if world > 1:
        torch.distributed.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            t1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    w4_us = []
    with torch.cuda.stream(stream):
        for _ in range(5):
            graph_ev.replay()
            torch.cuda.synchronize(dev)
            w4_us += [ev[i][0].elapsed_time(ev[i][1]) * 1e3 for i in range(LAYERS)]

    # every kernel of the step on its own: its 16 launches (one per layer) back to
    # back, chained with PDL as in the step ("chained"), and the same 16 launches
    # without PDL, so that each starts only after the previous one has finished
    # ("serialized": the single-call latency on the device)
    def kernel_times(run):
        out = {}
        for name, flags in (("chained", PDL), ("serialized", 0)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for L in layers:
                    run(L, flags)
            out[name] = _time_graph(g, stream, 50, dev) * 1e3 / LAYERS
        return out
    per_kernel = {
        "w8": kernel_times(lambda L, f: L.run_w8(wq, f, s)),
        "w3": kernel_times(lambda L, f: L.run_w3(wq, f, s)),
        "w4": kernel_times(lambda L, f: L.run_w4(wq, f, s)),
    }
    w4_chain_us = per_kernel["w4"]["chained"]

    # the online act-order kernel (g_idx gathered per k, no prepared copy), chained over the layers
    g_on = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for L in layers:
            L.run_w4_online(wq, PDL, s)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(g_on, stream=stream, capture_error_mode="relaxed"):
        for L in layers:
            L.run_w4_online(wq, PDL, s)
    w4_online_us = _time_graph(g_on, stream, 50, dev) * 1e3 / LAYERS
    ms = max_over_ranks(ms, world, dev)

    # end to end through the public API, host buffers: every step copies all 48 x
    # vectors in from pinned host memory (one packed copy), launches the 48 GEMVs
    # through the Python binding, and copies all 48 y vectors back (one packed copy)
    e2e_steps = max(3, min(args.steps, 50))
    hx = torch.empty_like(xbuf, device="cpu").pin_memory()
    hy = torch.empty_like(ybuf, device="cpu").pin_memory()
    hx.copy_(xbuf)
    h2d = int(hx.numel())
    d2h = int(hy.numel())

    def e2e_step():
        with torch.cuda.stream(stream):
            xbuf.copy_(hx, non_blocking=True)
            for L in layers:
                L.run_w4(wq, PDL, s)
                L.run_w8(wq, PDL, s)
                L.run_w3(wq, PDL, s)
            hy.copy_(ybuf, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    if world > 1:
        torch.distributed.barrier()
    te = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    te = time.perf_counter() - te
    te = max_over_ranks(te, world, dev)

    return dict(ms=ms, w4_us=w4_us, w4_chain_us=w4_chain_us, w4_online_us=w4_online_us, per_kernel=per_kernel,
                clocks=clk.summary(),
                step_bytes=step_bytes,
                e2e_s_per_step=te / e2e_steps, h2d=h2d, d2h=d2h, e2e_steps=e2e_steps)


# ------------------------------------------------------------- the oracle ----

def oracle_step(d8, d3, d4, cols8=None, cols3=None, cols4=None):
    import numpy as np

    import oracle
    oracle.wq8_gemv(d8["x"], d8["w"], d8["scales"], 128, cols=cols8)
    oracle.wq3_gemv(d3["x"].view(np.uint16), d3["mat"], d3["scales"].view(np.uint16), d3["zeros"].view(np.uint16),
                    cols=cols3)
    oracle.wq4_gemm(d4["x"].view(np.uint16), 0, d4["qweight"], d4["scales"].view(np.uint16), d4["qzeros"],
                    d4["g_idx"], 128, cols=cols4)


def sample_bytes(n8, n3, n4):
    """Algorithmic bytes of the oracle sample restricted to n8/n3/n4 output columns."""
    return (alg_bytes_w8() * n8 / 4096 + alg_bytes_w3() * n3 / 4096 + alg_bytes_w4g() * n4 / 11008)


def host_cores():
    """Host core count and the cores this process may run on."""
    try:
        allowed = sorted(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        allowed = list(range(os.cpu_count() or 1))
    return os.cpu_count() or len(allowed), allowed


def pin_to_one_core():
    """Pin the calling thread to one allowed core (the oracle is single-threaded);
    returns that core, or None where the platform has no affinity call."""
    _, allowed = host_cores()
    try:
        os.sched_setaffinity(0, {allowed[-1]})
        return allowed[-1]
    except (AttributeError, OSError):
        return None


def cpu_baseline(budget_s=10.0):
    """The oracle as it stands, single-threaded and pinned to one core, on whole
    steps of one layer."""
    import oracle
    oracle.build()
    d8, d3, d4 = make_layer_inputs(0)
    total, allowed = host_cores()
    saved = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    core = pin_to_one_core()
    try:
        t = time.perf_counter()
        n = 0
        while True:
            oracle_step(d8, d3, d4)
            n += 1
            if time.perf_counter() - t >= budget_s:
                break
        dt = time.perf_counter() - t
    finally:
        if saved is not None:
            os.sched_setaffinity(0, saved)
    b = n * sample_bytes(4096, 4096, 11008)
    return {"value": b / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "host_cores": total, "affinity_cores": len(allowed), "pinned_core": core,
            "sample": f"{n} full single-layer steps (W8 + W3 + W4 act-order GEMVs, every output column), "
                      f"{dt:.1f} s single-threaded C oracle pinned to one of the host's {total} cores"}


def run_reference(args):
    """The oracle as the reference arm: each step a column sample of one layer's GEMVs,
    sized so that the whole run takes about a minute."""
    import numpy as np

    import oracle
    oracle.build()
    d8, d3, d4 = make_layer_inputs(0)
    total, allowed = host_cores()
    core = pin_to_one_core()
    r = np.random.default_rng(0)
    probe = r.choice(4096, 64, replace=False)
    t = time.perf_counter()
    oracle_step(d8, d3, d4, probe, probe, probe)
    per_col = (time.perf_counter() - t) / 64
    total_steps = max(1, args.steps + args.warmup)
    ncols = int(max(1, min(4096, args.ref_budget / (total_steps * max(per_col, 1e-9)))))
    c8, c3 = r.choice(4096, ncols, replace=False), r.choice(4096, ncols, replace=False)
    c4 = r.choice(11008, ncols, replace=False)
    for _ in range(args.warmup):
        oracle_step(d8, d3, d4, c8, c3, c4)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(d8, d3, d4, c8, c3, c4)
    dt = time.perf_counter() - t
    b = args.steps * sample_bytes(ncols, ncols, ncols)
    value = b / dt / 1e9
    sample = (f"each step: {ncols} sampled output columns of each of the three GEMVs of one layer "
              f"(single-threaded C oracle)")
    return {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": 1, "M": 1, "sample_columns": ncols},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                             "host_cores": total, "affinity_cores": len(allowed), "pinned_core": core},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------- the other two workloads ----

def _time_graph(graph, stream, reps, dev):
    import torch
    with torch.cuda.stream(stream):  # CUDAGraph.replay() launches on the current stream
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps  # ms per replay


def run_wq4_sweep(args, dev):
    """W4A16 (symmetric uint4, group 128, bf16) at K=8192, N=28672 for each M:
    three weight copies (363 MB, larger than L2) cycled in one CUDA graph."""
    import torch

    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    peak, peak_kind = measured_peaks()
    K, N, g = 8192, 28672, 128
    base = syn.make_wq4_sym(seed=4, M=1, K=K, N=N, group=g)
    copies = 3
    qws = [to_dev(base["qweight"], dev) for _ in range(copies)]
    scs = [to_dev(base["scales"], dev) for _ in range(copies)]
    stream = torch.cuda.Stream(device=dev)
    lines = []
    for M in (1, 2, 4, 8, 16, 32):
        x = to_dev(syn.f32_to_bf16_bits(syn.normal(4 + M, 1, (M, K))), dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        with torch.cuda.stream(stream):
            for c in range(copies):
                wq.wq4_gemm(x, qws[c], scs[c], None, None, y, M, K, N, g, wq.WQ_BF16, flags=wq.WQ_FLAG_PDL,
                            stream=stream)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        per = 8
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
            for r in range(per):
                c = r % copies
                wq.wq4_gemm(x, qws[c], scs[c], None, None, y, M, K, N, g, wq.WQ_BF16, flags=wq.WQ_FLAG_PDL,
                            stream=stream)
        ms = _time_graph(graph, stream, args.extra_reps, dev) / per
        nbytes = (K // 8) * N * 4 + (K // g) * N * 2 + M * K * 2 + M * N * 2
        gbs = nbytes / (ms * 1e-3) / 1e9
        lines.append({"workload": f"W4A16 sym g128 K={K} N={N} M={M}", "M": M,
                      "path": ("mma.sync m16n8k16 (warp-level tensor cores)"
                               + ("" if M <= 8 else f", {2 if M <= 16 else 4} n-tiles of 8 rows")),
                      "us_per_call": ms * 1e3,
                      "achieved_GBps": gbs, "frac_of_hbm": gbs / peak, "peak_source": peak_kind,
                      "tflops": 2 * M * K * N / (ms * 1e-3) / 1e12})
    return lines


def run_w8a8(args, dev):
    """W8A8 dynamic-quantization GEMM at M=2048, K=N=8192 (quantization + GEMM per call)."""
    import torch

    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    M, K, N = 2048, 8192, 8192
    d = syn.make_w8a8(seed=5, M=M, K=K, N=N)
    X, W, Sw = to_dev(d["X"], dev), to_dev(d["W"], dev), to_dev(d["Sw"], dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    nbytes = wq.w8a8_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        wq.w8a8_gemm(X, W, Sw, Y, M, K, N, workspace=ws, workspace_bytes=nbytes, stream=stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    per = 4
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        for _ in range(per):
            wq.w8a8_gemm(X, W, Sw, Y, M, K, N, workspace=ws, workspace_bytes=nbytes, flags=wq.WQ_FLAG_PDL,
                         stream=stream)
    ms = _time_graph(graph, stream, args.extra_reps, dev) / per
    pk, pk_kind = measured_bf16_peak()
    tf = 2 * M * K * N / (ms * 1e-3) / 1e12
    lines = [{"workload": f"W8A8 dynamic quant GEMM M={M} K={K} N={N}", "us_per_call": ms * 1e3, "tops": tf,
              "peak_tflops_f16_dense": pk, "peak_source": pk_kind, "frac_of_tensor_peak": tf / pk,
              "note": "exact int8 products on fp16 tcgen05 MMA; the int8 legacy mma.sync path measured 158 TOPS"}]

    # the two variants on the same shape: LLM.int8() with 8 outlier columns (0.1 % of K,
    # values 8..15 in one row each, threshold 6) and Smoothquant with s = sqrt(max_m |X[m,k]|)
    import numpy as np
    Xo = d["X"].copy()
    r = np.random.default_rng(5)
    cols = r.choice(K, size=8, replace=False)
    for i, c in enumerate(cols):
        Xo[r.integers(0, M), c] = syn.f32_to_bf16_bits(np.array([8.0 + i], np.float32))[0]
    Xo_d = to_dev(Xo, dev)
    nbo = wq.w8a8_gemm_outlier_workspace_bytes(M, K, N)
    wso = torch.empty(nbo, dtype=torch.uint8, device=dev)
    nout = torch.zeros((4,), dtype=torch.int32, device=dev)

    def outlier(flags):
        wq.w8a8_gemm_outlier(Xo_d, W, Sw, Y, M, K, N, 6.0, n_outliers_out=nout, workspace=wso, workspace_bytes=nbo,
                             flags=flags, stream=stream)
    smooth = to_dev(np.sqrt(np.maximum(np.abs(syn.bf16_bits_to_f32(d["X"])).max(axis=0), 1e-3)).astype(np.float32),
                    dev)

    def smoothed(flags):
        wq.w8a8_gemm_smooth(X, smooth, W, Sw, Y, M, K, N, workspace=ws, workspace_bytes=nbytes, flags=flags,
                            stream=stream)
    for name, fn in (("LLM.int8() decomposition, 8 outlier columns, threshold 6", outlier),
                     ("Smoothquant activation smoothing", smoothed)):
        with torch.cuda.stream(stream):
            fn(0)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for _ in range(per):
                fn(wq.WQ_FLAG_PDL)
        msv = _time_graph(g, stream, args.extra_reps, dev) / per
        line = {"workload": f"W8A8 M={M} K={K} N={N}, {name}", "us_per_call": msv * 1e3,
                "overhead_vs_plain": msv / ms - 1, "tops": 2 * M * K * N / (msv * 1e-3) / 1e12}
        if fn is outlier:
            line["outlier_columns"] = int(nout[0])
        lines.append(line)
    return lines


def run_unfused(args, dev):
    """The unfused baseline beside the fused kernels ("融合反量化与GEMM", 核心优化思路):
    dequantize into a dense matrix in HBM, then a dense product (torch.matmul,
    i.e. cuBLAS), against the fused call, for the three GEMVs and W4A16 at M = 1
    and 16.  The packed weights rotate over enough copies to exceed the L2 three
    times; the dense matrix is one scratch buffer, written and read every call."""
    import torch

    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    peak, peak_kind = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(device=dev)
    s = stream.cuda_stream
    lines = []

    def timed(issue, copies):
        with torch.cuda.stream(stream):
            for c in range(copies):
                issue(c)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        per = max(copies, 4)
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
            for r in range(per):
                issue(r % copies)
        return _time_graph(graph, stream, 20, dev) / per * 1e3  # us per call

    def case(name, packed, extra, dense_bytes, fused, dequant, product):
        copies = max(2, -(-3 * l2 // max(packed, 1)))
        state = [extra(c) for c in range(copies)]
        f_us = timed(lambda c: fused(state[c]), copies)
        d_us = timed(lambda c: dequant(state[c]), copies)
        u_us = timed(lambda c: (dequant(state[c]), product(state[c])), copies)
        fused_bytes = state[0]["alg_bytes"]
        unfused_bytes = fused_bytes + 2 * dense_bytes
        lines.append({"workload": name, "fused_us": f_us, "dequant_us": d_us, "unfused_us": u_us,
                      "dense_product_us": u_us - d_us, "fused_speedup": u_us / f_us,
                      "alg_bytes_fused": fused_bytes, "bytes_unfused": unfused_bytes,
                      "traffic_saved_by_fusion": 1 - fused_bytes / unfused_bytes,
                      "fused_GBps": fused_bytes / (f_us * 1e-6) / 1e9, "peak_GBps": peak, "peak_source": peak_kind,
                      "dense_product": "torch.matmul (cuBLAS)", "copies": copies})

    # W8: x fp32 [1, 4096], dense fp32 weights
    d8 = syn.make_wq8(seed=1)
    K, N = 4096, 4096
    x8 = to_dev(d8["x"], dev)
    y8 = torch.empty((1, N), dtype=torch.float32, device=dev)
    W8 = torch.empty((K, N), dtype=torch.float32, device=dev)
    b8 = alg_bytes_w8()

    def e8(c):
        return {"w": to_dev(d8["w"], dev), "s": to_dev(d8["scales"], dev), "alg_bytes": b8}
    case("W8 g128 GEMV 4096x4096, M=1", K * N + (K // 128) * N * 4, e8, K * N * 4,
         lambda t: wq.wq8_gemv(x8, t["w"], t["s"], y8, 1, K, N, 128, stream=s),
         lambda t: wq.wq8_dequant(t["w"], t["s"], W8, K, N, 128, stream=s),
         lambda t: torch.matmul(x8, W8, out=y8))

    # W3: x fp16, dense fp16 weights
    d3 = syn.make_wq3(seed=2)
    x3 = to_dev(d3["x"], dev)
    y3 = torch.empty((1, N), dtype=torch.float16, device=dev)
    W3 = torch.empty((K, N), dtype=torch.float16, device=dev)
    b3 = alg_bytes_w3()

    def e3(c):
        return {"m": to_dev(d3["mat"], dev), "s": to_dev(d3["scales"], dev), "z": to_dev(d3["zeros"], dev),
                "alg_bytes": b3}
    case("W3 per-column GEMV 4096x4096, M=1", 3 * K // 32 * N * 4, e3, K * N * 2,
         lambda t: wq.wq3_gemv(x3, t["m"], t["s"], t["z"], y3, 1, K, N, stream=s),
         lambda t: wq.wq3_dequant(t["m"], t["s"], t["z"], W3, K, N, stream=s),
         lambda t: torch.matmul(x3, W3, out=y3))

    # W4 act-order: fused = the sorted-rows GEMV of the decode step; dense fp16 weights
    d4 = syn.make_wq4_actorder(seed=3)
    N4 = 11008
    x4 = to_dev(d4["x"], dev)
    y4 = torch.empty((1, N4), dtype=torch.float16, device=dev)
    W4 = torch.empty((K, N4), dtype=torch.float16, device=dev)
    b4 = alg_bytes_w4g()

    def e4(c):
        t = {"qw": to_dev(d4["qweight"], dev), "s": to_dev(d4["scales"], dev), "z": to_dev(d4["qzeros"], dev),
             "g": to_dev(d4["g_idx"], dev), "alg_bytes": b4}
        t["qs"], t["perm"] = torch.empty_like(t["qw"]), torch.empty_like(t["g"])
        wq.wq4_actorder_prepare(t["qw"], t["g"], K, N4, 128, t["qs"], t["perm"])
        return t
    case("W4 act-order g128 GEMV 4096x11008, M=1", K // 8 * N4 * 4 + (K // 128) * N4 * 3, e4, K * N4 * 2,
         lambda t: wq.wq4_gemm_sorted(x4, t["qs"], t["s"], t["z"], t["perm"], y4, 1, K, N4, 128, wq.WQ_F16,
                                      stream=s),
         lambda t: wq.wq4_dequant(t["qw"], t["s"], t["z"], t["g"], W4, K, N4, 128, wq.WQ_F16, stream=s),
         lambda t: torch.matmul(x4, W4, out=y4))

    # W4A16 8192 x 28672, symmetric, bf16: M = 1 and M = 16
    dw = syn.make_wq4_sym(seed=4, M=1, K=8192, N=28672, group=128)
    Kw, Nw = 8192, 28672
    Ww = torch.empty((Kw, Nw), dtype=torch.bfloat16, device=dev)
    packed_w = Kw // 8 * Nw * 4 + (Kw // 128) * Nw * 2

    def ew(c):
        return {"qw": to_dev(dw["qweight"], dev), "s": to_dev(dw["scales"], dev), "alg_bytes": 0}
    for M in (1, 16):
        xw = to_dev(syn.f32_to_bf16_bits(syn.normal(4 + M, 1, (M, Kw))), dev)
        yw = torch.empty((M, Nw), dtype=torch.bfloat16, device=dev)
        bw = packed_w + M * Kw * 2 + M * Nw * 2

        def ewm(c, bw=bw):
            t = ew(c)
            t["alg_bytes"] = bw
            return t
        case(f"W4A16 sym g128 8192x28672, M={M}", packed_w, ewm, Kw * Nw * 2,
             lambda t, xw=xw, yw=yw, M=M: wq.wq4_gemm(xw, t["qw"], t["s"], None, None, yw, M, Kw, Nw, 128,
                                                        wq.WQ_BF16, stream=s),
             lambda t: wq.wq4_dequant(t["qw"], t["s"], None, None, Ww, Kw, Nw, 128, wq.WQ_BF16, stream=s),
             lambda t, xw=xw, yw=yw: torch.matmul(xw, Ww, out=yw))
    return lines


# -------------------------------------------------------------------- main ----

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of oracle work the reference arm aims for")
    ap.add_argument("--workload", default="gemv_step", choices=["gemv_step", "wq4_sweep", "w8a8", "unfused"],
                    help="gemv_step is the headline; the others print one extra line per case")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="leave the W4A16 sweep and W8A8 out of the headline line")
    ap.add_argument("--extra-reps", type=int, default=10,
                    help="graph replays timed per case of the W4A16 sweep and W8A8")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    dev = torch.device(f"cuda:{local}")
    if args.workload != "gemv_step":
        torch.cuda.set_device(dev)
        fn = {"wq4_sweep": run_wq4_sweep, "w8a8": run_w8a8, "unfused": run_unfused}[args.workload]
        for ln in fn(args, dev):
            print(json.dumps(ln), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(dev)
        torch.distributed.init_process_group("nccl", device_id=dev)
    res = run_ours(args, rank, world, dev)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    peak, peak_kind = measured_peaks()
    value = job_throughput(res["step_bytes"], args.steps, world, res["ms"])
    w4_us = statistics.mean(res["w4_us"])
    alg = {"w8": alg_bytes_w8(), "w3": alg_bytes_w3(), "w4": alg_bytes_w4g()}
    kernels = {}
    for k, t in res["per_kernel"].items():
        kernels[k] = {"kernel": KERNEL_NAMES[k], "alg_bytes": alg[k],
                      "us_per_call_chained": t["chained"], "us_per_call_serialized": t["serialized"],
                      "GBps_chained": alg[k] / (t["chained"] * 1e-6) / 1e9,
                      "GBps_serialized": alg[k] / (t["serialized"] * 1e-6) / 1e9,
                      "frac_chained": alg[k] / (t["chained"] * 1e-6) / 1e9 / peak,
                      "frac_serialized": alg[k] / (t["serialized"] * 1e-6) / 1e9 / peak}
    # the dominant kernel: the largest share of the step (16 chained launches of each)
    dom = max(kernels, key=lambda k: kernels[k]["us_per_call_chained"])
    achieved = kernels[dom]["GBps_chained"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": LAYERS, "M": 1,
                   "l2": f"inputs larger than L2: {LAYERS} distinct weight sets, "
                         f"{res['step_bytes'] / 1e6:.0f} MB per step",
                   "us_per_call_mean": res["ms"] / args.steps * 1e3 / (3 * LAYERS),
                   "w4_actorder_us_per_launch_in_step": w4_us,
                   "w4_actorder_path": "rows sorted by group once at weight-load time (wq4_actorder_prepare), "
                                       "then wq4_gemm_sorted",
                   "w4_actorder_online_us_per_call": res["w4_online_us"]},
        "kernels": kernels,
        "roofline": {"bound": "hbm", "kernel": KERNEL_NAMES[dom],
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "traffic": TRAFFIC_BYTES[dom],
                     "launch_time": "average of 16 PDL-chained launches, CUDA events on the launching stream"},
        "e2e": {"value": world * res["step_bytes"] / res["e2e_s_per_step"] / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "steps": res["e2e_steps"]},
        "gpu_launches": 3 * LAYERS * args.steps,
        "clocks": res["clocks"],
    }
    if not args.no_extra_configs:
        line["configs"] = {"w4a16_sweep": run_wq4_sweep(args, dev), "w8a8": run_w8a8(args, dev)}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
