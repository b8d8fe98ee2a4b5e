#!/usr/bin/env python
"""Benchmark of the quantized-weight matmul on GB300.

Default workload (one "step"): the decode GEMV at nt = 1 on two Llama-7B-shaped
Q4_K projections, od x K = 4096 x 4096 and 11008 x 4096, with x ~ N(0, 1) plus
0.1% outliers x20.  A step runs the whole path for both: q8_1 quantization of
x and the MMVQ matmul (the decode branch of the dispatch, one fused kernel per
projection), through the C ABI.

value   weight GB/s of the whole job: weight bytes of all steps on all ranks /
        max-over-ranks wall time of the timed region, inputs resident in HBM.
        Each step reads the next of 16 rotating weight copies (557 MB > 4x L2),
        so no step finds its weights in L2.  The steps are replayed from CUDA
        graphs of up to 1024 consecutive steps (one graph for K <= 1024),
        right after the warm-up steps.
e2e     the same metric with the activations copied from pinned host memory and
        the outputs copied back inside every step, one qmm_matmul call per
        projection; copy-in, matmuls and copy-out are pipelined on three
        streams (double-buffered) and replayed from CUDA graphs.
roofline  the dominant kernel of the step -- the fused quantize + MMVQ kernel of
        the 11008 x 4096 projection -- alone: algorithmic bytes (weights, f32
        activations read, q8_1 activations and f32 outputs written) per launch
        / its mean launch time (CUDA events around back-to-back launches over
        rotating copies), against the measured HBM copy bandwidth.
per_nt  the rest of the metric, one record per (shape, nt): Q4_K 4096x4096 and
        14336x4096 at nt in {1, 2, 4, 8, 16, 128, 512, 2048}, Q6_K 32000x4096 at
        nt in {1, 8, 32, 64, 80, 256}.  Each case is timed twice from a CUDA
        graph of back-to-back calls over rotating weight copies (>= 4x L2):
        the matmul on q8_1 input (us_kernel: qmm_gemv / qmm_gemm, the latter
        with its operand prepass) and the whole path from f32 activations
        (us_path: qmm_matmul).  TOPS, weight GB/s and the fractions of the
        measured HBM copy bandwidth and bf16 tensor peak come from us_kernel.
roofline_gemm  the prefill GEMM (Q4_K 14336x4096, nt = 512) as its own
        roofline object: 2*nt*od*K per launch / us_kernel against the measured
        dense bf16 peak (the tensor-core route issues kind::f16 MMAs).
cpu_baseline  the CPU oracle (plain scalar C, all host cores) on the same step.

--impl reference   times the CPU oracle alone as the reference arm.
--sweep            one JSON line per case of every workload family (or of
                   --shape QTYPE:ODxKxNT[,...]), timed as a per_nt record;
                   not the contract line.
--profile SPEC     a fixed number (--calls) of eager calls of one case, for
                   ncu captures; no timing.
Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one rank per GPU, each rank running the same workload on
its own GPU (replicas; weak scaling).
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
sys.path.insert(0, ROOT)

METRIC = "Q4_K×q8_1 matmul TOPS & weight GB/s vs nt (1..512), % of HBM/int8 roofline"
WORKLOAD = "decode_gemv_q4k"
NCOPIES = 16

# ncu capture of the fused quantize + MMVQ kernel (nt = 1, 11008 x 4096): dram
# read + write bytes per launch, and the hash of qmm_gemv.cu it was taken on.
# Reported as roofline.traffic only while the kernel source is unchanged.
NCU_TRAFFIC = {"source_sha1": "900ded15ef97c4d3bd765a7119389836497d7b4d", "bytes_per_launch": 25408256}
# The same for the tensor-core GEMM (Q4_K 14336 x 4096, nt = 512; prepass and
# GEMM kernel launches added), keyed on qmm_gemm_tc.cu.
NCU_TRAFFIC_GEMM = {"source_sha1": "768f14d907062ea2d9a3bcbe55ad9bad7d06e4cb",
                    "bytes_per_launch": 2639616 + 38106112 + 951808}

# The cases of the per_nt array: (qtype name, od, K, nt values).
PER_NT = [("Q4_K", 4096, 4096, (1, 2, 4, 8, 16, 128, 512, 2048)),
          ("Q4_K", 14336, 4096, (1, 2, 4, 8, 16, 128, 512, 2048)),
          ("Q6_K", 32000, 4096, (1, 8, 32, 64, 80, 256))]
GEMM_ROOFLINE_CASE = ("Q4_K", 14336, 4096, 512)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def source_sha1(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------- clocks ------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ oracle -----
def time_oracle(cases, budget_s: float, threads: int):
    """Run whole oracle steps (quantize + matmul of every case) until the time
    budget is spent; return (seconds per step, steps)."""
    import oracle
    ora = oracle.Oracle()
    data = [c.generate() for c in cases]
    steps, t0 = 0, time.perf_counter()
    while True:
        for c, (W, x) in zip(cases, data):
            ora.matmul(c.qtype, W, x, c.od, nthreads=threads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s and steps >= 1:
            return el / steps, steps


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------- main ------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(value: float, world: int, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank_step: float, steps: int, ms_max: float, scale: float = 1e9) -> float:
    """Whole-job throughput of N replicas: every rank processes the same units
    per step, so the job's units are world * units * steps, over the slowest
    rank's time (ms_max, already reduced with max_over_ranks)."""
    return world * units_per_rank_step * steps / (ms_max / 1e3) / scale


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args):
    """The CPU oracle as the reference arm.  Each step is a bounded sample of
    the workload -- a rotating contiguous block of rows of each projection,
    sized so that warm-up plus timed steps take about `--ref-seconds` -- and
    the value is weight bytes actually processed per second."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    from quantized_weight_matmul_gb300 import synth
    cases = synth.WORKLOADS[WORKLOAD].cases
    cores = cpu_cores()
    ora = oracle.Oracle()
    data = [c.generate() for c in cases]
    t0 = time.perf_counter()
    for c, (W, x) in zip(cases, data):
        ora.matmul(c.qtype, W, x, c.od, nthreads=cores)
    t_full = time.perf_counter() - t0
    frac = min(1.0, args.ref_seconds / max(1, args.steps + args.warmup) / max(t_full, 1e-9))
    nrows = [max(1, int(c.od * frac)) for c in cases]
    starts = [0] * len(cases)

    def one_step():
        done_bytes = done_macs = 0
        for i, (c, (W, x)) in enumerate(zip(cases, data)):
            r0 = starts[i]
            r1 = min(c.od, r0 + nrows[i])
            ora.matmul(c.qtype, np.ascontiguousarray(W[r0:r1]), x, r1 - r0, nthreads=cores)
            done_bytes += (r1 - r0) * (c.K // 256) * synth.BLOCK_BYTES[c.qtype]
            done_macs += (r1 - r0) * c.K * c.nt
            starts[i] = 0 if r1 >= c.od else r1
        return done_bytes, done_macs

    for _ in range(args.warmup):
        one_step()
    tot_b = tot_m = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        b, m = one_step()
        tot_b += b
        tot_m += m
    t = time.perf_counter() - t0
    value = tot_b / t / 1e9
    sample = (f"{nrows[0]} of {cases[0].od} and {nrows[1]} of {cases[1].od} rows per step "
              f"(rotating row blocks; quantize + matmul)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 dots, f64 sums",
        "data": "synthetic", "tops": 2 * tot_m / t / 1e12,
        "config": {"workload": WORKLOAD, "shapes": [[c.od, c.K] for c in cases], "nt": 1, "qtype": "Q4_K",
                   "x": "N(0,1) + 0.1% x20 outliers", "seed": 0},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class GraphSteps:
    """Replays `n` consecutive steps from at most two CUDA graphs: one of
    `period` steps and one of the remainder n mod period, so that the calls
    stay programmatic dependents of each other inside each graph whatever n
    is.  `capture(m)` returns a graph of m consecutive steps (step k on
    rotating copy k); by default one of `body(k, stream)` per step."""

    def __init__(self, body, period, stream, capture=None):
        self.body, self.period, self.stream = body, period, stream
        self.capture = capture or self._capture_body
        self.graphs = {}

    def _capture_body(self, n):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            cs = torch.cuda.current_stream().cuda_stream
            for k in range(n):
                self.body(k % self.period, cs)
        return g


    def _graph(self, n):
        if n not in self.graphs:
            self.graphs[n] = self.capture(n)
        return self.graphs[n]

    def _chunks(self, n):
        """Graph sizes run(n) replays: one graph of n steps up to `span`
        (a multiple of the rotation period), else whole graphs of `span`
        steps and one of the remainder."""
        if n <= self.span:
            return [n] if n else []
        out = [self.span] * (n // self.span)
        if n % self.span:
            out.append(n % self.span)
        return out

    span = 1024  # steps per graph: graph boundaries break the dependent-launch chain

    def prepare(self, n):
        """Capture the graphs run(n) replays, and replay each new one once,
        outside any timed region: a graph's first launch also uploads it."""
        import torch
        for m in set(self._chunks(n)):
            if m not in self.graphs:
                g = self._graph(m)
                with torch.cuda.stream(self.stream):
                    g.replay()
        torch.cuda.synchronize()

    def run(self, n):
        for m in self._chunks(n):
            self.graphs[m].replay()


def time_calls(torch, stream, call, ncopy, reps):
    """Mean µs of one call(k, stream) over `reps` back-to-back calls replayed
    from one CUDA graph (k cycles over ncopy weight copies), after one
    untimed replay."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cs = torch.cuda.current_stream().cuda_stream
        for k in range(reps):
            rc = call(k % ncopy, cs)
            if rc != 0:
                raise RuntimeError(f"call failed with status {rc}")
    with torch.cuda.stream(stream):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps * 1e3


def case_bytes(c, with_f32_x):
    """Algorithmic HBM bytes of one matmul: weights, q8_1 activations, f32
    outputs (and the f32 activations the whole path reads)."""
    return c.weight_bytes + c.nt * c.K * 1.25 + c.nt * c.od * 4 + (c.nt * c.K * 4 if with_f32_x else 0)


def measure_case(torch, qmm, synth, c, dev, stream, peaks, l2, min_gpu_ms=25.0):
    """Both timings of one case (see per_nt in the module docstring)."""
    W, x = c.generate()
    ncopy = max(2, min(32, int(4 * l2 // c.weight_bytes) + 1))
    Ws = [torch.from_numpy(W).to(dev) for _ in range(ncopy)]
    xd = torch.from_numpy(x).to(dev)
    with torch.cuda.stream(stream):
        xq, xds = qmm.quantize_q8_1(xd)
    xq8 = torch.empty((c.nt, c.K), dtype=torch.int8, device=dev)
    xds8 = torch.empty((c.nt, c.K // 32, 2), dtype=torch.float32, device=dev)
    out = torch.empty((c.nt, c.od), dtype=torch.float32, device=dev)
    route = qmm.qmm_matmul_path(c.qtype, c.od, c.K, c.nt)
    if route < 0:
        raise RuntimeError(f"{c.name}: {qmm.qmm_strerror(route)}")
    use_gemv = route != qmm.QMM_PATH_MMQ
    need_k = 0 if use_gemv else qmm.qmm_gemm_workspace_bytes(c.qtype, c.od, c.K, c.nt)
    need_p = qmm.qmm_matmul_workspace_bytes(c.qtype, c.od, c.K, c.nt)
    ws = qmm.workspace(max(need_k, need_p), dev)

    def kernel(k, s):
        if use_gemv:
            return qmm.qmm_gemv(c.qtype, Ws[k].data_ptr(), xq.data_ptr(), xds.data_ptr(), out.data_ptr(),
                                c.od, c.K, c.nt, s)
        return qmm.qmm_gemm(c.qtype, Ws[k].data_ptr(), xq.data_ptr(), xds.data_ptr(), out.data_ptr(),
                            c.od, c.K, c.nt, ws.data_ptr(), need_k, s)

    def path(k, s):
        return qmm.qmm_matmul(c.qtype, Ws[k].data_ptr(), xd.data_ptr(), xq8.data_ptr(), xds8.data_ptr(),
                              out.data_ptr(), c.od, c.K, c.nt, ws.data_ptr(), need_p,
                              qmm.QMM_FLAG_STATIC_WEIGHTS, s)

    # a first eager call of each (first-call set-up outside any capture), then
    # a rough timing to size the graphs
    with torch.cuda.stream(stream):
        assert kernel(0, stream.cuda_stream) == 0 and path(0, stream.cuda_stream) == 0
    torch.cuda.synchronize()
    est = time_calls(torch, stream, path, ncopy, ncopy)
    reps = int(max(2 * ncopy, min(4000, min_gpu_ms * 1e3 / max(est, 1e-3))))
    reps = (reps + ncopy - 1) // ncopy * ncopy
    us_k = time_calls(torch, stream, kernel, ncopy, reps)
    us_p = time_calls(torch, stream, path, ncopy, reps)
    assert qmm.qmm_sync_status(stream.cuda_stream) == qmm.QMM_OK
    names = {qmm.QMM_PATH_FUSED_MMVQ: "fused quantize+MMVQ (dp4a)", qmm.QMM_PATH_MMVQ: "quantize, MMVQ",
             qmm.QMM_PATH_MMQ: "quantize, MMQ (tcgen05)"}
    tops = 2 * c.macs / (us_k / 1e6) / 1e12
    rec = {"qtype": synth.QTYPE_NAMES[c.qtype], "od": c.od, "K": c.K, "nt": c.nt, "route": names[route],
           "kernel_calls": "qmm_gemv" if use_gemv else "qmm_gemm (operand prepass + GEMM)",
           "us_kernel": us_k, "us_path": us_p, "TOPS": tops,
           "weight_GBs": c.weight_bytes / (us_k / 1e6) / 1e9,
           "hbm_frac": case_bytes(c, False) / (us_k / 1e6) / 1e9 / peaks["hbm_gbs"],
           "tensor_frac": None if use_gemv else tops / peaks["bf16_tflops"],
           "TOPS_path": 2 * c.macs / (us_p / 1e6) / 1e12,
           "weight_GBs_path": c.weight_bytes / (us_p / 1e6) / 1e9,
           "hbm_frac_path": case_bytes(c, True) / (us_p / 1e6) / 1e9 / peaks["hbm_gbs"],
           "copies": ncopy, "reps": reps}
    del Ws, ws
    torch.cuda.empty_cache()
    return rec


def run_per_nt(torch, qmm, synth, dev, stream, peaks):
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    qt = {"Q4_K": synth.Q4_K, "Q6_K": synth.Q6_K}
    recs = []
    for name, od, K, nts in PER_NT:
        for nt in nts:
            c = synth.Case(qt[name], od, K, nt, outliers=True)
            recs.append(measure_case(torch, qmm, synth, c, dev, stream, peaks, l2))
    return recs


def run_gpu(args):
    import torch
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import quantized_weight_matmul_gb300 as qmm
    from quantized_weight_matmul_gb300 import synth

    qmm.load()
    peaks = load_peaks()
    cases = synth.WORKLOADS[WORKLOAD].cases
    stream = torch.cuda.Stream(device=dev)
    st = stream.cuda_stream

    host = [c.generate() for c in cases]
    Wcopies = [[torch.from_numpy(W).to(dev) for _ in range(NCOPIES)] for (W, _) in host]
    xs = [torch.from_numpy(x).to(dev) for (_, x) in host]
    xqs = [torch.empty((c.nt, c.K), dtype=torch.int8, device=dev) for c in cases]
    xdss = [torch.empty((c.nt, c.K // 32, 2), dtype=torch.float32, device=dev) for c in cases]
    outs = [torch.empty((c.nt, c.od), dtype=torch.float32, device=dev) for c in cases]
    wbytes = sum(c.weight_bytes for c in cases)
    macs = sum(c.macs for c in cases)
    routes = [qmm.qmm_matmul_path(c.qtype, c.od, c.K, c.nt) for c in cases]
    assert all(r > 0 for r in routes), routes
    launches_per_step = sum(qmm.PATH_LAUNCHES[r] for r in routes)

    def step(copy, s=st):
        for i, c in enumerate(cases):
            rc = qmm.qmm_matmul(c.qtype, Wcopies[i][copy].data_ptr(), xs[i].data_ptr(), xqs[i].data_ptr(),
                                xdss[i].data_ptr(), outs[i].data_ptr(), c.od, c.K, c.nt, 0, 0,
                                qmm.QMM_FLAG_STATIC_WEIGHTS, s)
            if rc != qmm.QMM_OK:
                raise qmm.QmmError(rc, "qmm_matmul")

    # warm up eagerly once (first-call set-up happens outside any capture),
    # then capture every graph the warm-up and the timed steps replay
    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    steps_g = GraphSteps(step, NCOPIES, stream)
    steps_g.prepare(args.warmup)
    steps_g.prepare(args.steps)
    torch.cuda.synchronize()
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK

    # ---- timed region: exactly K steps.  The clock sampler starts first and
    # the warm-up steps run right before the timed ones, so that the GPU is
    # not idle (and its clocks not lowered) when the timed region begins.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            steps_g.run(args.warmup)
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            steps_g.run(args.steps)
            ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world, dev)
    value = job_rate(world, wbytes, args.steps, ms_max)
    tops = job_rate(world, 2 * macs, args.steps, ms_max, 1e12)
    clocks = clk.summary()
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK

    # ---- roofline: the dominant kernel of the step -- the matmul kernel of the
    # largest projection -- launched back to back over the rotating copies
    # from one CUDA graph (no host cost), exactly as the step launches it
    big = max(range(len(cases)), key=lambda i: cases[i].weight_bytes)
    c = cases[big]
    route = routes[big]

    def kern_run(k, s):
        if route == qmm.QMM_PATH_FUSED_MMVQ:
            return qmm.qmm_matmul(c.qtype, Wcopies[big][k].data_ptr(), xs[big].data_ptr(),
                                  xqs[big].data_ptr(), xdss[big].data_ptr(), outs[big].data_ptr(), c.od, c.K,
                                  c.nt, 0, 0, qmm.QMM_FLAG_STATIC_WEIGHTS, s)
        return qmm.qmm_gemv(c.qtype, Wcopies[big][k].data_ptr(), xqs[big].data_ptr(),
                            xdss[big].data_ptr(), outs[big].data_ptr(), c.od, c.K, c.nt, s)

    kernel_us = time_calls(torch, stream, kern_run, NCOPIES, 32 * NCOPIES)
    act_q8 = c.nt * c.K + c.nt * (c.K // 32) * 8  # q8_1 codes + (d, s)
    if route == qmm.QMM_PATH_FUSED_MMVQ:
        # weights + f32 x read + q8_1 written + f32 out written
        alg_bytes = c.weight_bytes + c.nt * c.K * 4 + act_q8 + c.nt * c.od * 4
        kname = "mmvq_stream_kernel<Q4_K, nt=1, fused> (quantize + MMVQ)"
    else:
        alg_bytes = c.weight_bytes + act_q8 + c.nt * c.od * 4
        kname = "mmvq_stream_kernel (MMVQ)"
    achieved = alg_bytes / (kernel_us / 1e6) / 1e9
    traffic = (NCU_TRAFFIC["bytes_per_launch"]
               if NCU_TRAFFIC["source_sha1"] == source_sha1("quantized_weight_matmul_gb300/csrc/qmm_gemv.cu")
               else None)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": kname, "shape": [c.od, c.K], "kernel_us": kernel_us,
                "alg_bytes_per_launch": alg_bytes, "peak_source": peaks["source"] + " hbm_gbs (copy)"}

    # ---- e2e: host activations in, host outputs back, one C-ABI call per
    # projection.  Every step copies its activations (both projections, one
    # contiguous buffer) from pinned host memory, runs qmm_matmul for both
    # projections and copies the outputs back to pinned host memory.  As in a
    # serving loop the copies are pipelined with compute on their own streams:
    # activations and outputs are double-buffered on the device, step k's
    # copy-in overlaps step k-1's matmuls and its copy-out step k+1's.  The
    # steps are replayed from CUDA graphs of 16 steps (and one of the
    # remainder).
    nx = [cc.nt * cc.K for cc in cases]
    no = [cc.nt * cc.od for cc in cases]
    x_off = np.cumsum([0] + nx)
    o_off = np.cumsum([0] + no)
    xh_all = torch.from_numpy(np.concatenate([x.reshape(-1) for (_, x) in host])).pin_memory()
    oh_all = [torch.empty(sum(no), dtype=torch.float32).pin_memory() for _ in range(2)]
    xd_all = [torch.empty(sum(nx), dtype=torch.float32, device=dev) for _ in range(2)]
    od_all = [torch.empty(sum(no), dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cs = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(cs)
            s_in.wait_event(fork)
            s_out.wait_event(fork)
            done, out_done = {}, {}
            for k in range(n):
                buf = k % 2
                if k >= 2:
                    s_in.wait_event(done[k - 2])  # xd_all[buf] is free again
                with torch.cuda.stream(s_in):
                    xd_all[buf].copy_(xh_all, non_blocking=True)
                x_ready = torch.cuda.Event()
                x_ready.record(s_in)
                cs.wait_event(x_ready)
                if k >= 2:
                    cs.wait_event(out_done[k - 2])  # od_all[buf] has been copied out
                for i, cc in enumerate(cases):
                    rc = qmm.qmm_matmul(cc.qtype, Wcopies[i][k % NCOPIES].data_ptr(),
                                        xd_all[buf][x_off[i]:].data_ptr(),
                                        xqs[i].data_ptr(), xdss[i].data_ptr(), od_all[buf][o_off[i]:].data_ptr(),
                                        cc.od, cc.K, cc.nt, 0, 0, qmm.QMM_FLAG_STATIC_WEIGHTS, cs.cuda_stream)
                    if rc != qmm.QMM_OK:
                        raise qmm.QmmError(rc, "qmm_matmul")
                done[k] = torch.cuda.Event()
                done[k].record(cs)
                s_out.wait_event(done[k])
                with torch.cuda.stream(s_out):
                    oh_all[buf].copy_(od_all[buf], non_blocking=True)
                out_done[k] = torch.cuda.Event()
                out_done[k].record(s_out)
            join_in, join_out = torch.cuda.Event(), torch.cuda.Event()
            join_in.record(s_in)
            join_out.record(s_out)
            cs.wait_event(join_in)
            cs.wait_event(join_out)
        return g

    e2e_steps = max(1, min(args.steps, 16000))
    e2e_g = GraphSteps(None, NCOPIES, stream, capture=e2e_capture)
    e2e_g.span = 256  # the e2e graphs hold three streams' worth of nodes per step
    e2e_g.prepare(args.warmup)
    e2e_g.prepare(e2e_steps)
    with torch.cuda.stream(stream):
        e2e_g.run(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_g.run(e2e_steps)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK
    e2e_ok = all(torch.equal(oh_all[b_], od_all[b_].cpu()) for b_ in range(2))
    e2e = {"value": job_rate(world, wbytes, 1, e2e_ms), "unit": "GB/s",
           "h2d_bytes_per_step": sum(nx) * 4, "d2h_bytes_per_step": sum(no) * 4, "ms_per_step": e2e_ms,
           "steps": e2e_steps, "outputs_copied_back": bool(e2e_ok),
           "launch": "CUDA graphs of up to 256 steps; copy-in, matmuls and copy-out on three streams, "
                     "double-buffered"}
    del Wcopies
    torch.cuda.empty_cache()

    # ---- per_nt: the rest of the metric (rank 0 of each replica set times it
    # on its own GPU; every rank runs the same kernels, so one suffices)
    per_nt, roofline_gemm = None, None
    if rank == 0 and not args.no_per_nt:
        per_nt = run_per_nt(torch, qmm, synth, dev, stream, peaks)
        qn, od_, K_, nt_ = GEMM_ROOFLINE_CASE
        g = next(r for r in per_nt if (r["qtype"], r["od"], r["K"], r["nt"]) == (qn, od_, K_, nt_))
        flops = 2.0 * nt_ * od_ * K_
        ach = flops / (g["us_kernel"] / 1e6) / 1e12
        tr = (NCU_TRAFFIC_GEMM["bytes_per_launch"]
              if NCU_TRAFFIC_GEMM["source_sha1"] == source_sha1("quantized_weight_matmul_gb300/csrc/qmm_gemm_tc.cu")
              else None)
        roofline_gemm = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": ach / peaks["bf16_tflops"], "traffic": tr,
                         "kernel": "gemm_operand_prep_kernel + gemm_tc_kernel<Q4_K, BN=128> (qmm_gemm)",
                         "shape": [od_, K_], "nt": nt_, "kernel_us": g["us_kernel"],
                         "alg_flops_per_launch": flops, "alg_bytes_per_launch": case_bytes(synth.Case(synth.Q4_K, od_, K_, nt_), False),
                         "peak_source": peaks["source"] + " bf16_tflops (cuBLAS bf16 burst); the MMAs are "
                                        "kind::f16, whose dense rate equals bf16's"}

    # ---- CPU baseline: the oracle on this host's cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        sec, nsteps = time_oracle(cases, args.cpu_seconds, cores)
        cpu = {"value": wbytes / sec / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "cpu": cpu_model(),
               "sample": f"{nsteps} whole steps (both projections, quantize + matmul), {args.cpu_seconds:.0f} s budget"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8 dots (dp4a), f32 rescale",
            "data": "synthetic", "tops": tops,
            "config": {"workload": WORKLOAD, "shapes": [[cc.od, cc.K] for cc in cases], "nt": 1,
                       "qtype": "Q4_K", "x": "N(0,1) + 0.1% x20 outliers", "seed": 0,
                       "parallelism": f"replicas x{world}",
                       "l2": f"{NCOPIES} rotating weight copies ({NCOPIES * wbytes / 1e6:.0f} MB > L2)",
                       "graphs": "CUDA graphs of up to 1024 consecutive steps"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks, "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "per_nt": per_nt, "roofline_gemm": roofline_gemm,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Timing of every case of every workload family (see measure_case); one
    JSON line per case."""
    import torch
    import quantized_weight_matmul_gb300 as qmm
    from quantized_weight_matmul_gb300 import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    names = args.families.split(",") if args.families else list(synth.WORKLOADS)
    fams = [(fam, synth.WORKLOADS[fam].cases) for fam in names]
    if args.shape:  # e.g. Q4_K:44032x4096x1 -- one extra case, seeded like the others
        fams = []
        for spec in args.shape.split(","):
            qt, dims = spec.split(":")
            od_, K_, nt_ = (int(v) for v in dims.split("x"))
            fams.append(("shape", [synth.Case({"Q4_K": synth.Q4_K, "Q6_K": synth.Q6_K}[qt], od_, K_, nt_)]))
    for fam, fcases in fams:
        for c in fcases:
            if args.case and c.name != args.case:
                continue
            rec = measure_case(torch, qmm, synth, c, dev, stream, peaks, l2)
            rec["case"] = c.name
            print(json.dumps(rec), flush=True)
    return 0


def run_profile(args):
    """A fixed number of eager calls of one case, for ncu captures (not a
    timing): --profile QTYPE:ODxKxNT[:path|gemv|gemm] --calls N.  `path` is
    qmm_matmul from f32 x (the decode route's fused kernel at nt <= 4), `gemv`
    / `gemm` the matmul on q8_1 input; two weight copies alternate."""
    import torch
    import quantized_weight_matmul_gb300 as qmm
    from quantized_weight_matmul_gb300 import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    parts = args.profile.split(":")
    qt, dims = parts[0], parts[1]
    how = parts[2] if len(parts) > 2 else "path"
    od, K, nt = (int(v) for v in dims.split("x"))
    c = synth.Case({"Q4_K": synth.Q4_K, "Q6_K": synth.Q6_K}[qt], od, K, nt, outliers=True)
    W, x = c.generate()
    Ws = [torch.from_numpy(W).to(dev) for _ in range(2)]
    xd = torch.from_numpy(x).to(dev)
    xq, xds = qmm.quantize_q8_1(xd)
    xq8 = torch.empty_like(xq)
    xds8 = torch.empty_like(xds)
    out = torch.empty((nt, od), dtype=torch.float32, device=dev)
    need = max(qmm.qmm_matmul_workspace_bytes(c.qtype, od, K, nt), qmm.qmm_gemm_workspace_bytes(c.qtype, od, K, nt))
    ws = qmm.workspace(need, dev)
    s = torch.cuda.current_stream().cuda_stream
    for k in range(args.calls):
        w = Ws[k % 2].data_ptr()
        if how == "path":
            rc = qmm.qmm_matmul(c.qtype, w, xd.data_ptr(), xq8.data_ptr(), xds8.data_ptr(), out.data_ptr(), od, K,
                                nt, ws.data_ptr(), need, qmm.QMM_FLAG_STATIC_WEIGHTS, s)
        elif how == "gemv":
            rc = qmm.qmm_gemv(c.qtype, w, xq.data_ptr(), xds.data_ptr(), out.data_ptr(), od, K, nt, s)
        else:
            rc = qmm.qmm_gemm(c.qtype, w, xq.data_ptr(), xds.data_ptr(), out.data_ptr(), od, K, nt, ws.data_ptr(),
                              need, s)
        if rc != qmm.QMM_OK:
            raise qmm.QmmError(rc, how)
    torch.cuda.synchronize()
    if qmm.qmm_sync_status(s) != qmm.QMM_OK:
        raise RuntimeError("device status word set")
    print(json.dumps({"profile": args.profile, "calls": args.calls}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--families", default="")
    ap.add_argument("--case", default="", help="sweep: only the case with this name")
    ap.add_argument("--shape", default="", help="sweep: one case of this shape instead, QTYPE:ODxKxNT")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-nt", action="store_true", help="leave out the per_nt array and roofline_gemm")
    ap.add_argument("--profile", default="", help="QTYPE:ODxKxNT[:path|gemv|gemm]: eager calls for ncu, no timing")
    ap.add_argument("--calls", type=int, default=6, help="--profile: number of calls")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    if args.sweep:
        return run_sweep(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
