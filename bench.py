#!/usr/bin/env python
"""Benchmark of the group-quantized INT4-weight GEMM (W4A16 / W4A8) on GB300.

Default workload ("sweep"): every shape of the five configurations in one run.
  c0  W4A16 asym M16 K256 N256 g128 fp16 (a launch-latency case)
  c1  W4A16 asym decode M{1,4,16} x N{4096,11008}, K4096 (weight-bandwidth bound)
  c2  W4A16 asym batched M{64,128,256}, K = N = 8192, g128 and per-channel
  c3  W4A16 asym prefill, bf16 activations: M4096 K5120 N17408 and M4096 K17408 N5120
  c4  W4A8 per-token int8 activations, folded signed scales, M{16,256,2048} K5120 N17408
One "step" runs all 18 GEMMs once.  Each shape has its own resident copies of the
packed weights, enough of them to span more than twice the L2 size, and a step
uses the next copy.  `value` is the c3 prefill rate in TFLOP/s: 2*M*N*K of the c3
calls over their device time inside the K timed steps.  `per_shape` gives every
shape's TFLOP/s and weight GB/s, each the median of 20 windows of >= 50 ms of
CUDA-graph replays.  `roofline` is the prefill kernel against the dense bf16
tensor peak; `rooflines` holds each regime's kernel against its own bound.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl wq|reference]
                    [--workload sweep|c0|c1|c2|c3|c4|moe|moe8|swiglu|mlp]

--impl reference times the CPU oracle (plain C, fp64, naive loops) on a bounded
sample of the same workload.  Under torchrun each rank runs an independent
replica on its own GPU (the GEMM has no exchange step); rank 0 prints one JSON
line.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "W4A16 GEMM TFLOPS & weight GB/s vs M on 1 GB300; % of HBM / tensor-core roofline"
L2_BYTES = 129 * 2 ** 20
PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SWEEP = ("c0", "c1", "c2", "c3", "c4")
HEADLINE = "c3"
WORKLOAD_NAMES = {
    "sweep": "sweep of c0-c4 (18 GEMM shapes), headline c3 prefill",
    "c0": "W4A16 asym M16 K256 N256 g128 fp16",
    "c1": "W4A16 asym decode GEMV M{1,4,16} x N{4096,11008} K4096 g128 fp16",
    "c2": "W4A16 asym batched M{64,128,256} K8192 N8192 g128 and per-channel fp16",
    "c3": "W4A16 asym prefill M4096 K5120 N17408 + M4096 K17408 N5120 g128 bf16",
    "c4": "W4A8 sym M{16,256,2048} K5120 N17408 g128 int8 per-token",
    "moe": "W4A16 asym grouped (mixture of experts): 16 tokens top-1 over 8 experts, K256 N7168 g128 fp16",
    "moe8": "W4A8 zero-point grouped (mixture of experts): 16 int8 per-token rows top-1 over 8 experts, K256 N7168 g128",
    "swiglu": "W4A16 asym fused SwiGLU gate/up pair, decode M{1,4} K4096 N11008 (x2 projections) g128 fp16",
    "mlp": "W4A16 asym decode MLP block M{1,4}: gate/up pair K4096 N11008 (x2, SwiGLU) then down K11008 N4096, "
           "g128 fp16, one persistent chain launch per block",
}
# The unit of a single-configuration workload's `value`: TFLOP/s where the tensor cores
# bound most of its shapes, weight GB/s where the weight stream does.
TENSOR_CONFIGS = ("c2", "c3", "c4")
SHAPE_KEYS = ("M", "K", "N", "group_size", "a_dtype", "a_std", "mode")


# ----------------------------------------------------------------------------- helpers
def workload_shapes(workload: str):
    """(seed, shape) pairs of a workload; each shape carries its configuration name."""
    cfgs = SWEEP if workload == "sweep" else (workload,)
    out = []
    for c in cfgs:
        for seed, s in synth.shapes(c):
            d = dict(s)
            d["cfg"] = c
            out.append((seed, d))
    return out


def inputs_of(seed, s, **kw):
    return synth.make_inputs(seed, **{k: s[k] for k in SHAPE_KEYS}, **kw)


def label(s) -> str:
    t = f"{s.get('cfg', '?')} M{s['M']} K{s['K']} N{s['N']}"
    return t + (" per-channel" if s["group_size"] in (-1, s["K"]) else "")


def weight_bytes(s) -> int:
    K, N = s["K"], s["N"]
    G = synth.num_groups(K, s["group_size"])
    b = K * N // 2 + G * N * 2
    if s["mode"] == "w4a16":
        b += G * N * 4
    return b


def io_bytes(s) -> int:
    xb = 1 if s["mode"] == "w4a8" else 2
    return s["M"] * s["K"] * xb + s["M"] * s["N"] * 2 + (s["M"] * 4 if s["mode"] == "w4a8" else 0)


def flops(s) -> int:
    return 2 * s["M"] * s["N"] * s["K"]


def kernels_for(s):
    """The kernels one GEMM call of this shape launches, as the library dispatches it:
    W4A16 up to 8 tokens the weight-streaming kernel, 9..16 tokens the tcgen05 decode
    kernel, beyond that the correction pre-pass and the large-M kernel; W4A8 with
    9..16 tokens the activation pre-pass and the e4m3 decode kernel, beyond that the
    int8 -> fp16 pre-pass and the large-M kernel."""
    M = s["M"]
    gemm = ["gemm_kernel"] * (2 if M > 16 and large_m_tail(M, s["N"], s["K"]) else 1)
    if s["mode"] == "w4a8":
        return ["decode_prep_kernel", "decode_kernel"] if M <= 16 else ["i8_to_f16_kernel"] + gemm
    if M <= 8:
        return ["gemv_kernel"]
    if M <= 16:
        return ["decode16_kernel"]
    return ["corr_prep_kernel"] + gemm


def large_m_tail(M, N, K, sms=152, max_splits=8) -> bool:
    """Whether a large-M call runs its last, partial wave of tiles as a second launch
    split along K (the library's plan: token tiles of 32/64/128/256, two CTAs per SM
    up to 64 tokens, as many K segments as fill one wave; with one segment per tile
    of at least 96 k-blocks, a last wave at most half full goes to the second launch)."""
    bt = 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
    slots = 2 * sms if bt <= 64 else sms
    tiles = (N // 128) * (-(-M // bt))
    kb = K // 128
    splits = min(max(1, slots // tiles), max_splits, kb)
    kbps = -(-kb // splits)
    splits = -(-kb // kbps)
    if splits != 1 or tiles <= slots or kb < 96:
        return False
    rest = tiles % slots
    if rest == 0 or 2 * rest > slots:
        return False
    ts = min(slots // rest, max_splits, kb)
    kbps = -(-kb // ts)
    return -(-kb // kbps) > 1


def kernel_launches(s) -> int:
    return len(kernels_for(s))


def source_hash(sources) -> str:
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic(kernel: str, shape):
    """DRAM bytes of one launch of `kernel` on `shape` from a committed ncu capture
    (profiles/traffic.json), or None when no record matches or the kernel's sources
    changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f)
    for rec in recs.get("records", []):
        sh = rec["shape"]
        if rec["kernel"] != kernel or any(sh[k] != shape[k] for k in ("M", "K", "N", "group_size")):
            continue
        if source_hash(rec["sources"]) != rec["source_sha256"]:
            return None
        return rec
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAK_FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self) -> float:
        return time.perf_counter()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float = None, t1: float = None):
        """Median SM clock, max clock and the throttle reasons seen between t0 and t1."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


STEPS_PER_GRAPH = 8  # steps captured back to back in one CUDA graph (launch cost amortised)


def build_step_graphs(torch, stream, reps: int, step_fn, steps_per_graph: int):
    """CUDA graphs holding steps_per_graph consecutive steps each, the weight copy rotating
    step by step (graph g runs copies g*spg .. g*spg+spg-1 mod reps), plus one single-step
    graph per copy for a remainder.  Returns (multi, single)."""
    multi, single = [], []
    with torch.cuda.stream(stream):
        for g in range(reps):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for j in range(steps_per_graph):
                    step_fn((g * steps_per_graph + j) % reps)
            multi.append(gr)
        for r in range(reps):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                step_fn(r)
            single.append(gr)
    return multi, single


def replay_steps(multi, single, steps: int, steps_per_graph: int):
    """Run exactly `steps` steps: whole multi-step graphs, then single steps."""
    full, rest = divmod(steps, steps_per_graph)
    for i in range(full):
        multi[i % len(multi)].replay()
    base = full * steps_per_graph
    for j in range(rest):
        single[(base + j) % len(single)].replay()


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The job's time: the slowest rank's (all-reduce MAX over the process group)."""
    if ws <= 1:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(ws: int, units_per_rank_step: float, ms_per_step: float, scale: float = 1e9) -> float:
    """Whole-job throughput: every rank processes units_per_rank_step per step (weak scaling)."""
    return ws * units_per_rank_step / (ms_per_step * 1e-3) / scale


def cpu_threads() -> int:
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def headline_unit(workload: str) -> str:
    return "TFLOP/s" if workload == "sweep" or workload in TENSOR_CONFIGS else "GB/s"


# ----------------------------------------------------------------------------- oracle arm
class OracleProblem:
    """One shape's seeded inputs in the oracle's form, and its fp64 product on a column
    window (the oracle as it stands: plain C, naive loops, OpenMP over rows)."""

    def __init__(self, seed, s):
        import oracle
        self.s = s
        d = inputs_of(seed, s)
        self.q = d["q"]
        if s["mode"] == "w4a8":
            self.Xq, self.xs = oracle.quantize_per_token(d["A"])
            self.qf, self.sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), s["group_size"])
        else:
            self.A = oracle.activations_to_double(d["A"], s["a_dtype"])
            self.sb = oracle.half_bits(d["scale"])
            self.zb = oracle.half_bits(d["zero"])

    def run(self, c0: int, c1: int):
        """Columns [c0, c1) of the product; returns (flops, weight bytes) of that window."""
        import oracle
        s = self.s
        N = s["N"]
        c0, c1 = c0 % N, c0 % N + min(c1 - c0, N)
        c1 = min(c1, N)
        if s["mode"] == "w4a8":
            oracle.gemm_w4a8(self.Xq, self.xs, self.qf, self.sf, s["group_size"], cols=(c0, c1))
        else:
            oracle.gemm_asym_plain(self.A, self.q, self.sb, self.zb, s["group_size"], cols=(c0, c1))
        w = c1 - c0
        G = synth.num_groups(s["K"], s["group_size"])
        wb = s["K"] * w // 2 + G * w * 2 + (G * w * 4 if s["mode"] == "w4a16" else 0)
        return 2 * s["M"] * s["K"] * w, wb


def oracle_rate(shapes, budget_s: float, cols: int):
    """Run the oracle on successive column windows of every shape until budget_s has
    passed; returns (TFLOP/s, weight GB/s, seconds, windows per shape)."""
    probs = [OracleProblem(seed, s) for seed, s in shapes]
    done_f = done_b = 0
    passes = 0
    t0 = time.perf_counter()
    while True:
        for p in probs:
            f, b = p.run(passes * cols, passes * cols + cols)
            done_f += f
            done_b += b
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done_f / el / 1e12, done_b / el / 1e9, el, passes


def run_reference(args, shapes, ws, rank):
    """The CPU oracle on the arm's own metric: every step computes one column window of
    every shape of the headline configuration (the whole workload's, for a single
    configuration) and the rate is counted over the K timed steps."""
    if rank != 0:
        return 0
    workload = getattr(args, "workload", "sweep")
    unit = headline_unit(workload)
    head = [(seed, s) for seed, s in shapes if s.get("cfg", workload) == HEADLINE] if workload == "sweep" else shapes
    probs = [OracleProblem(seed, s) for seed, s in head]
    cols = 64 if unit == "TFLOP/s" else 256
    for i in range(args.warmup):
        for p in probs:
            p.run(i * 8, i * 8 + 8)
    done_f = done_b = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        for p in probs:
            f, b = p.run(i * cols, i * cols + cols)
            done_f += f
            done_b += b
    el = time.perf_counter() - t0
    val = done_f / el / 1e12 if unit == "TFLOP/s" else done_b / el / 1e9
    threads = cpu_threads()
    sample = (f"{args.steps} steps, step i the columns [{cols} i, {cols} i + {cols}) of "
              + ", ".join(label(p.s) for p in probs) + "; all rows and the full K, fp64 naive loops")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 9), "unit": unit,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / max(1, args.steps), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": WORKLOAD_NAMES.get(workload, workload), "sampled": True,
                   "shapes": [label(p.s) for p in probs]},
        "cpu_baseline": {"value": round(val, 9), "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 9), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def setup_problem(torch, wq, dev, seed, s, min_rot_bytes: int, max_copies: int = 64):
    """Pack one shape's seeded inputs on the device: the activations, enough copies of the
    packed weights to span min_rot_bytes (so that consecutive calls read their weights
    from HBM), the output and the GEMM workspace."""
    d = inputs_of(seed, s)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    gs = s["group_size"]
    if s["mode"] == "w4a8":
        Bp, S = wq.pack_w4a8(cu(d["q"]), cu(d["scale"]), gs)
        dl = None
        Xq, xs = wq.quantize_per_token(cu(d["A"]))
        X = (Xq, xs)
    else:
        Bp, S, dl = wq.pack_w4a16(cu(d["q"]), cu(d["scale"]), cu(d["zero"]), gs)
        X = cu(d["A"].view(np.int16)).view(torch.bfloat16) if s["a_dtype"] == "bf16" else cu(d["A"])
    wb = weight_bytes(s)
    copies = min(max_copies, max(1, math.ceil(min_rot_bytes / wb) + 1))
    w = [(Bp, S, dl)] + [(Bp.clone(), S.clone(), dl.clone() if dl is not None else None)
                         for _ in range(copies - 1)]
    variant = wq.VARIANT_W4A8 if s["mode"] == "w4a8" else wq.VARIANT_W4A16
    need = wq.workspace_size(variant, s["M"], s["N"], s["K"], gs)
    return {"s": s, "seed": seed, "w": w, "X": X,
            "Y": torch.empty((s["M"], s["N"]), dtype=torch.float16, device=dev),
            "ws": torch.zeros(max(need, 4096), dtype=torch.uint8, device=dev),
            "A_host": d["A"] if s.get("cfg") == HEADLINE else None}


def call(wq, p, r):
    """One GEMM call of problem p on weight copy r (mod the copies it has)."""
    s = p["s"]
    Bp, S, dl = p["w"][r % len(p["w"])]
    if s["mode"] == "w4a8":
        return wq.gemm_w4a8(p["X"][0], p["X"][1], Bp, S, s["group_size"], out=p["Y"], workspace=p["ws"])
    return wq.gemm_w4a16(p["X"], Bp, S, dl, s["group_size"], out=p["Y"], workspace=p["ws"])


def time_shape(torch, wq, stream, p, windows: int, min_window_ms: float):
    """Per-call device time of one shape: a CUDA graph of consecutive calls on rotating
    weight copies, replayed in `windows` windows of at least min_window_ms each;
    returns (median, min, max) microseconds per call over the windows."""
    per = max(8, 2 * len(p["w"]))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for j in range(per):
                call(wq, p, j)
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    reps = max(1, math.ceil(min_window_ms / max(1e-3, e0.elapsed_time(e1))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(windows)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 / (reps * per) for a, b in evs)
    del g
    return statistics.median(us), us[0], us[-1], reps * per


def regime_roofline(rows, kernel, bound, peaks, peaks_src, what):
    """Aggregate fraction of a kernel over its shapes: algorithmic bytes (bound "hbm") or
    FLOPs (bound "tensor") over the summed per-call times."""
    sel = [r for r in rows if r["kernel"] == kernel and r["_use"](bound)]
    if not sel:
        return None
    t = sum(r["us"] for r in sel) * 1e-6
    if bound == "hbm":
        ach = sum(r["_alg"] for r in sel) / t / 1e9
        pk = peaks["hbm_gbs"]
        src = f"{peaks_src} hbm_gbs (copy)"
        unit = "GB/s"
    else:
        ach = sum(r["_flops"] for r in sel) / t / 1e12
        pk = peaks["bf16_tflops"]
        src = f"{peaks_src} bf16_tflops (burst, cuBLAS bf16; fp16 runs at the bf16 rate)"
        unit = "TFLOP/s"
    return {"bound": bound, "kernel": kernel, "achieved": round(ach, 1), "peak": pk, "unit": unit,
            "frac": round(ach / pk, 4), "peak_source": src, "shapes": [r["shape"] for r in sel], "what": what}


def run_gpu(args, shapes, ws, rank, local):
    import torch

    import weight_only_int4_g128_gb300 as wq

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wq.load_library(build_if_missing=True)
    if not wq.device_supported(local):
        raise RuntimeError("not an sm_103 device")
    # The weights are packed once before the timed region and never written again, so
    # the decode kernels may start copying them before the preceding GEMM finishes.
    wq.set_weight_prefetch(True)
    workload = args.workload
    unit = headline_unit(workload)

    probs = [setup_problem(torch, wq, dev, seed, s, 2 * L2_BYTES) for seed, s in shapes]
    cfg_order = [c for c in SWEEP if any(p["s"]["cfg"] == c for p in probs)]
    groups = {c: [p for p in probs if p["s"]["cfg"] == c] for c in cfg_order}
    head_cfg = HEADLINE if workload == "sweep" else workload
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)

    def step(r, evs=None):
        for i, c in enumerate(cfg_order):
            if evs is not None:
                evs[i].record(stream)
            for p in groups[c]:
                call(wq, p, r)
        if evs is not None:
            evs[-1].record(stream)

    with torch.cuda.stream(stream):
        for r in range(args.warmup):
            step(r)
    torch.cuda.synchronize()

    # --- timed region: exactly K steps, one event at each configuration boundary
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_timed0 = clocks.mark()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(cfg_order) + 1)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for t in range(args.steps):
            step(args.warmup + t, evs[t])
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    t_timed1 = clocks.mark()
    ms_total = max_over_ranks(evs[0][0].elapsed_time(evs[-1][-1]), ws, dev)
    ms_per_step = ms_total / args.steps
    cfg_ms = {c: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i, c in enumerate(cfg_order)}
    cfg_ms = {c: max_over_ranks(v, ws, dev) for c, v in cfg_ms.items()}
    head_probs = groups[head_cfg]
    head_flops = sum(flops(p["s"]) for p in head_probs)
    head_wb = sum(weight_bytes(p["s"]) for p in head_probs)
    if unit == "TFLOP/s":
        value = job_rate(ws, head_flops, cfg_ms[head_cfg], 1e12)
    else:
        value = job_rate(ws, head_wb, cfg_ms[head_cfg])
    launches_per_step = sum(kernel_launches(p["s"]) for p in probs)
    peaks, peaks_src = load_peaks()

    if args.quick:
        clocks.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(value, 3), "unit": unit,
                              "ms_per_step": round(ms_per_step, 6), "quick": True,
                              "config_ms_per_step": {c: round(v, 6) for c, v in cfg_ms.items()},
                              "clocks": clocks.summary(t_timed0, t_timed1)}), flush=True)
        return 0

    # --- per-shape device time: median of 20 windows of >= 50 ms of graph replays
    rows = []
    for p in probs:
        s = p["s"]
        us, us_lo, us_hi, calls = time_shape(torch, wq, stream, p, args.windows, args.window_ms)
        alg = weight_bytes(s) + io_bytes(s)
        t = us * 1e-6
        t_hbm = alg / (peaks["hbm_gbs"] * 1e9)
        t_tc = flops(s) / (peaks["bf16_tflops"] * 1e12)
        kern = kernels_for(s)[-1]
        row = {"shape": label(s), "config": s["cfg"], "M": s["M"], "K": s["K"], "N": s["N"],
               "group_size": s["group_size"], "kernels": kernels_for(s), "kernel": kern,
               "us": round(us, 3), "us_min": round(us_lo, 3), "us_max": round(us_hi, 3),
               "calls_per_window": calls, "windows": args.windows,
               "tflops": round(flops(s) / t / 1e12, 3),
               "weight_GBps": round(weight_bytes(s) / t / 1e9, 1),
               "alg_GBps": round(alg / t / 1e9, 1),
               "frac_hbm": round(alg / t / 1e9 / peaks["hbm_gbs"], 4),
               "frac_tensor": round(flops(s) / t / 1e12 / peaks["bf16_tflops"], 4),
               "bound": "latency" if s["cfg"] == "c0" else ("hbm" if t_hbm >= t_tc else "tensor"),
               "copies": len(p["w"])}
        row["_alg"], row["_flops"] = alg, flops(s)
        rows.append(row)
    t_shapes1 = clocks.mark()

    def use(r, b):
        return r["bound"] == b or (b == "hbm" and r["M"] <= 16 and r["config"] != "c0")
    for r in rows:
        r["_use"] = (lambda b, r=r: use(r, b))
    rooflines = {}
    for name, kern, bound, what in [
            ("decode_w4a16_le8", "gemv_kernel", "hbm", "W4A16 decode, M <= 8 (c1)"),
            ("decode_w4a16_9to16", "decode16_kernel", "hbm", "W4A16 decode, M 9..16 (c1 M16)"),
            ("decode_w4a8_9to16", "decode_kernel", "hbm", "W4A8 decode, M 16 (c4 M16)"),
            ("large_m_tensor", "gemm_kernel", "tensor", "large M: c2 M128/M256, c3, c4 M256/M2048")]:
        rl = regime_roofline(rows, kern, bound, peaks, peaks_src, what)
        if rl:
            rooflines[name] = rl
    # the headline configuration's own rows
    for c in cfg_order:
        crow = [r for r in rows if r["config"] == c]
        t = sum(r["us"] for r in crow) * 1e-6
        rooflines.setdefault("per_config", {})[c] = {
            "tflops": round(sum(r["_flops"] for r in crow) / t / 1e12, 3),
            "weight_GBps": round(sum(weight_bytes(p["s"]) for p in groups[c]) / t / 1e9, 1),
            "us_per_step": round(t * 1e6, 3)}
    for r in rows:
        del r["_alg"], r["_flops"], r["_use"]

    # --- the headline kernel's roofline, from the timed steps themselves
    hk = kernels_for(head_probs[0]["s"])[-1]
    n_launch = len(head_probs)
    if unit == "TFLOP/s":
        achieved = head_flops / (cfg_ms[head_cfg] * 1e-3) / 1e12
        pk = peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk, "unit": "TFLOP/s",
                    "frac": round(achieved / pk, 4),
                    "peak_source": f"{peaks_src} bf16_tflops (burst, cuBLAS bf16 8192^3)"}
    else:
        alg = sum(weight_bytes(p["s"]) + io_bytes(p["s"]) for p in head_probs)
        achieved = alg / (cfg_ms[head_cfg] * 1e-3) / 1e9
        pk = peaks["hbm_gbs"]
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk, "unit": "GB/s",
                    "frac": round(achieved / pk, 4), "peak_source": f"{peaks_src} hbm_gbs (copy)"}
    tr = load_traffic(hk, head_probs[0]["s"])
    roofline.update({
        "kernel": f"wq::{hk}",
        "calls_per_step": n_launch,
        "launches_per_step": sum(kernel_launches(p["s"]) for p in head_probs),
        "time": (f"device time of the {head_cfg} calls inside the {args.steps} timed steps "
                 f"(CUDA events on the launching stream), {1e3 * cfg_ms[head_cfg] / n_launch:.1f} us per call"
                 + (" including its pre-pass launch" if len(kernels_for(head_probs[0]['s'])) > 1 else "")),
        "traffic": tr["dram_bytes_per_launch"] if tr else None,
        "traffic_launch": ({"shape": tr["shape"], "algorithmic_bytes": tr["algorithmic_bytes_per_launch"],
                            "capture": tr["capture"]} if tr else None)})

    # --- end to end through the host-buffer C-ABI entry: per step, every headline call
    # copies its activations in from pinned host memory, runs and copies Y back out;
    # synchronised each step
    e2e = None
    if all(p["s"]["mode"] == "w4a16" for p in head_probs):
        hx, hy, hws = [], [], []
        for p in head_probs:
            s = p["s"]
            a = torch.from_numpy(np.ascontiguousarray(p["A_host"] if p["A_host"] is not None
                                                      else inputs_of(p["seed"], s)["A"]).view(np.int16))
            hx.append((a.view(torch.bfloat16) if s["a_dtype"] == "bf16" else a.view(torch.float16)).pin_memory())
            hy.append(torch.empty((s["M"], s["N"]), dtype=torch.float16).pin_memory())
            need = int(wq.load_library().wq_host_workspace_size(wq.VARIANT_W4A16, s["M"], s["N"], s["K"],
                                                                 s["group_size"], wq.DTYPE_F16))
            hws.append(torch.empty(need, dtype=torch.uint8, device=dev))
        n_e2e = max(10, args.steps)
        with torch.cuda.stream(stream):
            for i in range(2 + n_e2e):
                if i == 2:
                    torch.cuda.synchronize()
                    t0 = time.perf_counter()
                for j, p in enumerate(head_probs):
                    Bp, S, dl = p["w"][i % len(p["w"])]
                    wq.gemm_w4a16_host(hx[j], Bp, S, dl, p["s"]["group_size"], out=hy[j], workspace=hws[j])
                stream.synchronize()
        e2e_s = (time.perf_counter() - t0) / n_e2e
        e2e_val = (job_rate(ws, head_flops, e2e_s * 1e3, 1e12) if unit == "TFLOP/s"
                   else job_rate(ws, head_wb, e2e_s * 1e3))
        e2e = {"value": round(e2e_val, 3), "unit": unit,
               "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in hx),
               "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in hy),
               "api": "wq_gemm_w4a16_host (C ABI, host buffers) through its Python binding",
               "note": f"{n_e2e} steps of the {head_cfg} calls, wall clock, each call copying X in from pinned "
                       "host memory and Y back, the stream synchronised every step"}
    t_end = clocks.mark()
    clocks.stop()
    clk = clocks.summary(t_timed0, t_end)
    clk["timed_steps_samples"] = clocks.summary(t_timed0, t_timed1)["samples"]

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if head_cfg == "c3" else "f16",
        "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": WORKLOAD_NAMES[workload], "headline": f"{head_cfg}: {WORKLOAD_NAMES[head_cfg]}",
                   "value_is": (f"{unit} of the {head_cfg} calls over their device time inside the timed steps"),
                   "config_ms_per_step": {c: round(v, 6) for c, v in cfg_ms.items()},
                   "shapes": [label(p["s"]) for p in probs],
                   "l2": ("every shape rotates over copies of its packed weights spanning > 2x L2 (c0: 64 "
                          "copies of 36 KB, L2-resident: a launch-latency case); a step reads ~1 GB of "
                          "distinct weights, activations and outputs, so no shape finds its weights in L2"),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "launch": "eager launches, programmatic dependent launch, weight prefetch enabled; "
                             "per-shape rows: CUDA graphs of consecutive calls"},
        "roofline": roofline,
        "rooflines": rooflines,
        "per_shape": rows,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        head_shapes = [(p["seed"], p["s"]) for p in head_probs]
        cols = 64 if unit == "TFLOP/s" else 256
        tfl, gbs, el, passes = oracle_rate(head_shapes, args.cpu_seconds, cols)
        line["cpu_baseline"] = {
            "value": round(tfl if unit == "TFLOP/s" else gbs, 9), "unit": unit, "cores": cpu_threads(),
            "kind": "oracle", "seconds": round(el, 2),
            "sample": (f"{passes} column window(s) of {cols} columns of each of "
                       + ", ".join(label(s) for _, s in head_shapes) + "; all rows, full K, fp64 naive loops")}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- MoE workload
def moe_weight_bytes(d) -> int:
    """Weight bytes the grouped call must read: codes, scales and delta of every expert that
    received at least one token."""
    E, K, N = d["q"].shape
    G = d["scale"].shape[1]
    live = int(np.count_nonzero(np.diff(d["offsets"])))
    return live * (K * N // 2 + G * N * 6)


def moe_oracle(d, budget_s, w4a8=False):
    import oracle
    A = d["A"].astype(np.float64)
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    if w4a8:
        Xq, xs = oracle.quantize_per_token(d["A"])
    n = 0
    t0 = time.perf_counter()
    while True:
        if w4a8:
            oracle.gemm_grouped_w4a8(Xq, xs, d["offsets"], d["q"], sb, zb, synth.MOE["group_size"])
        else:
            oracle.gemm_grouped_asym(A, d["offsets"], d["q"], sb, zb, synth.MOE["group_size"])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return n * moe_weight_bytes(d) / el / 1e9, el, threads, f"{n} full grouped call(s), fp64 naive loops"


def run_moe(args, ws, rank, local):
    d = synth.moe_inputs()
    w4a8 = args.workload == "moe8"
    name = WORKLOAD_NAMES[args.workload]
    if args.impl == "reference":
        if rank != 0:
            return 0
        gbs, el, threads, sample = moe_oracle(d, max(2.0, min(20.0, 4.0 * args.steps)), w4a8)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
            "config": {"workload": name, "sampled": False},
            "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return 0
    import torch
    import weight_only_int4_g128_gb300 as wq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wq.load_library(build_if_missing=True)
    if not wq.device_supported(local):
        raise RuntimeError("not an sm_103 device")
    wq.set_weight_prefetch(True)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    E = d["q"].shape[0]
    gs = synth.MOE["group_size"]
    packs = [wq.pack_w4a16(cu(d["q"][e]), cu(d["scale"][e]), cu(d["zero"][e]), gs) for e in range(E)]
    w0 = (torch.stack([p_[0] for p_ in packs]), torch.stack([p_[1] for p_ in packs]),
          torch.stack([p_[2] for p_ in packs]))
    wb = moe_weight_bytes(d)
    set_bytes = sum(t.numel() * t.element_size() for t in w0)
    reps = max(1, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
    W = [w0] + [tuple(t.clone() for t in w0) for _ in range(reps - 1)]
    offs = [int(v) for v in d["offsets"]]
    X = cu(d["A"])
    Y = torch.empty((X.shape[0], w0[1].shape[-1]), dtype=torch.float16, device=dev)
    if w4a8:
        Xq, xs = wq.quantize_per_token(X)
        gws = torch.zeros(max(wq.workspace_size(wq.VARIANT_W4A8_ASYM, offs[e + 1] - offs[e], Y.shape[1],
                                                X.shape[1], gs) for e in range(E) if offs[e + 1] > offs[e]),
                          dtype=torch.uint8, device=dev)

    def grouped(r, x=None, out=None):
        if w4a8:
            xq, xsc = (Xq, xs) if x is None else x
            return wq.gemm_w4a8_grouped(xq, xsc, *W[r], offs, gs, out=Y if out is None else out, workspace=gws)
        return wq.gemm_w4a16_grouped(X if x is None else x, *W[r], offs, gs, out=Y if out is None else out)

    for r in range(reps):
        grouped(r)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    spg = 4 * STEPS_PER_GRAPH
    graphs, graphs1 = build_step_graphs(torch, stream, reps, grouped, spg)
    with torch.cuda.stream(stream):
        replay_steps(graphs, graphs1, args.warmup, spg)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        e0.record(stream)
        replay_steps(graphs, graphs1, args.steps, spg)
        e1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks.stop()
    clk = clocks.summary()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / args.steps
    xbytes = X.numel() * (1 if w4a8 else 2) + (X.shape[0] * 4 if w4a8 else 0)
    value = job_rate(ws, wb + xbytes + Y.numel() * 2, ms)
    peaks, src = load_peaks()
    achieved = wb / (ms * 1e-3) / 1e9
    # end to end: pinned host rows in (W4A8: the int8 rows and their scales), grouped
    # call, Y to pinned host, synchronised each step
    if w4a8:
        hx = [Xq.cpu().pin_memory(), xs.cpu().pin_memory()]
    else:
        hx = [torch.from_numpy(np.ascontiguousarray(d["A"])).pin_memory()]
    hy = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    dx = [torch.empty_like(h, device=dev) for h in hx]
    n_e2e = max(20, min(500, args.steps // 20))
    with torch.cuda.stream(stream):
        for i in range(3 + n_e2e):
            if i == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            for a, h in zip(dx, hx):
                a.copy_(h, non_blocking=True)
            grouped(i % reps, x=tuple(dx) if w4a8 else dx[0])
            hy.copy_(Y, non_blocking=True)
            stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": name, "tokens_per_expert": [offs[e + 1] - offs[e] for e in range(E)],
                   "l2": f"weights rotate over {reps} copies ({reps * set_bytes / 2**20:.0f} MiB > 3x L2)",
                   "graph": "CUDA graphs of 32 consecutive grouped calls, the weight copy rotating call by call",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "kernel": "wq::gemv_kernel, grouped launch (grid.z = expert); weight bytes of experts with tokens"
                               + ("; int8 rows read directly, per-token scale at the store" if w4a8 else ""),
                     "peak_source": src},
        "gpu_launches": args.steps,
        "clocks": clk,
        "e2e": {"value": round(ws * wb / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in hx),
                "d2h_bytes_per_step": hy.numel() * 2},
    }
    if rank == 0 and not args.no_cpu_baseline:
        gbs, el, threads, sample = moe_oracle(d, args.cpu_seconds, w4a8)
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": sample, "seconds": round(el, 2)}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def swiglu_weight_bytes(d) -> int:
    """Weight bytes of one pair call: codes, scales and delta of the gate and the up weight."""
    K, N = d["gate"]["q"].shape
    G = d["gate"]["scale"].shape[0]
    return 2 * (K * N // 2 + G * N * 6)


def swiglu_oracle(d, budget_s, cols: int = 512):
    """The oracle on a column window of both projections, every token count, until budget_s."""
    import oracle
    gs = synth.SWIGLU["group_size"]
    ws = []
    for w in (d["gate"], d["up"]):
        ws.append((np.ascontiguousarray(w["q"][:, :cols]), oracle.half_bits(w["scale"][:, :cols]),
                   oracle.half_bits(w["zero"][:, :cols])))
    K = d["gate"]["q"].shape[0]
    G = d["gate"]["scale"].shape[0]
    n = 0
    t0 = time.perf_counter()
    while True:
        for A in d["A"]:
            oracle.gemm_swiglu_pair(A.astype(np.float64), ws[0], ws[1], gs)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    wb = n * len(d["A"]) * 2 * (K * cols // 2 + G * cols * 6)
    return wb / el / 1e9, el, threads, f"{n} pass(es) of both token counts on {cols} of {d['gate']['q'].shape[1]} columns, fp64 naive loops"


def run_swiglu(args, ws, rank, local):
    d = synth.swiglu_inputs()
    name = WORKLOAD_NAMES["swiglu"]
    if args.impl == "reference":
        if rank != 0:
            return 0
        gbs, el, threads, sample = swiglu_oracle(d, max(2.0, min(20.0, 4.0 * args.steps)))
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
            "config": {"workload": name, "sampled": True},
            "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return 0
    import torch
    import weight_only_int4_g128_gb300 as wq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wq.load_library(build_if_missing=True)
    if not wq.device_supported(local):
        raise RuntimeError("not an sm_103 device")
    wq.set_weight_prefetch(True)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    gs = synth.SWIGLU["group_size"]
    g, u = d["gate"], d["up"]
    w0 = wq.pack_w4a16_pair(cu(g["q"]), cu(g["scale"]), cu(g["zero"]), cu(u["q"]), cu(u["scale"]), cu(u["zero"]), gs)
    wb = swiglu_weight_bytes(d)
    set_bytes = sum(t.numel() * t.element_size() for t in w0)
    reps = max(1, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
    W = [w0] + [tuple(t.clone() for t in w0) for _ in range(reps - 1)]
    Xs = [cu(A) for A in d["A"]]
    N = g["q"].shape[1]
    Ys = [torch.empty((X.shape[0], N), dtype=torch.float16, device=dev) for X in Xs]
    io_bytes = sum(X.numel() * 2 + Y.numel() * 2 for X, Y in zip(Xs, Ys))

    def step(r):
        for X, Y in zip(Xs, Ys):
            wq.gemm_w4a16_swiglu(X, *W[r], gs, out=Y)

    for r in range(reps):
        step(r)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    graphs, graphs1 = build_step_graphs(torch, stream, reps, step, STEPS_PER_GRAPH)
    with torch.cuda.stream(stream):
        replay_steps(graphs, graphs1, args.warmup, STEPS_PER_GRAPH)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        e0.record(stream)
        replay_steps(graphs, graphs1, args.steps, STEPS_PER_GRAPH)
        e1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks.stop()
    clk = clocks.summary()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / args.steps
    calls = len(Xs)
    value = job_rate(ws, calls * wb + io_bytes, ms)
    peaks, src = load_peaks()
    achieved = calls * wb / (ms * 1e-3) / 1e9
    # end to end: the step's activations copied in from one pinned host buffer, the fused
    # calls on views of the device copy, the outputs copied back in one piece; synchronised
    # each step
    hx = torch.from_numpy(np.concatenate([np.ascontiguousarray(A).reshape(-1) for A in d["A"]])).pin_memory()
    hy = torch.empty(sum(Y.numel() for Y in Ys), dtype=torch.float16).pin_memory()
    dx, dy = torch.empty_like(hx, device=dev), torch.empty_like(hy, device=dev)
    xv, yv, ox, oy = [], [], 0, 0
    for X, Y in zip(Xs, Ys):
        xv.append(dx[ox:ox + X.numel()].view(X.shape))
        yv.append(dy[oy:oy + Y.numel()].view(Y.shape))
        ox += X.numel()
        oy += Y.numel()
    n_e2e = max(20, min(500, args.steps // 20))
    with torch.cuda.stream(stream):
        for i in range(3 + n_e2e):
            if i == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            dx.copy_(hx, non_blocking=True)
            for j in range(calls):
                wq.gemm_w4a16_swiglu(xv[j], *W[i % reps], gs, out=yv[j])
            hy.copy_(dy, non_blocking=True)
            stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": name, "calls_per_step": calls, "us_per_call": round(1e3 * ms / calls, 3),
                   "l2": f"weights rotate over {reps} copies ({reps * set_bytes / 2**20:.0f} MiB > 3x L2)",
                   "graph": f"CUDA graphs of {STEPS_PER_GRAPH} consecutive steps, the weight copy rotating step by step",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "kernel": "wq::gemv_kernel, gate/up pair instance (SwiGLU epilogue); weight bytes of both projections",
                     "peak_source": src},
        "gpu_launches": args.steps * calls,
        "clocks": clk,
        "e2e": {"value": round(ws * calls * wb / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hy.numel() * 2},
    }
    if rank == 0 and not args.no_cpu_baseline:
        gbs, el, threads, sample = swiglu_oracle(d, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": sample, "seconds": round(el, 2)}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def mlp_weight_bytes(d) -> int:
    """Weight bytes of one decode MLP block: codes, scales and delta of gate, up and down."""
    total = 0
    for w in (d["gate"], d["up"], d["down"]):
        K, N = w["q"].shape
        G = w["scale"].shape[0]
        total += K * N // 2 + G * N * 6
    return total


def mlp_oracle(d, budget_s, cols: int = 256):
    """The oracle on column windows: the pair on `cols` of its columns and the down
    projection on `cols` of its outputs (its input a seeded stand-in for the pair's
    output), every token count, until budget_s."""
    import oracle
    gs = synth.MLP["group_size"]
    win = lambda w: (np.ascontiguousarray(w["q"][:, :cols]), oracle.half_bits(w["scale"][:, :cols]),
                     oracle.half_bits(w["zero"][:, :cols]))
    gate, up, down = win(d["gate"]), win(d["up"]), win(d["down"])
    F = d["down"]["q"].shape[0]
    H = [synth.make_activations(synth.MLP["seed"] + 20 + i, A.shape[0], F).astype(np.float64)
         for i, A in enumerate(d["A"])]
    n = 0
    t0 = time.perf_counter()
    while True:
        for A, h in zip(d["A"], H):
            oracle.gemm_swiglu_pair(A.astype(np.float64), gate, up, gs)
            oracle.gemm_asym_plain(h, down[0], down[1], down[2], gs)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    wb = 0
    for w in (d["gate"], d["up"], d["down"]):
        K = w["q"].shape[0]
        wb += K * cols // 2 + w["scale"].shape[0] * cols * 6
    wb *= n * len(d["A"])
    return wb / el / 1e9, el, threads, (f"{n} pass(es) of both token counts on {cols} columns of each projection, "
                                        "fp64 naive loops")


def run_mlp(args, ws, rank, local):
    """The decode MLP block as one chain launch per token count, against the same block as
    two single-GEMM calls (fused SwiGLU pair, then down) timed the same way."""
    d = synth.mlp_inputs()
    name = WORKLOAD_NAMES["mlp"]
    if args.impl == "reference":
        if rank != 0:
            return 0
        gbs, el, threads, sample = mlp_oracle(d, max(2.0, min(20.0, 4.0 * args.steps)))
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
            "config": {"workload": name, "sampled": True},
            "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return 0
    import torch
    import weight_only_int4_g128_gb300 as wq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wq.load_library(build_if_missing=True)
    if not wq.device_supported(local):
        raise RuntimeError("not an sm_103 device")
    wq.set_weight_prefetch(True)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    gs = synth.MLP["group_size"]
    g, u, dn = d["gate"], d["up"], d["down"]
    pair0 = wq.pack_w4a16_pair(cu(g["q"]), cu(g["scale"]), cu(g["zero"]), cu(u["q"]), cu(u["scale"]),
                               cu(u["zero"]), gs)
    down0 = wq.pack_w4a16(cu(dn["q"]), cu(dn["scale"]), cu(dn["zero"]), gs)
    wb = mlp_weight_bytes(d)
    set_bytes = sum(t.numel() * t.element_size() for t in pair0 + down0)
    reps = max(1, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
    W = [(pair0, down0)] + [(tuple(t.clone() for t in pair0), tuple(t.clone() for t in down0))
                            for _ in range(reps - 1)]
    Xs = [cu(A) for A in d["A"]]
    F, N = g["q"].shape[1], dn["q"].shape[1]
    Hs = [torch.empty((X.shape[0], F), dtype=torch.float16, device=dev) for X in Xs]
    Ys = [torch.empty((X.shape[0], N), dtype=torch.float16, device=dev) for X in Xs]
    wsp = torch.zeros(16 << 20, dtype=torch.uint8, device=dev)  # chain workspace, zeroed once
    io_bytes = sum(X.numel() * 2 + Y.numel() * 2 for X, Y in zip(Xs, Ys))

    def chain(X, H, Y, r):
        (Bp, Sp, Dp), (Bd, Sd, Dd) = W[r]
        wq.gemm_w4a16_chain(X, [{"B": Bp, "S": Sp, "delta": Dp, "pair": True, "out": H},
                                {"B": Bd, "S": Sd, "delta": Dd, "src": 0, "out": Y}], workspace=wsp)

    def two_calls(X, H, Y, r):
        (Bp, Sp, Dp), (Bd, Sd, Dd) = W[r]
        wq.gemm_w4a16_swiglu(X, Bp, Sp, Dp, gs, out=H)
        wq.gemm_w4a16(H, Bd, Sd, Dd, gs, out=Y)

    def timed(fn):
        def step(r):
            for X, H, Y in zip(Xs, Hs, Ys):
                fn(X, H, Y, r)
        for r in range(reps):
            step(r)
        torch.cuda.synchronize()
        stream = torch.cuda.Stream(device=dev)
        graphs, graphs1 = build_step_graphs(torch, stream, reps, step, STEPS_PER_GRAPH)
        with torch.cuda.stream(stream):
            replay_steps(graphs, graphs1, args.warmup, STEPS_PER_GRAPH)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda.synchronize()
            e0.record(stream)
            replay_steps(graphs, graphs1, args.steps, STEPS_PER_GRAPH)
            e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), ws, dev) / args.steps, stream

    ms_two, _ = timed(two_calls)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms, stream = timed(chain)
    clocks.stop()
    clk = clocks.summary()
    if ws > 1:
        torch.distributed.barrier()
    calls = len(Xs)
    value = job_rate(ws, calls * wb + io_bytes, ms)
    peaks, src = load_peaks()
    achieved = calls * wb / (ms * 1e-3) / 1e9
    # end to end: the step's activations copied in from one pinned host buffer, the chain
    # calls on views of the device copy, the block outputs copied back; synchronised each step
    hx = torch.from_numpy(np.concatenate([np.ascontiguousarray(A).reshape(-1) for A in d["A"]])).pin_memory()
    hy = torch.empty(sum(Y.numel() for Y in Ys), dtype=torch.float16).pin_memory()
    dx, dy = torch.empty_like(hx, device=dev), torch.empty_like(hy, device=dev)
    xv, yv, ox, oy = [], [], 0, 0
    for X, Y in zip(Xs, Ys):
        xv.append(dx[ox:ox + X.numel()].view(X.shape))
        yv.append(dy[oy:oy + Y.numel()].view(Y.shape))
        ox += X.numel()
        oy += Y.numel()
    n_e2e = max(20, min(500, args.steps // 20))
    with torch.cuda.stream(stream):
        for i in range(3 + n_e2e):
            if i == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            dx.copy_(hx, non_blocking=True)
            for j in range(calls):
                chain(xv[j], Hs[j], yv[j], i % reps)
            hy.copy_(dy, non_blocking=True)
            stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": name, "blocks_per_step": calls, "us_per_block": round(1e3 * ms / calls, 3),
                   "us_per_block_two_calls": round(1e3 * ms_two / calls, 3),
                   "two_calls": "wq_gemm_w4a16_swiglu then wq_gemm_w4a16 (down), timed the same way",
                   "l2": f"weights rotate over {reps} copies ({reps * set_bytes / 2**20:.0f} MiB > 3x L2)",
                   "graph": f"CUDA graphs of {STEPS_PER_GRAPH} consecutive steps, the weight copy rotating step by step",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "frac_two_calls": round(calls * wb / (ms_two * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "kernel": "wq::chain_kernel (persistent, cooperative); weight bytes of gate, up and down",
                     "peak_source": src},
        "gpu_launches": args.steps * calls,
        "clocks": clk,
        "e2e": {"value": round(ws * calls * wb / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hy.numel() * 2},
    }
    if rank == 0 and not args.no_cpu_baseline:
        gbs, el, threads, sample = mlp_oracle(d, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": sample, "seconds": round(el, 2)}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["wq", "reference"], default="wq")
    ap.add_argument("--workload", choices=list(WORKLOAD_NAMES), default="sweep")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--windows", type=int, default=20, help="per-shape timing windows (median reported)")
    ap.add_argument("--window-ms", type=float, default=50.0, help="minimum device time of one window")
    ap.add_argument("--shapes", type=str, default=None,
                    help="comma-separated indices into the workload's shape list (profiling)")
    ap.add_argument("--quick", action="store_true",
                    help="timed steps only: no per-shape timing, e2e or CPU baseline (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_init()
    if args.workload in ("moe", "moe8"):
        return run_moe(args, ws, rank, local)
    if args.workload == "swiglu":
        return run_swiglu(args, ws, rank, local)
    if args.workload == "mlp":
        return run_mlp(args, ws, rank, local)
    shapes = workload_shapes(args.workload)
    if args.shapes:
        shapes = [shapes[int(i)] for i in args.shapes.split(",")]
    if args.quick:
        args.no_cpu_baseline = True
    if args.impl == "reference":
        return run_reference(args, shapes, ws, rank)
    return run_gpu(args, shapes, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
