#!/usr/bin/env python
"""Benchmark of the W4A16 group-quantized INT4-weight GEMM on GB300.

Default workload: the decode GEMV shapes, M in {1, 4, 16} x N in {4096, 11008},
K = 4096, group 128, asymmetric weights, fp16 activations and output.  One
"step" runs all six GEMMs (each on its own resident copy of the packed
weights); the weight copies rotate over >3x the L2 size so every GEMM reads its
weights from HBM.  The metric is weight GB/s (codes + fp16 scales + fp32 delta
per second) for the whole job; TFLOPS is reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl wq|reference]
                    [--workload c1|c0|c2|c3|c4|moe|moe8|swiglu]

--impl reference times the CPU oracle (plain C, fp64, naive loops) on a bounded
sample of the same workload.  Under torchrun each rank runs an independent
replica on its own GPU (the GEMM has no exchange step); rank 0 prints one JSON
line.
"""
from __future__ import annotations

import argparse
import json
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
WORKLOAD_NAMES = {
    "c0": "W4A16 asym M16 K256 N256 g128 fp16",
    "c1": "W4A16 asym decode GEMV M{1,4,16} x N{4096,11008} K4096 g128 fp16",
    "c2": "W4A16 asym batched M{64,128,256} K8192 N8192 g128 and per-channel fp16",
    "c3": "W4A16 asym prefill M4096 K5120 N17408 + M4096 K17408 N5120 g128 bf16",
    "c4": "W4A8 sym M{16,256,2048} K5120 N17408 g128 int8 per-token",
    "moe": "W4A16 asym grouped (mixture of experts): 16 tokens top-1 over 8 experts, K256 N7168 g128 fp16",
    "moe8": "W4A8 zero-point grouped (mixture of experts): 16 int8 per-token rows top-1 over 8 experts, K256 N7168 g128",
    "swiglu": "W4A16 asym fused SwiGLU gate/up pair, decode M{1,4} K4096 N11008 (x2 projections) g128 fp16",
}


# ----------------------------------------------------------------------------- helpers
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


def kernel_launches(s) -> int:
    """Kernels one GEMM call enqueues (the decode kernel is a single launch for W4A16;
    the large-M path adds one correction pre-pass (group sums and delta columns), W4A8
    an activation pre-pass)."""
    if s["mode"] == "w4a8":
        return 2
    return 1 if s["M"] <= 16 else 2


def flops(s) -> int:
    return 2 * s["M"] * s["N"] * s["K"]


def load_traffic(shapes):
    """DRAM bytes of one launch of the decode kernel from the committed ncu capture
    (profiles/traffic.json), or None when the kernel's sources changed since the
    capture or the captured shape is not part of this workload."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec["source_sha256"]:
        return None
    sh = rec["shape"]
    if not any(s["M"] == sh["M"] and s["K"] == sh["K"] and s["N"] == sh["N"] and s["group_size"] == sh["group_size"]
               and s["mode"] == "w4a16" for _, s in shapes):
        return None
    return rec


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
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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


# ----------------------------------------------------------------------------- oracle arm
def oracle_sample(shapes, budget_s: float, cols: int = 2048):
    """Time the CPU oracle on column windows of every shape until budget_s has passed."""
    import oracle
    probs = []
    for seed, s in shapes:
        d = synth.make_inputs(seed, **s)
        w = min(cols, s["N"])
        G = synth.num_groups(s["K"], s["group_size"])
        wb = s["K"] * w // 2 + G * w * 2 + (G * w * 4 if s["mode"] == "w4a16" else 0)
        probs.append((s, d, w, wb))
    done_bytes = 0
    done_flops = 0
    passes = 0
    t0 = time.perf_counter()
    while True:
        for s, d, w, wb in probs:
            if s["mode"] == "w4a8":
                Xq, xs = oracle.quantize_per_token(d["A"])
                qf, sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), s["group_size"])
                oracle.gemm_w4a8(Xq, xs, qf, sf, s["group_size"], cols=(0, w))
            else:
                A = oracle.activations_to_double(d["A"], s["a_dtype"])
                oracle.gemm_asym_plain(A, d["q"], oracle.half_bits(d["scale"]),
                                       oracle.half_bits(d["zero"]), s["group_size"], cols=(0, w))
            done_bytes += wb
            done_flops += 2 * s["M"] * s["K"] * w
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"{passes} pass(es) over the {len(probs)} shapes, columns [0, {cols}) of each, "
              f"all rows and the full K, fp64 naive loops")
    return done_bytes / el / 1e9, done_flops / el / 1e12, el, threads, sample


def run_reference(args, shapes, ws, rank):
    if rank != 0:
        return 0
    budget = max(2.0, min(20.0, 4.0 * args.steps))
    steps = []
    for _ in range(args.warmup and 1):
        oracle_sample(shapes, 0.5, cols=256)
    gbs, tfl, el, threads, sample = oracle_sample(shapes, budget)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
        "tflops": round(tfl, 9), "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": WORKLOAD_NAMES[args.workload], "sampled": True},
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    del steps
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
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
    # the decode kernel may start copying them before the preceding GEMM finishes.
    wq.set_weight_prefetch(True)

    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # --- problems: inputs resident in HBM, weights replicated to rotate past L2
    probs = []
    set_bytes = 0
    for seed, s in shapes:
        d = synth.make_inputs(seed, **s)
        gs = s["group_size"]
        if s["mode"] == "w4a8":
            Bp, S = wq.pack_w4a8(cu(d["q"]), cu(d["scale"]), gs)
            dl = None
            X16 = cu(d["A"])
            Xq, xs = wq.quantize_per_token(X16)
            X = (Xq, xs)
        else:
            Bp, S, dl = wq.pack_w4a16(cu(d["q"]), cu(d["scale"]), cu(d["zero"]), gs)
            if s["a_dtype"] == "bf16":
                X = cu(d["A"].view(np.int16)).view(torch.bfloat16)
            else:
                X = cu(d["A"])
        probs.append({"s": s, "w": [(Bp, S, dl)], "X": X, "A_host": d["A"]})
        set_bytes += weight_bytes(s)
        del d
    reps = max(1, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
    for p in probs:
        Bp, S, dl = p["w"][0]
        for _ in range(reps - 1):
            p["w"].append((Bp.clone(), S.clone(), dl.clone() if dl is not None else None))
    for p in probs:
        s = p["s"]
        p["Y"] = torch.empty((s["M"], s["N"]), dtype=torch.float16, device=dev)
        variant = wq.VARIANT_W4A8 if s["mode"] == "w4a8" else wq.VARIANT_W4A16
        need = wq.workspace_size(variant, s["M"], s["N"], s["K"], s["group_size"])
        p["ws"] = torch.zeros(max(need, 4096), dtype=torch.uint8, device=dev)

    def call(p, r, out=None, X=None):
        s = p["s"]
        Bp, S, dl = p["w"][r]
        X = p["X"] if X is None else X
        if s["mode"] == "w4a8":
            return wq.gemm_w4a8(X[0], X[1], Bp, S, s["group_size"], out=p["Y"] if out is None else out,
                                workspace=p["ws"])
        return wq.gemm_w4a16(X, Bp, S, dl, s["group_size"], out=p["Y"] if out is None else out,
                             workspace=p["ws"])

    # eager warm-up (sets kernel attributes, checks the calls work)
    for p in probs:
        for r in range(reps):
            call(p, r)
    torch.cuda.synchronize()

    # --- one CUDA graph per weight replica: a whole step (all shapes)
    stream = torch.cuda.Stream(device=dev)
    def step(r):
        for p in probs:
            call(p, r)

    spg = STEPS_PER_GRAPH
    graphs, graphs1 = build_step_graphs(torch, stream, reps, step, spg)
    torch.cuda.synchronize()

    launches_per_step = sum(kernel_launches(p["s"]) for p in probs)

    with torch.cuda.stream(stream):
        replay_steps(graphs, graphs1, args.warmup, spg)
    torch.cuda.synchronize()

    # --- timed region
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        replay_steps(graphs, graphs1, args.steps, spg)
        ev1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    ms_per_step = ms / args.steps
    step_wbytes = sum(weight_bytes(p["s"]) for p in probs)
    step_flops = sum(flops(p["s"]) for p in probs)
    value = job_rate(ws, step_wbytes, ms_per_step)
    tflops = job_rate(ws, step_flops, ms_per_step, 1e12)

    peaks, peaks_src = load_peaks()
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(value, 2), "unit": "GB/s",
                              "tflops": round(tflops, 3), "ms_per_step": round(ms_per_step, 6),
                              "quick": True, "clocks": clk}), flush=True)
        return 0

    # --- per-shape launch timing of the GEMM call (graphs of `per` calls on rotating weights)
    per = 2 * reps
    shape_rows = []
    tot_alg = 0
    tot_ms = 0.0
    for p in probs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for j in range(per):
                    call(p, j % reps)
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            nrep = 20
            for _ in range(nrep):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (nrep * per)
        s = p["s"]
        alg = weight_bytes(s) + io_bytes(s)
        tot_alg += alg
        tot_ms += us * 1e-3
        shape_rows.append({"M": s["M"], "N": s["N"], "K": s["K"], "us": round(us, 3),
                           "weight_GBps": round(weight_bytes(s) / (us * 1e-6) / 1e9, 1),
                           "tflops": round(flops(s) / (us * 1e-6) / 1e12, 3)})

    traffic = load_traffic(shapes)
    tot_flops = sum(flops(p["s"]) for p in probs)
    # Which roofline bounds the workload: its bytes at the measured HBM copy rate
    # against its FLOPs at the measured dense bf16/fp16 rate (fp16 runs at the bf16
    # rate on this part; W4A8 is computed in fp16 or e4m3, never at an int8 rate).
    # The per-shape loops run for seconds, so the sustained tensor figure applies.
    t_hbm = tot_alg / (peaks["hbm_gbs"] * 1e9)
    t_tc = tot_flops / (peaks["bf16_tflops_sustained"] * 1e12)
    if t_hbm >= t_tc:
        achieved = tot_alg / (tot_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peaks_src} (MEASURED_PEAKS.json hbm_gbs, copy)"
                    if peaks_src == "measured" else "fallback 6.8 TB/s"}
    else:
        achieved = tot_flops / (tot_ms * 1e-3) / 1e12
        pk = peaks["bf16_tflops_sustained"]
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk, "unit": "TFLOP/s",
                    "frac": round(achieved / pk, 4),
                    "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                    "peak_source": f"{peaks_src} (MEASURED_PEAKS.json bf16_tflops_sustained, cuBLAS bf16)"
                    if peaks_src == "measured" else "fallback 1.7 PFLOP/s sustained"}
    roofline.update({
        "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
        "kernel": "wq::gemv_kernel (W4A16, M <= 8) / wq::decode16_kernel (M 9..16) / wq::gemm_kernel; time per GEMM call",
        "traffic_launch": ({"shape": traffic["shape"], "algorithmic_bytes": traffic["algorithmic_bytes_per_launch"],
                            "source": traffic["capture"]} if traffic else None),
        "per_shape": shape_rows})

    # --- end to end through the public API.  The step's activations (every shape) sit in
    # one pinned host buffer that one cudaMemcpyAsync copies in; each GEMM call reads its
    # view of the device copy (W4A8 shapes: the fp16 rows, quantized per token inside the
    # call by gemm_w4a8_fp16) and writes its view of one device output buffer, which one
    # copy brings back to pinned host memory; synchronised every step.
    e2e_steps = max(20, min(200, args.steps // 50))
    sizes_x = [p["s"]["M"] * p["s"]["K"] for p in probs]
    sizes_y = [p["s"]["M"] * p["s"]["N"] for p in probs]
    hx_all = torch.empty(sum(sizes_x), dtype=torch.int16).pin_memory()
    hy_all = torch.empty(sum(sizes_y), dtype=torch.float16).pin_memory()
    dx_all = torch.empty_like(hx_all, device=dev)
    dy_all = torch.empty_like(hy_all, device=dev)
    xv, yv = [], []
    ox = oy = 0
    for p, nx, ny in zip(probs, sizes_x, sizes_y):
        s = p["s"]
        hx_all[ox:ox + nx].copy_(torch.from_numpy(np.ascontiguousarray(p["A_host"]).view(np.int16).reshape(-1)))
        x = dx_all[ox:ox + nx].view(s["M"], s["K"])
        xv.append(x.view(torch.bfloat16) if s["a_dtype"] == "bf16" else x.view(torch.float16))
        yv.append(dy_all[oy:oy + ny].view(s["M"], s["N"]))
        p["xs"] = torch.empty((s["M"],), dtype=torch.float32, device=dev)
        ox += nx
        oy += ny
    h2d = hx_all.numel() * hx_all.element_size()
    d2h = hy_all.numel() * hy_all.element_size()

    def e2e_call(j, p, r):
        s = p["s"]
        Bp, S, dl = p["w"][r]
        if s["mode"] == "w4a8":
            wq.gemm_w4a8_fp16(xv[j], Bp, S, None, s["group_size"], out=yv[j], x_scale=p["xs"], workspace=p["ws"])
        else:
            wq.gemm_w4a16(xv[j], Bp, S, dl, s["group_size"], out=yv[j], workspace=p["ws"])

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(3 + e2e_steps):
            if i == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            dx_all.copy_(hx_all, non_blocking=True)
            for j, p in enumerate(probs):
                e2e_call(j, p, i % reps)
            hy_all.copy_(dy_all, non_blocking=True)
            stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_val = ws * step_wbytes / e2e_s / 1e9

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "tflops": round(tflops, 3),
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded PCG64, recipe in synth/__init__.py)",
        "config": {"workload": WORKLOAD_NAMES[args.workload],
                   "shapes": [f"M{p['s']['M']} K{p['s']['K']} N{p['s']['N']}" for p in probs],
                   "l2": f"weights rotate over {reps} copies ({reps * set_bytes / 2**20:.0f} MiB "
                         f"> 3x L2); activations resident",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "graph": f"CUDA graphs of {STEPS_PER_GRAPH} consecutive steps, the weight copy rotating step by step",
                   "launch": "programmatic dependent launch, weight prefetch enabled"},
        "roofline": roofline,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "every step: the step's activations copied from one pinned host buffer, the "
                        "GEMM calls of the public API on the device copy (gemm_w4a16; W4A8: "
                        "gemm_w4a8_fp16 quantizing inside), the outputs copied back to pinned host "
                        "memory, synchronised"},
    }
    if rank == 0 and not args.no_cpu_baseline:
        gbs, tfl, el, threads, sample = oracle_sample(shapes, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": sample, "seconds": round(el, 2)}
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
    clk = clocks.stop()
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
    clk = clocks.stop()
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["wq", "reference"], default="wq")
    ap.add_argument("--workload", choices=list(WORKLOAD_NAMES), default="c1")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shapes", type=str, default=None,
                    help="comma-separated indices into the workload's shape list (profiling)")
    ap.add_argument("--quick", action="store_true",
                    help="timed region only: no per-shape timing, e2e or CPU baseline (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_init()
    if args.workload in ("moe", "moe8"):
        return run_moe(args, ws, rank, local)
    if args.workload == "swiglu":
        return run_swiglu(args, ws, rank, local)
    shapes = synth.shapes(args.workload)
    if args.shapes:
        shapes = [shapes[int(i)] for i in args.shapes.split(",")]
    if args.quick:
        args.no_cpu_baseline = True
    if args.impl == "reference":
        return run_reference(args, shapes, ws, rank)
    return run_gpu(args, shapes, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
