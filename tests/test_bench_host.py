"""Host-side logic of bench.py's multi-rank path, on CPU: two gloo ranks agree on the
slowest rank's time, the job rate counts every rank's work, and the reference arm runs
and prints on rank 0 only.  No GPU needed."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws, torch.device("cpu"))
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ws = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_job_rate_counts_every_rank():
    one = bench.job_rate(1, 1e9, 2.0)
    assert one == pytest.approx(500.0)
    assert bench.job_rate(4, 1e9, 2.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.5, 1, None) == 3.5


def test_reference_arm_prints_on_rank_0_only():
    class A:
        steps, warmup, workload = 1, 3, "c0"
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(A, synth.shapes("c0"), 2, 1) == 0
    assert buf.getvalue() == ""


@pytest.mark.parametrize("workload", ["moe", "moe8", "swiglu"])
def test_grouped_and_pair_reference_arms_print_one_line(workload):
    """The oracle arms of the grouped (W4A16, W4A8) and SwiGLU pair workloads print one JSON
    line on rank 0 with the contract's keys; other ranks print nothing."""
    import json

    class A:
        steps, warmup, impl = 1, 3, "reference"
    A.workload = workload
    run = bench.run_swiglu if workload == "swiglu" else bench.run_moe
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert run(A, 2, 1, 0) == 0
    assert buf.getvalue() == ""
    with redirect_stdout(buf):
        assert run(A, 1, 0, 0) == 0
    line = json.loads(buf.getvalue().strip())
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["config"]["workload"] == bench.WORKLOAD_NAMES[workload]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_sweep_reference_arm_reports_the_headline_metric():
    """The default workload's oracle arm prints one line on rank 0, in the GPU arm's
    unit (TFLOP/s of the c3 prefill shapes), with the contract's keys."""
    import json

    class A:
        steps, warmup, workload = 1, 3, "sweep"
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(A, bench.workload_shapes("sweep"), 1, 0) == 0
    line = json.loads(buf.getvalue().strip())
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["config"]["shapes"] == ["c3 M4096 K5120 N17408", "c3 M4096 K17408 N5120"]
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"


def test_workload_shapes_and_dispatch_table():
    """The sweep holds every configuration's shapes in order; the kernel table follows
    the library's dispatch rule (M <= 8, 9..16, large M; W4A8 decode and large M)."""
    sh = [s for _, s in bench.workload_shapes("sweep")]
    assert [s["cfg"] for s in sh] == ["c0"] + ["c1"] * 6 + ["c2"] * 6 + ["c3"] * 2 + ["c4"] * 3
    k = {bench.label(s): bench.kernels_for(s) for s in sh}
    assert k["c1 M1 K4096 N4096"] == ["gemv_kernel"]
    assert k["c1 M16 K4096 N11008"] == ["decode16_kernel"]
    # c3 K17408: 640 tiles of 256 tokens leave the last wave of 152 one-CTA slots 32
    # tiles of 136 k-blocks: those go to a second, K-split launch; with K = 5120 (40
    # k-blocks) the split does not pay and the last wave stays partial
    assert k["c3 M4096 K5120 N17408"] == ["corr_prep_kernel", "gemm_kernel"]
    assert k["c3 M4096 K17408 N5120"] == ["corr_prep_kernel", "gemm_kernel", "gemm_kernel"]
    assert k["c4 M16 K5120 N17408"] == ["decode_prep_kernel", "decode_kernel"]
    assert k["c4 M2048 K5120 N17408"] == ["i8_to_f16_kernel", "gemm_kernel"]
    # one partial wave (136 tiles), or a last wave more than half full: one launch
    assert k["c4 M256 K5120 N17408"] == ["i8_to_f16_kernel", "gemm_kernel"]
    assert not bench.large_m_tail(4096, 8192, 8192)  # 1024 tiles: last wave 112 of 152
    assert bench.headline_unit("sweep") == "TFLOP/s" and bench.headline_unit("c1") == "GB/s"
