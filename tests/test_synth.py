"""The seeded input recipe (synth/__init__.py) that every parity test and the bench
draw from: deterministic per seed, the stated shapes and value ranges.  No GPU."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import synth  # noqa: E402


def test_same_seed_same_problem_other_seed_other_problem():
    a, b = synth.make_inputs(7, 4, 256, 128), synth.make_inputs(7, 4, 256, 128)
    c = synth.make_inputs(8, 4, 256, 128)
    for k in ("A", "q", "scale", "zero"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["q"], c["q"])


def test_value_ranges_follow_the_recipe():
    d = synth.make_inputs(11, 8, 1024, 256)
    assert d["q"].dtype == np.uint8 and d["q"].min() == 0 and d["q"].max() == 15
    s = d["scale"].astype(np.float64)
    assert d["scale"].dtype == np.float16 and s.min() >= 0.005 * (1 - 2 ** -10) and s.max() <= 0.02 * (1 + 2 ** -10)
    ratio = d["zero"].astype(np.float64) / s  # zero = -scale * U(6, 10), rounded to fp16
    assert ratio.min() >= -10.02 and ratio.max() <= -5.98
    w8 = synth.make_inputs(12, 8, 1024, 256, mode="w4a8")
    assert "zero" not in w8
    neg = (w8["scale"].astype(np.float64) < 0).mean()
    assert 0.45 < neg < 0.55  # about half the group scales negative (folded at pack)


def test_workload_shapes():
    c1 = synth.shapes("c1")
    assert [(s["M"], s["K"], s["N"]) for _, s in c1] == [(m, 4096, n) for n in (4096, 11008) for m in (1, 4, 16)]
    assert all(s["a_dtype"] == "bf16" for _, s in synth.shapes("c3"))
    assert all(s["mode"] == "w4a8" for _, s in synth.shapes("c4"))
    assert len({seed for w in ("c0", "c1", "c2", "c3", "c4") for seed, _ in synth.shapes(w)}) == 1 + 6 + 6 + 2 + 3


def test_moe_and_swiglu_inputs():
    d = synth.moe_inputs()
    E, K, N = d["q"].shape
    assert (E, K, N) == (8, 256, 7168)
    off = d["offsets"]
    assert off[0] == 0 and off[-1] == 16 and np.all(np.diff(off) >= 0) and len(off) == E + 1
    assert d["A"].shape == (16, 256) and d["scale"].shape == (8, 2, 7168)
    sw = synth.swiglu_inputs()
    assert [a.shape for a in sw["A"]] == [(1, 4096), (4, 4096)]
    assert sw["gate"]["q"].shape == sw["up"]["q"].shape == (4096, 11008)
    assert not np.array_equal(sw["gate"]["q"], sw["up"]["q"])
