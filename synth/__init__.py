"""Seeded synthetic inputs for the INT4-weight GEMM workloads.

This module only draws random numbers and casts them to their storage dtypes;
it holds none of the quantized-GEMM arithmetic.  Both the CUDA path (tests,
bench) and the CPU oracle take their inputs from here.

Recipe (numpy PCG64; one generator per shape, seed = 1000*config + index;
draw order A, q, |scale|, zero factor, sign):
  A      ~ N(0, a_std) cast to fp16 (bf16 for the prefill workload)
  q      uniform integers in [0, 15], shape [K, N]
  scale  U(0.005, 0.02) cast to fp16, shape [G, N]
  zero   fp16(-scale * U(6, 10))                (asymmetric workloads)
  sign   Bernoulli(0.5) per (g, n) negates the scale  (W4A8 workload)
The workload list mirrors the shapes these pages discuss: the K=256 MoE test
shape of the SGLang W4A8 write-up, 4096-wide decode projections, 8192-square
batched GEMMs, and the 5120 x 17408 / 17408 x 5120 Qwen projections of the
HyperQwen article.  No dataset or checkpoint is involved.
"""
from __future__ import annotations

import numpy as np

GROUP = 128


def _bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (a storage cast, via torch's CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


# name -> (config index, list of shapes).  A shape is a dict with M, K, N,
# group_size, a_dtype, a_std, mode.
WORKLOADS = {
    "c0": (0, [dict(M=16, K=256, N=256)]),
    "c1": (1, [dict(M=m, K=4096, N=n) for n in (4096, 11008) for m in (1, 4, 16)]),
    "c2": (2, [dict(M=m, K=8192, N=8192, group_size=gs) for gs in (128, -1)
               for m in (64, 128, 256)]),
    "c3": (3, [dict(M=4096, K=5120, N=17408), dict(M=4096, K=17408, N=5120)]),
    "c4": (4, [dict(M=m, K=5120, N=17408) for m in (16, 256, 2048)]),
}

_DEFAULTS = {
    0: dict(group_size=GROUP, a_dtype="f16", a_std=1.0, mode="w4a16"),
    1: dict(group_size=GROUP, a_dtype="f16", a_std=1.0, mode="w4a16"),
    2: dict(group_size=GROUP, a_dtype="f16", a_std=0.5, mode="w4a16"),
    3: dict(group_size=GROUP, a_dtype="bf16", a_std=1.0, mode="w4a16"),
    4: dict(group_size=GROUP, a_dtype="f16", a_std=1.0, mode="w4a8"),
}


def shapes(workload: str):
    """List of (seed, shape dict) for a named workload."""
    cfg, lst = WORKLOADS[workload]
    out = []
    for i, s in enumerate(lst):
        d = dict(_DEFAULTS[cfg])
        d.update(s)
        out.append((1000 * cfg + i, d))
    return out


def num_groups(K: int, group_size: int) -> int:
    return 1 if group_size in (-1, K) else K // group_size


def make_inputs(seed: int, M: int, K: int, N: int, group_size: int = GROUP,
                a_dtype: str = "f16", a_std: float = 1.0, mode: str = "w4a16",
                weights_only: bool = False) -> dict:
    """Draw one problem.

    Returns a dict of numpy arrays:
      A        [M, K] float16, or uint16 bf16 bit patterns when a_dtype == "bf16"
               (for mode == "w4a8" this is the fp16 activation before quantization)
      q        [K, N] uint8 codes 0..15
      scale    [G, N] float16 (signed for w4a8)
      zero     [G, N] float16 (w4a16 only)
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    G = num_groups(K, group_size)
    out = {"M": M, "K": K, "N": N, "group_size": group_size, "a_dtype": a_dtype,
           "mode": mode}
    a = rng.standard_normal((M, K), dtype=np.float32) * np.float32(a_std)
    if not weights_only:
        out["A"] = _bf16_bits(a) if a_dtype == "bf16" else a.astype(np.float16)
    out["q"] = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, size=(G, N)).astype(np.float16)
    zf = rng.uniform(6.0, 10.0, size=(G, N))
    if mode == "w4a16":
        out["scale"] = s
        out["zero"] = (-(s.astype(np.float64)) * zf).astype(np.float16)
    else:
        neg = rng.random((G, N)) < 0.5
        out["scale"] = np.where(neg, -s, s).astype(np.float16)
    return out


def make_activations(seed: int, M: int, K: int, a_dtype: str = "f16", a_std: float = 1.0):
    """Activations only (same recipe as make_inputs' A, separate stream)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, K), dtype=np.float32) * np.float32(a_std)
    return _bf16_bits(a) if a_dtype == "bf16" else a.astype(np.float16)


# Mixture-of-experts workload: 16 tokens routed (top-1) over 8 experts, each expert
# a K=256 x N=7168 asymmetric g128 weight (the grouped W4A8 test shape of the SGLang
# MoE article, batch 16, k 256, n 7168, 8 experts), fp16 activations.
MOE = dict(experts=8, tokens=16, K=256, N=7168, group_size=GROUP, seed=5000)


def moe_inputs(seed: int = MOE["seed"], experts: int = MOE["experts"], tokens: int = MOE["tokens"],
               K: int = MOE["K"], N: int = MOE["N"], group_size: int = MOE["group_size"]):
    """Routing counts (uniform top-1 choice per token, tokens sorted by expert), the
    activations [tokens, K] fp16, and per-expert weights (make_inputs recipe)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    choice = rng.integers(0, experts, size=tokens)
    counts = np.bincount(choice, minlength=experts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    A = make_activations(seed + 1, tokens, K)
    ws = [make_inputs(seed + 2 + e, 1, K, N, group_size=group_size, weights_only=True) for e in range(experts)]
    return {"offsets": offsets, "A": A, "q": np.stack([w["q"] for w in ws]),
            "scale": np.stack([w["scale"] for w in ws]), "zero": np.stack([w["zero"] for w in ws])}


SWIGLU = dict(tokens=(1, 4), K=4096, N=11008, group_size=GROUP, seed=5100)


def swiglu_inputs(seed: int = SWIGLU["seed"], tokens=SWIGLU["tokens"], K: int = SWIGLU["K"],
                  N: int = SWIGLU["N"], group_size: int = SWIGLU["group_size"]):
    """Decode-time gated MLP input projections: activations [m, K] fp16 for each token count
    and one gate and one up weight [K, N] (make_inputs recipe, asymmetric, group 128)."""
    A = [make_activations(seed + 1 + i, m, K) for i, m in enumerate(tokens)]
    gate = make_inputs(seed + 10, 1, K, N, group_size=group_size, weights_only=True)
    up = make_inputs(seed + 11, 1, K, N, group_size=group_size, weights_only=True)
    return {"A": A, "gate": gate, "up": up}



# Decode MLP block of the c1 model dimensions (hidden 4096, intermediate 11008): the
# gate/up pair on the token rows, then the down projection of its SwiGLU output.
MLP = dict(tokens=(1, 4), K=4096, F=11008, N=4096, group_size=GROUP, seed=5200)


def mlp_inputs(seed: int = MLP["seed"], tokens=MLP["tokens"], K: int = MLP["K"], F: int = MLP["F"],
               N: int = MLP["N"], group_size: int = MLP["group_size"]):
    """Activations [m, K] fp16 for each token count, gate and up weights [K, F] and the down
    weight [F, N] (make_inputs recipe, asymmetric, group 128)."""
    A = [make_activations(seed + 1 + i, m, K) for i, m in enumerate(tokens)]
    gate = make_inputs(seed + 10, 1, K, F, group_size=group_size, weights_only=True)
    up = make_inputs(seed + 11, 1, K, F, group_size=group_size, weights_only=True)
    down = make_inputs(seed + 12, 1, F, N, group_size=group_size, weights_only=True)
    return {"A": A, "gate": gate, "up": up, "down": down}
