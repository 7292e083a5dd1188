"""CPU oracle for the group-quantized INT4-weight GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never imports, links or calls it, and this package never imports the
product package: the two share no code.  Every stored expected value under
``tests/golden/`` is either a value the pages print (cited there) or written by
``tests/golden/make_golden.py``, which calls only this package.

The arithmetic lives in ``wq_oracle.c`` (plain C, IEEE binary64, naive loops);
this module compiles it with ``gcc`` on first use and marshals numpy arrays to
it.  Sources: "Marlin INT4 on Ada -- how it works" (TinyLoop docs), sections
"The core mismatch: symmetric vs asymmetric", "The pipeline, end to end" and
"Gaps and follow-ups" (the fused SwiGLU pair); the HyperQwen W4A8 article,
sections "hidden mine: the negative group scale bug" and "int8 tensor cores:
how the numbers were verified"; the SGLang W4A8 article, section "task split"
(the grouped mixture-of-experts GEMM).  The grouped and SwiGLU functions are
plain Python loops over the C routines.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, library routines, brute force or printed values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile wq_oracle.c into oracle/_build/liboracle.so with gcc (-O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.wq_o_half_to_double.restype = ctypes.c_double
            lib.wq_o_half_to_double.argtypes = [ctypes.c_uint16]
            lib.wq_o_bf16_to_double.restype = ctypes.c_double
            lib.wq_o_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.wq_o_double_to_half_rn.restype = ctypes.c_uint16
            lib.wq_o_double_to_half_rn.argtypes = [ctypes.c_double]
            lib.wq_o_double_to_bf16_rn.restype = ctypes.c_uint16
            lib.wq_o_double_to_bf16_rn.argtypes = [ctypes.c_double]
            lib.wq_o_double_to_half_array.argtypes = [P, ctypes.c_int64, P]
            lib.wq_o_double_to_bf16_array.argtypes = [P, ctypes.c_int64, P]
            lib.wq_o_pack.argtypes = [P, I, I, P]
            lib.wq_o_unpack.argtypes = [P, I, I, P]
            lib.wq_o_delta.argtypes = [P, P, I, I, P]
            lib.wq_o_fold.argtypes = [P, P, I, I, I, P, P]
            lib.wq_o_dequant_sym_f16.argtypes = [P, P, I, I, I, P]
            lib.wq_o_dequant_sym_bf16.argtypes = [P, P, I, I, I, P]
            lib.wq_o_gemm_asym_plain.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
            lib.wq_o_gemm_asym_identity.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
            lib.wq_o_group_sum.argtypes = [P, I, I, I, P]
            lib.wq_o_gemm_w4a8.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
            lib.wq_o_gemm_w4a8_asym.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P]
            lib.wq_o_quantize_per_token.argtypes = [P, I, I, P, P]
            lib.wq_o_rel_fro.restype = ctypes.c_double
            lib.wq_o_rel_fro.argtypes = [P, P, ctypes.c_int64]
            lib.wq_o_set_mutation.argtypes = [I]
            lib.wq_o_get_mutation.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _gs(K: int, group_size: int) -> int:
    """group_size == K (or -1) means one group per column ("How the dispatcher chooses")."""
    return K if group_size in (-1, K) else group_size


# -- formats ------------------------------------------------------------------

def half_bits(x: np.ndarray) -> np.ndarray:
    """binary16 array -> its uint16 bit patterns (a view, no arithmetic)."""
    return _c(x, np.float16).view(np.uint16)


def half_to_double(bits) -> np.ndarray:
    lib = _load()
    b = _c(bits, np.uint16)
    return np.array([lib.wq_o_half_to_double(int(v)) for v in b.ravel()]).reshape(b.shape)


def bf16_to_double(bits) -> np.ndarray:
    lib = _load()
    b = _c(bits, np.uint16)
    return np.array([lib.wq_o_bf16_to_double(int(v)) for v in b.ravel()]).reshape(b.shape)


def activations_to_double(a: np.ndarray, dtype: str) -> np.ndarray:
    """fp16 array, or bf16 given as uint16 bits, -> float64 (exact)."""
    if dtype == "f16":
        return _c(a, np.float16).astype(np.float64)
    if dtype == "bf16":
        bits = _c(a, np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def double_to_half(x: np.ndarray) -> np.ndarray:
    """float64 -> binary16 bits, round-to-nearest-even (written from IEEE-754)."""
    lib = _load()
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib.wq_o_double_to_half_array(_p(x), x.size, _p(out))
    return out


def double_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bits, round-to-nearest-even (written from IEEE-754)."""
    lib = _load()
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib.wq_o_double_to_bf16_array(_p(x), x.size, _p(out))
    return out


# -- pack / fold / delta -----------------------------------------------------------

def pack(q: np.ndarray) -> np.ndarray:
    """codes q [K, N] (0..15) -> packed words [N/128, K/128, 128, 16] uint32 (the library's
    blocked layout; see wq_oracle.c).  K and N must be multiples of 128."""
    lib = _load()
    q = _c(q, np.uint8)
    K, N = q.shape
    out = np.empty((N // 128, K // 128, 128, 16), np.uint32)
    lib.wq_o_pack(_p(q), K, N, _p(out))
    return out


def unpack(words: np.ndarray, K: int, N: int) -> np.ndarray:
    lib = _load()
    w = _c(words, np.uint32).reshape(-1)
    q = np.empty((K, N), np.uint8)
    lib.wq_o_unpack(_p(w), K, N, _p(q))
    return q


def delta(scale_bits: np.ndarray, zero_bits: np.ndarray) -> np.ndarray:
    """delta = zero + 8*scale, exact in fp64, stored as fp32 [G, N]."""
    lib = _load()
    s = _c(scale_bits, np.uint16)
    z = _c(zero_bits, np.uint16)
    G, N = s.shape
    out = np.empty((G, N), np.float32)
    lib.wq_o_delta(_p(s), _p(z), G, N, _p(out))
    return out


def fold(q: np.ndarray, scale_bits: np.ndarray, group_size: int):
    """Sign fold: for negative group scales, s -> -s and v -> min(16 - v, 15)."""
    lib = _load()
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    K, N = q.shape
    gs = _gs(K, group_size)
    q_out = np.empty_like(q)
    s_out = np.empty_like(s)
    lib.wq_o_fold(_p(q), _p(s), K, N, gs, _p(q_out), _p(s_out))
    return q_out, s_out


def dequant_sym_f16(q, scale_bits, group_size) -> np.ndarray:
    """fp16_RN((q - 8) * scale) as uint16 bits [K, N]."""
    lib = _load()
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    K, N = q.shape
    out = np.empty((K, N), np.uint16)
    lib.wq_o_dequant_sym_f16(_p(q), _p(s), K, N, _gs(K, group_size), _p(out))
    return out


def dequant_sym_bf16(q, scale_bits, group_size) -> np.ndarray:
    """bf16_RN((q - 8) * scale) as uint16 bits [K, N]."""
    lib = _load()
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    K, N = q.shape
    out = np.empty((K, N), np.uint16)
    lib.wq_o_dequant_sym_bf16(_p(q), _p(s), K, N, _gs(K, group_size), _p(out))
    return out


# -- GEMMs --------------------------------------------------------------------------

def _cols(N, cols):
    return (0, N) if cols is None else (int(cols[0]), int(cols[1]))


def gemm_asym_plain(A64, q, scale_bits, zero_bits, group_size, cols=None) -> np.ndarray:
    """C = A @ (q*scale + zero) in fp64 (the plain definition); columns cols=(n0,n1)."""
    lib = _load()
    A = _c(A64, np.float64)
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    z = _c(zero_bits, np.uint16)
    M, K = A.shape
    N = q.shape[1]
    n0, n1 = _cols(N, cols)
    C = np.empty((M, n1 - n0), np.float64)
    lib.wq_o_gemm_asym_plain(_p(A), _p(q), _p(s), _p(z), M, K, N, _gs(K, group_size),
                             n0, n1, _p(C))
    return C


def gemm_asym_identity(A64, q, scale_bits, zero_bits, group_size, cols=None) -> np.ndarray:
    """C = A @ W_sym + A_group_sum @ delta in fp64; zero_bits=None gives A @ W_sym."""
    lib = _load()
    A = _c(A64, np.float64)
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    M, K = A.shape
    N = q.shape[1]
    n0, n1 = _cols(N, cols)
    C = np.empty((M, n1 - n0), np.float64)
    if zero_bits is None:
        zp = None
    else:
        z = _c(zero_bits, np.uint16)
        zp = _p(z)
    lib.wq_o_gemm_asym_identity(_p(A), _p(q), _p(s), zp, M, K, N, _gs(K, group_size),
                                n0, n1, _p(C))
    return C


def group_sum(A64, group_size) -> np.ndarray:
    lib = _load()
    A = _c(A64, np.float64)
    M, K = A.shape
    gs = _gs(K, group_size)
    out = np.empty((M, K // gs), np.float64)
    lib.wq_o_group_sum(_p(A), M, K, gs, _p(out))
    return out


def gemm_w4a8(Xq, x_scale, q, scale_bits, group_size, cols=None) -> np.ndarray:
    """C = x_scale[m] * sum_k Xq[m,k] (q-8) scale, fp64 (folded weights)."""
    lib = _load()
    X = _c(Xq, np.int8)
    xs = _c(x_scale, np.float32)
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    M, K = X.shape
    N = q.shape[1]
    n0, n1 = _cols(N, cols)
    C = np.empty((M, n1 - n0), np.float64)
    lib.wq_o_gemm_w4a8(_p(X), _p(xs), _p(q), _p(s), M, K, N, _gs(K, group_size), n0, n1,
                       _p(C))
    return C


def gemm_w4a8_asym(Xq, x_scale, q, scale_bits, zero_bits, group_size, cols=None) -> np.ndarray:
    """C = x_scale[m] * sum_k Xq[m,k] (q*scale + zero), fp64 (unsigned codes with a
    zero point, no fold; HyperQwen W4A8 article, "int8 tensor cores: how the numbers
    were verified", item 2)."""
    lib = _load()
    X = _c(Xq, np.int8)
    xs = _c(x_scale, np.float32)
    q = _c(q, np.uint8)
    s = _c(scale_bits, np.uint16)
    z = _c(zero_bits, np.uint16)
    M, K = X.shape
    N = q.shape[1]
    n0, n1 = _cols(N, cols)
    C = np.empty((M, n1 - n0), np.float64)
    lib.wq_o_gemm_w4a8_asym(_p(X), _p(xs), _p(q), _p(s), _p(z), M, K, N, _gs(K, group_size), n0, n1,
                            _p(C))
    return C


def gemm_grouped_asym(A64, expert_offsets, q, scale_bits, zero_bits, group_size) -> np.ndarray:
    """Mixture-of-experts GEMM: rows expert_offsets[e] .. expert_offsets[e+1] of A times expert
    e's weight q[e]*scale[e] + zero[e] (zero_bits None: (q - 8)*scale), fp64 (SGLang W4A8
    article, section "task split": one GEMM per group).  q [E, K, N], scale/zero [E, G, N]."""
    A = np.asarray(A64, np.float64)
    E = len(expert_offsets) - 1
    N = q.shape[2]
    C = np.zeros((A.shape[0], N), np.float64)
    wrong = _load().wq_o_get_mutation() == 7  # planted mistake: each segment takes the next expert
    for e in range(E):
        r0, r1 = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if r1 == r0:
            continue
        w = (e + 1) % E if wrong else e
        if zero_bits is None:
            C[r0:r1] = gemm_asym_identity(A[r0:r1], q[w], scale_bits[w], None, group_size)
        else:
            C[r0:r1] = gemm_asym_plain(A[r0:r1], q[w], scale_bits[w], zero_bits[w], group_size)
    return C


def gemm_grouped_w4a8(Xq, x_scale, expert_offsets, q, scale_bits, zero_bits, group_size) -> np.ndarray:
    """Mixture-of-experts W4A8 (SGLang W4A8 article, section "task split": one GEMM per group):
    int8 rows expert_offsets[e] .. expert_offsets[e+1] of Xq, scaled per token, times expert
    e's weight: (q[e] - 8)*scale[e] with non-negative (folded) scales when zero_bits is None,
    else q[e]*scale[e] + zero[e].  q [E, K, N], scale/zero [E, G, N]; fp64."""
    Xq = np.asarray(Xq)
    xs = np.asarray(x_scale, np.float32)
    E = len(expert_offsets) - 1
    N = q.shape[2]
    C = np.zeros((Xq.shape[0], N), np.float64)
    wrong = _load().wq_o_get_mutation() == 7  # planted mistake: each segment takes the next expert
    for e in range(E):
        r0, r1 = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if r1 == r0:
            continue
        w = (e + 1) % E if wrong else e
        if zero_bits is None:
            C[r0:r1] = gemm_w4a8(Xq[r0:r1], xs[r0:r1], q[w], scale_bits[w], group_size)
        else:
            C[r0:r1] = gemm_w4a8_asym(Xq[r0:r1], xs[r0:r1], q[w], scale_bits[w], zero_bits[w], group_size)
    return C


def pair_interleave(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """Column order of the library's gate/up pair weight (its own layout choice): in every
    group of 16 combined columns the first 8 are gate columns 8i .. 8i+7 and the next 8 the
    same up columns.  gate/up [R, N] (N a multiple of 8) -> [R, 2N]."""
    gate, up = np.asarray(gate), np.asarray(up)
    R, N = gate.shape
    out = np.empty((R, 2 * N), gate.dtype)
    for i in range(N // 8):
        out[:, 16 * i:16 * i + 8] = gate[:, 8 * i:8 * i + 8]
        out[:, 16 * i + 8:16 * i + 16] = up[:, 8 * i:8 * i + 8]
    return out


def silu(x) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + e^-x), fp64 (e^-x = inf gives -0)."""
    x = np.asarray(x, np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def gemm_swiglu_pair(A64, gate, up, group_size) -> np.ndarray:
    """Fused SwiGLU pair ("Marlin INT4 on Ada", section "Gaps and follow-ups": mlp_gate and
    mlp_up in one kernel): silu(A @ W_gate) * (A @ W_up), each product the plain W4A16 GEMM
    (gate / up = (q, scale_bits, zero_bits); zero_bits None: (q - 8) * scale), fp64."""
    def product(w):
        q, sb, zb = w
        if zb is None:
            return gemm_asym_identity(A64, q, sb, None, group_size)
        return gemm_asym_plain(A64, q, sb, zb, group_size)
    G, U = product(gate), product(up)
    if _load().wq_o_get_mutation() == 8:  # planted mistake: the activation on the up projection
        G, U = U, G
    return silu(G) * U


def quantize_per_token(x_f16: np.ndarray):
    """Per-token absmax int8 quantization: returns (Xq int8 [M,K], x_scale fp32 [M])."""
    lib = _load()
    xb = half_bits(x_f16)
    M, K = xb.shape
    Xq = np.empty((M, K), np.int8)
    xs = np.empty((M,), np.float32)
    lib.wq_o_quantize_per_token(_p(xb), M, K, _p(Xq), _p(xs))
    return Xq, xs


def rel_fro(X, R) -> float:
    """||X - R||_F / ||R||_F in fp64."""
    lib = _load()
    X = _c(X, np.float64)
    R = _c(R, np.float64)
    assert X.shape == R.shape
    return float(lib.wq_o_rel_fro(_p(X), _p(R), X.size))


class mutation:
    """Context manager planting one known mistake in the oracle (pin sensitivity tests).

    1: delta = zero - 8*scale   2: fold clamps 16 to 0   3: W_sym uses q-7
    4: identity form drops the correction term   5: W4A8 ignores x_scale
    """

    def __init__(self, mid: int):
        self.mid = mid

    def __enter__(self):
        _load().wq_o_set_mutation(self.mid)
        return self

    def __exit__(self, *exc):
        _load().wq_o_set_mutation(0)
        return False
