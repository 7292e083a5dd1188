"""Python binding of libwq.so, the GB300 (sm_103a) group-quantized INT4-weight GEMM.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/wq.h.  PyTorch supplies device
memory and the current stream.  There is no CPU or PyTorch fallback: if the
library is not built, or the device is not sm_103, calls raise.

    Bpacked, S, delta = pack_w4a16(q, scale, zero, group_size)
    Y = gemm_w4a16(X, Bpacked, S, delta, group_size)       # X fp16 or bf16 [M, K]
    Bpacked, S_abs = pack_w4a8(q, scale_signed, group_size)
    Xq, x_scale = quantize_per_token(x)
    Y = gemm_w4a8(Xq, x_scale, Bpacked, S_abs, group_size)
    Y = gemm_w4a8_asym(Xq, x_scale, *pack_w4a16(q, scale, zero, group_size), group_size)
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "WQError", "load_library", "library_path", "pack_w4a16", "pack_w4a8", "unpack_w4",
    "dequant_w4", "quantize_per_token", "gemm_w4a16", "gemm_w4a16_host", "gemm_w4a8", "gemm_w4a8_asym",
    "gemm_w4a8_fp16", "gemm_w4a16_grouped", "gemm_w4a8_grouped", "pack_w4a16_pair", "gemm_w4a16_swiglu", "workspace_size",
    "device_supported", "device_status", "debug_wait_probe", "version", "Workspace",
    "EXPORTS", "DTYPE_F16", "DTYPE_BF16", "DTYPE_F32",
    "VARIANT_W4A16", "VARIANT_W4A16_SYM", "VARIANT_W4A8", "VARIANT_W4A8_ASYM", "VARIANT_W4A16_SWIGLU",
    "VARIANT_W4A16_SWIGLU_SYM", "set_weight_prefetch",
    "OPTION_WEIGHT_PREFETCH", "gemm_w4a16_chain", "chain_workspace", "ChainGemm",
]

DTYPE_F16, DTYPE_BF16, DTYPE_F32 = 0, 1, 2
VARIANT_W4A16, VARIANT_W4A16_SYM, VARIANT_W4A8, VARIANT_W4A8_ASYM = 0, 1, 2, 3
VARIANT_W4A16_SWIGLU, VARIANT_W4A16_SWIGLU_SYM = 4, 5
ERRORS = {1: "WQ_ERR_INVALID_ARG", 2: "WQ_ERR_UNSUPPORTED_SHAPE", 3: "WQ_ERR_WORKSPACE",
          4: "WQ_ERR_ARCH", 5: "WQ_ERR_CUDA", 6: "WQ_ERR_TIMEOUT"}

_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


class ChainGemm(ctypes.Structure):
    """wq_chain_gemm of include/wq.h: one GEMM of a persistent decode chain."""
    _fields_ = [("X", _P), ("src", _I), ("Bpacked", _P), ("S", _P), ("delta", _P), ("Y", _P),
                ("y_dtype", _I), ("N", _I), ("K", _I), ("group_size", _I), ("pair", _I)]


# name -> (restype, argtypes); one entry per function declared in include/wq.h
EXPORTS = {
    "wq_pack_w4a16": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "wq_pack_w4a8": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "wq_unpack_w4": (_I, [_P, _P, _I, _I, _P]),
    "wq_dequant_w4": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "wq_gemm_w4a16": (_I, [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_gemm_w4a8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_gemm_w4a8_asym": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_gemm_w4a8_fp16": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_gemm_w4a16_grouped": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_gemm_w4a8_grouped": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_pack_w4a16_pair": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "wq_gemm_w4a16_swiglu": (_I, [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_quantize_per_token": (_I, [_P, _P, _P, _I, _I, _P]),
    "wq_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "wq_device_supported": (_I, [_I]),
    "wq_last_error": (ctypes.c_char_p, []),
    "wq_version": (ctypes.c_char_p, []),
    "wq_device_status": (_I, [ctypes.POINTER(ctypes.c_uint), _I, _P]),
    "wq_debug_wait_probe": (_I, [ctypes.c_ulonglong, _P]),
    "wq_set_option": (_I, [_I, ctypes.c_longlong]),
    "wq_gemm_w4a16_noalloc": (_I, [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "wq_get_option": (_I, [_I, ctypes.POINTER(ctypes.c_longlong)]),
    "wq_gemm_w4a16_host": (_I, [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "wq_host_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "wq_chain_workspace_size": (_SZ, [ctypes.POINTER(ChainGemm), _I, _I, _I]),
    "wq_gemm_w4a16_chain": (_I, [ctypes.POINTER(ChainGemm), _I, _I, _I, _P, _SZ, _P]),
}
OPTION_WEIGHT_PREFETCH = 1

_lib = None
_lock = threading.Lock()


class WQError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libwq.so.  Raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and _build.is_stale():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    "libwq.so is not built: run `python -m weight_only_int4_g128_gb300.build` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(_build.LIB)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _torch():
    import torch
    return torch


def _check(rc: int, where: str):
    if rc != 0:
        raise WQError(rc, where, load_library().wq_last_error().decode())


def _raw_stream(device_index: int) -> int:
    """Handle of the current CUDA stream of a device, as an integer.  torch's own
    accessor for it is used when present (a cheap call), else the public API."""
    torch = _torch()
    get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if get is not None:
        return get(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _stream(t=None):
    torch = _torch()
    return ctypes.c_void_p(_raw_stream(t.device.index if t is not None else torch.cuda.current_device()))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


_DTYPE_CODES = {}


def _dtype_code(dt) -> int:
    if not _DTYPE_CODES:
        torch = _torch()
        _DTYPE_CODES.update({torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32})
    return _DTYPE_CODES[dt]


def _gs(K: int, group_size: int) -> int:
    return K if group_size in (-1, K) else group_size


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# -- packing -------------------------------------------------------------------------

def pack_w4a16(q, scale, zero, group_size: int = 128):
    """q [K,N] uint8 codes, scale/zero [G,N] fp16 -> (Bpacked, S, delta fp32).

    Bpacked is int32 [N/128, K/128, 128, 16] holding the library's blocked layout."""
    torch = _torch()
    _require_cuda(q, scale, zero)
    K, N = q.shape
    G = K // _gs(K, group_size)
    Bp = torch.empty((N // 128, K // 128, 128, 16), dtype=torch.int32, device=q.device)
    S = torch.empty((G, N), dtype=torch.float16, device=q.device)
    d = torch.empty((G, N), dtype=torch.float32, device=q.device)
    _check(load_library().wq_pack_w4a16(_ptr(q), _ptr(scale), _ptr(zero), _ptr(Bp), _ptr(S),
                                        _ptr(d), K, N, group_size, _stream()), "wq_pack_w4a16")
    return Bp, S, d


def pack_w4a16_pair(q_gate, scale_gate, zero_gate, q_up, scale_up, zero_up, group_size: int = 128):
    """Gate/up projection pair ([K,N] codes, [G,N] fp16 scales and zeros each) -> the
    (Bpacked, S, delta) of one [K,2N] weight with the columns interleaved in groups of 16
    (8 gate columns, then the same 8 up columns), for gemm_w4a16_swiglu."""
    torch = _torch()
    _require_cuda(q_gate, scale_gate, zero_gate, q_up, scale_up, zero_up)
    K, N = q_gate.shape
    if tuple(q_up.shape) != (K, N):
        raise ValueError("gate and up codes must have the same shape")
    G = K // _gs(K, group_size)
    Bp = torch.empty((2 * N // 128, K // 128, 128, 16), dtype=torch.int32, device=q_gate.device)
    S = torch.empty((G, 2 * N), dtype=torch.float16, device=q_gate.device)
    d = torch.empty((G, 2 * N), dtype=torch.float32, device=q_gate.device)
    _check(load_library().wq_pack_w4a16_pair(_ptr(q_gate), _ptr(scale_gate), _ptr(zero_gate), _ptr(q_up),
                                             _ptr(scale_up), _ptr(zero_up), _ptr(Bp), _ptr(S), _ptr(d), K, N,
                                             group_size, _stream()), "wq_pack_w4a16_pair")
    return Bp, S, d


def pack_w4a8(q, scale_signed, group_size: int = 128):
    """q [K,N] uint4b8 codes, signed scale [G,N] fp16 -> (Bpacked, S_abs) with the sign fold."""
    torch = _torch()
    _require_cuda(q, scale_signed)
    K, N = q.shape
    G = K // _gs(K, group_size)
    Bp = torch.empty((N // 128, K // 128, 128, 16), dtype=torch.int32, device=q.device)
    S = torch.empty((G, N), dtype=torch.float16, device=q.device)
    _check(load_library().wq_pack_w4a8(_ptr(q), _ptr(scale_signed), _ptr(Bp), _ptr(S), K, N,
                                       group_size, _stream()), "wq_pack_w4a8")
    return Bp, S


def unpack_w4(Bpacked, K: int, N: int):
    torch = _torch()
    _require_cuda(Bpacked)
    q = torch.empty((K, N), dtype=torch.uint8, device=Bpacked.device)
    _check(load_library().wq_unpack_w4(_ptr(Bpacked), _ptr(q), K, N, _stream()), "wq_unpack_w4")
    return q


def dequant_w4(Bpacked, S, K: int, N: int, group_size: int = 128, dtype=None):
    torch = _torch()
    dtype = dtype or torch.float16
    _require_cuda(Bpacked, S)
    W = torch.empty((K, N), dtype=dtype, device=Bpacked.device)
    _check(load_library().wq_dequant_w4(_ptr(Bpacked), _ptr(S), _ptr(W), _dtype_code(dtype), K, N,
                                        group_size, _stream()), "wq_dequant_w4")
    return W


def quantize_per_token(x):
    torch = _torch()
    _require_cuda(x)
    M, K = x.shape
    Xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(load_library().wq_quantize_per_token(_ptr(x), _ptr(Xq), _ptr(xs), M, K, _stream()),
           "wq_quantize_per_token")
    return Xq, xs


# -- workspace -------------------------------------------------------------------------

def workspace_size(variant: int, M: int, N: int, K: int, group_size: int) -> int:
    return int(load_library().wq_workspace_size(variant, M, N, K, group_size))


class Workspace:
    """Zero-initialised device scratch for one stream, grown on demand (torch-allocated)."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        torch = _torch()
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=self.device)
        return self.buf


_ws = {}


def _stream_workspace(device, stream: int) -> Workspace:
    key = (device.index, stream)
    ws = _ws.get(key)
    if ws is None:
        ws = _ws[key] = Workspace(device)
    return ws


def _workspace(device, nbytes):
    return _stream_workspace(device, _raw_stream(device.index)).get(nbytes)


def _call_gemm(fn, where, args_head, args_tail, workspace, variant, M, N, K, group_size, device, stream):
    """Run a GEMM entry point.  Without a caller workspace the stream's cached
    scratch is passed as it is; only if the library reports it too small is its
    size queried, the scratch grown and the call repeated (the library checks the
    workspace before it launches anything)."""
    lib = _lib or load_library()
    if workspace is not None:
        ws = workspace
    else:
        ws = _stream_workspace(device, stream).buf
    rc = fn(*args_head, ws.data_ptr() if ws is not None else None, ws.numel() if ws is not None else 0,
            stream, *args_tail)
    if rc == 3 and workspace is None:  # WQ_ERR_WORKSPACE: grow the stream's scratch and retry
        ws = _stream_workspace(device, stream).get(workspace_size(variant, M, N, K, group_size))
        rc = fn(*args_head, ws.data_ptr(), ws.numel(), stream, *args_tail)
    if rc != 0:
        raise WQError(rc, where, lib.wq_last_error().decode())


# -- GEMMs -----------------------------------------------------------------------------

def gemm_w4a16(X, Bpacked, S, delta, group_size: int = 128, out_dtype=None, out=None,
               workspace=None):
    """Y = X @ W_sym + A_group_sum @ delta  (delta None: symmetric).  X [M,K] fp16/bf16."""
    torch = _torch()
    _require_cuda(X, Bpacked, S, delta, out)
    M, K = X.shape
    N = Bpacked.numel() * 8 // K
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=X.device)
    variant = VARIANT_W4A16 if delta is not None else VARIANT_W4A16_SYM
    lib = _lib or load_library()
    _call_gemm(lib.wq_gemm_w4a16, "wq_gemm_w4a16",
               (X.data_ptr(), _dtype_code(X.dtype), Bpacked.data_ptr(), S.data_ptr(),
                delta.data_ptr() if delta is not None else None, Y.data_ptr(), _dtype_code(Y.dtype),
                M, N, K, group_size), (), workspace, variant, M, N, K, group_size, X.device,
               _raw_stream(X.device.index))
    return Y


def gemm_w4a16_swiglu(X, Bpacked, S, delta, group_size: int = 128, out_dtype=None, out=None,
                      workspace=None):
    """Y = silu(X @ W_gate) * (X @ W_up) on a pack_w4a16_pair weight (delta None: symmetric).
    X [M,K] fp16/bf16; Y [M,N] with N half the pair weight's columns."""
    torch = _torch()
    _require_cuda(X, Bpacked, S, delta, out)
    M, K = X.shape
    N = Bpacked.numel() * 8 // K // 2
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=X.device)
    variant = VARIANT_W4A16_SWIGLU if delta is not None else VARIANT_W4A16_SWIGLU_SYM
    lib = _lib or load_library()
    _call_gemm(lib.wq_gemm_w4a16_swiglu, "wq_gemm_w4a16_swiglu",
               (X.data_ptr(), _dtype_code(X.dtype), Bpacked.data_ptr(), S.data_ptr(),
                delta.data_ptr() if delta is not None else None, Y.data_ptr(), _dtype_code(Y.dtype),
                M, N, K, group_size), (), workspace, variant, M, N, K, group_size, X.device,
               _raw_stream(X.device.index))
    return Y


_chain_ws = {}


def chain_workspace(device=None, nbytes: int = 0):
    """The zero-initialised chain workspace of a device's current stream, grown (as a new
    zeroed buffer) when a chain needs more.  Chain calls keep its control words consistent,
    so it is never cleared between calls."""
    torch = _torch()
    device = torch.device(device if device is not None else "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    key = (device.index, _raw_stream(device.index))
    buf = _chain_ws.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = _chain_ws[key] = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=device)
    return buf


def gemm_w4a16_chain(X, steps, workspace=None):
    """One persistent launch over a list of decode GEMMs (X [M,K] fp16/bf16, M <= 8).

    steps[i] is a dict: "B", "S", "delta" (None: symmetric) from pack_w4a16, or from
    pack_w4a16_pair with "pair": True (output silu(gate) * up); optional "group_size" (128),
    "src" (index of an earlier step whose output is this step's input; default: X, or "x"
    for another input tensor), "out_dtype" (fp16) or "out".  A step read by a later one must
    have the activation dtype.  Returns the list of outputs."""
    torch = _torch()
    M = X.shape[0]
    n = len(steps)
    arr = (ChainGemm * max(n, 1))()
    outs = []
    for i, st in enumerate(steps):
        B, S, dl = st["B"], st["S"], st.get("delta")
        src = st.get("src")
        x = None if src is not None else st.get("x", X)
        K = outs[src].shape[1] if src is not None else x.shape[1]
        pair = bool(st.get("pair", False))
        N = B.numel() * 8 // K // (2 if pair else 1)
        _require_cuda(x, B, S, dl, st.get("out"))
        Y = st.get("out")
        if Y is None:
            Y = torch.empty((M, N), dtype=st.get("out_dtype", torch.float16), device=X.device)
        outs.append(Y)
        arr[i] = ChainGemm(x.data_ptr() if x is not None else None, -1 if src is None else src, B.data_ptr(),
                           S.data_ptr(), dl.data_ptr() if dl is not None else None, Y.data_ptr(),
                           _dtype_code(Y.dtype), N, K, st.get("group_size", 128), 1 if pair else 0)
    lib = _lib or load_library()
    xd = _dtype_code(X.dtype)
    if workspace is None:
        need = int(lib.wq_chain_workspace_size(arr, n, M, xd))
        workspace = chain_workspace(X.device, need)
    _check(lib.wq_gemm_w4a16_chain(arr, n, M, xd, workspace.data_ptr(), workspace.numel(),
                                   _raw_stream(X.device.index)), "wq_gemm_w4a16_chain")
    return outs


def gemm_w4a16_host(X, Bpacked, S, delta, group_size: int = 128, out_dtype=None, out=None,
                    workspace=None):
    """gemm_w4a16 between host tensors: X [M,K] fp16/bf16 on the host (pinned for
    asynchronous copies) is copied to the weights' device, multiplied, and Y comes
    back into a host tensor (`out`, or a new pinned one).  The copies and the GEMM
    are enqueued on the device's current stream; Y is valid after that stream is
    synchronized."""
    torch = _torch()
    if X.is_cuda or not X.is_contiguous() or (out is not None and (out.is_cuda or not out.is_contiguous())):
        raise ValueError("X and out must be contiguous host tensors")
    _require_cuda(Bpacked, S, delta)
    M, K = X.shape
    N = Bpacked.numel() * 8 // K
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, pin_memory=True)
    variant = VARIANT_W4A16 if delta is not None else VARIANT_W4A16_SYM
    lib = _lib or load_library()
    device = Bpacked.device
    stream = _raw_stream(device.index)
    ydt = _dtype_code(Y.dtype)
    ws = workspace if workspace is not None else _stream_workspace(device, stream).buf
    head = (X.data_ptr(), _dtype_code(X.dtype), Bpacked.data_ptr(), S.data_ptr(),
            delta.data_ptr() if delta is not None else None, Y.data_ptr(), ydt, M, N, K, group_size)
    rc = lib.wq_gemm_w4a16_host(*head, ws.data_ptr() if ws is not None else None,
                                ws.numel() if ws is not None else 0, stream)
    if rc == 3 and workspace is None:  # WQ_ERR_WORKSPACE: grow the stream's scratch and retry
        need = int(lib.wq_host_workspace_size(variant, M, N, K, group_size, ydt))
        ws = _stream_workspace(device, stream).get(need)
        rc = lib.wq_gemm_w4a16_host(*head, ws.data_ptr(), ws.numel(), stream)
    if rc != 0:
        raise WQError(rc, "wq_gemm_w4a16_host", lib.wq_last_error().decode())
    return Y


def gemm_w4a8(Xq, x_scale, Bpacked, S_abs, group_size: int = 128, out_dtype=None, out=None,
              workspace=None):
    """Y = x_scale[m] * Xq @ W_sym  (folded weights).  Xq [M,K] int8."""
    torch = _torch()
    _require_cuda(Xq, x_scale, Bpacked, S_abs, out)
    M, K = Xq.shape
    N = Bpacked.numel() * 8 // K
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=Xq.device)
    lib = _lib or load_library()
    _call_gemm(lib.wq_gemm_w4a8, "wq_gemm_w4a8",
               (Xq.data_ptr(), x_scale.data_ptr(), Bpacked.data_ptr(), S_abs.data_ptr(), Y.data_ptr(),
                _dtype_code(Y.dtype), M, N, K, group_size), (), workspace, VARIANT_W4A8, M, N, K,
               group_size, Xq.device, _raw_stream(Xq.device.index))
    return Y


def gemm_w4a8_asym(Xq, x_scale, Bpacked, S, delta, group_size: int = 128, out_dtype=None, out=None,
                   workspace=None):
    """Y = x_scale[m] * (Xq @ W_sym + A_group_sum(Xq) @ delta): zero-point uint4 weights
    packed by pack_w4a16 (delta None: symmetric with the scales as given).  Xq [M,K] int8."""
    torch = _torch()
    _require_cuda(Xq, x_scale, Bpacked, S, delta, out)
    M, K = Xq.shape
    N = Bpacked.numel() * 8 // K
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=Xq.device)
    lib = _lib or load_library()
    _call_gemm(lib.wq_gemm_w4a8_asym, "wq_gemm_w4a8_asym",
               (Xq.data_ptr(), x_scale.data_ptr(), Bpacked.data_ptr(), S.data_ptr(),
                delta.data_ptr() if delta is not None else None, Y.data_ptr(), _dtype_code(Y.dtype), M, N, K,
                group_size), (), workspace, VARIANT_W4A8_ASYM if delta is not None else VARIANT_W4A8, M, N, K,
               group_size, Xq.device, _raw_stream(Xq.device.index))
    return Y


def gemm_w4a8_fp16(X, Bpacked, S, delta=None, group_size: int = 128, out_dtype=None, out=None,
                   x_scale=None, workspace=None):
    """W4A8 on fp16 activations X [M,K], quantized per token inside the call.  Returns
    (Y, x_scale); Y equals gemm_w4a8_asym (delta given) / gemm_w4a8 (delta None) on the
    codes of quantize_per_token(X), bit for bit."""
    torch = _torch()
    _require_cuda(X, Bpacked, S, delta, out, x_scale)
    M, K = X.shape
    N = Bpacked.numel() * 8 // K
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=X.device)
    xs = x_scale if x_scale is not None else torch.empty((M,), dtype=torch.float32, device=X.device)
    lib = _lib or load_library()
    _call_gemm(lib.wq_gemm_w4a8_fp16, "wq_gemm_w4a8_fp16",
               (X.data_ptr(), Bpacked.data_ptr(), S.data_ptr(), delta.data_ptr() if delta is not None else None,
                xs.data_ptr(), Y.data_ptr(), _dtype_code(Y.dtype), M, N, K, group_size), (), workspace,
               VARIANT_W4A8_ASYM if delta is not None else VARIANT_W4A8, M, N, K, group_size, X.device,
               _raw_stream(X.device.index))
    return Y, xs


def gemm_w4a16_grouped(X, Bpacked, S, delta, expert_offsets, group_size: int = 128, out_dtype=None,
                       out=None, workspace=None):
    """Mixture-of-experts W4A16: rows expert_offsets[e] .. expert_offsets[e+1] of X (sorted by
    expert) times expert e's weights.  Bpacked [E, ...], S / delta [E, G, N] are the stacked
    pack_w4a16 outputs; expert_offsets is a host sequence of E + 1 ints."""
    torch = _torch()
    _require_cuda(X, Bpacked, S, delta, out)
    M, K = X.shape
    E = int(S.shape[0])
    N = int(S.shape[-1])
    offs = (ctypes.c_int * (E + 1))(*[int(v) for v in expert_offsets])
    if len(expert_offsets) != E + 1 or offs[E] != M:
        raise ValueError("expert_offsets must have experts + 1 entries ending at X.shape[0]")
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=X.device)
    lib = _lib or load_library()
    stream = _raw_stream(X.device.index)
    if workspace is None:
        variant = VARIANT_W4A16 if delta is not None else VARIANT_W4A16_SYM
        counts = {offs[e + 1] - offs[e] for e in range(E)} - {0}
        need = max(workspace_size(variant, m, N, K, group_size) for m in counts) if counts else 0
        workspace = _stream_workspace(X.device, stream).get(need) if need > 0 else None
    rc = lib.wq_gemm_w4a16_grouped(X.data_ptr(), _dtype_code(X.dtype), Bpacked.data_ptr(), S.data_ptr(),
                                   delta.data_ptr() if delta is not None else None, Y.data_ptr(),
                                   _dtype_code(Y.dtype), offs, E, N, K, group_size,
                                   workspace.data_ptr() if workspace is not None else None,
                                   workspace.numel() if workspace is not None else 0, stream)
    if rc != 0:
        raise WQError(rc, "wq_gemm_w4a16_grouped", lib.wq_last_error().decode())
    return Y


def gemm_w4a8_grouped(Xq, x_scale, Bpacked, S, delta, expert_offsets, group_size: int = 128, out_dtype=None,
                      out=None, workspace=None):
    """Mixture-of-experts W4A8: int8 rows expert_offsets[e] .. expert_offsets[e+1] of Xq (sorted
    by expert, per-token scales x_scale) times expert e's weights: stacked pack_w4a8 outputs
    (delta None) or stacked pack_w4a16 outputs (zero-point weights, delta [E, G, N])."""
    torch = _torch()
    _require_cuda(Xq, x_scale, Bpacked, S, delta, out)
    M, K = Xq.shape
    E = int(S.shape[0])
    N = int(S.shape[-1])
    offs = (ctypes.c_int * (E + 1))(*[int(v) for v in expert_offsets])
    if len(expert_offsets) != E + 1 or offs[E] != M:
        raise ValueError("expert_offsets must have experts + 1 entries ending at Xq.shape[0]")
    Y = out if out is not None else torch.empty((M, N), dtype=out_dtype or torch.float16, device=Xq.device)
    lib = _lib or load_library()
    stream = _raw_stream(Xq.device.index)
    if workspace is None:
        variant = VARIANT_W4A8_ASYM if delta is not None else VARIANT_W4A8
        counts = {offs[e + 1] - offs[e] for e in range(E)} - {0}
        need = max(workspace_size(variant, m, N, K, group_size) for m in counts) if counts else 0
        workspace = _stream_workspace(Xq.device, stream).get(need) if need > 0 else None
    rc = lib.wq_gemm_w4a8_grouped(Xq.data_ptr(), x_scale.data_ptr(), Bpacked.data_ptr(), S.data_ptr(),
                                  delta.data_ptr() if delta is not None else None, Y.data_ptr(),
                                  _dtype_code(Y.dtype), offs, E, N, K, group_size,
                                  workspace.data_ptr() if workspace is not None else None,
                                  workspace.numel() if workspace is not None else 0, stream)
    if rc != 0:
        raise WQError(rc, "wq_gemm_w4a8_grouped", lib.wq_last_error().decode())
    return Y


# -- device queries ------------------------------------------------------------------------

def device_supported(device: int = 0) -> bool:
    return bool(load_library().wq_device_supported(device))


def device_status(reset: bool = True) -> int:
    st = ctypes.c_uint(0)
    load_library().wq_device_status(ctypes.byref(st), 1 if reset else 0, _stream())
    return int(st.value)


def debug_wait_probe(limit_ns: int):
    _check(load_library().wq_debug_wait_probe(limit_ns, _stream()), "wq_debug_wait_probe")


def set_weight_prefetch(enabled: bool):
    """Let the decode kernel start copying weights before the preceding kernel in the
    stream finishes (only valid when that kernel does not write the weights)."""
    _check(load_library().wq_set_option(OPTION_WEIGHT_PREFETCH, 1 if enabled else 0),
           "wq_set_option")


def version() -> str:
    return load_library().wq_version().decode()
