"""wq_gemm_w4a16_noalloc: the GEMM entry point for callers that cannot allocate.

Some callers cannot give the library a workspace because they cannot allocate
device memory at the point of the call (a framework that allows allocations only
through its own allocator, host code running during stream capture, loops where a
cudaMalloc could synchronize the device).  This entry point takes its scratch from
a fixed 16 MiB array of device memory inside the library.  The test calls it
through the C ABI and checks it, bit for bit, against wq_gemm_w4a16 with a
workspace (the same kernels on the same inputs) and against the oracle, on two
calls in a row with a call of another shape in between, so the shared array holds
unrelated data when the second call starts.  It also checks that a problem too
large for the array is refused without a launch, after the argument checks.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the W4A16 parity bar used throughout the GPU tests


@pytest.fixture(scope="module")
def wq():
    import weight_only_int4_g128_gb300 as m
    m.load_library(build_if_missing=True)
    assert m.device_supported(torch.cuda.current_device())
    return m


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _noalloc(lib, X, Bp, S, dl, Y, M, N, K, gs):
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    xd = 1 if X.dtype == torch.bfloat16 else 0
    yd = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}[Y.dtype]
    return lib.wq_gemm_w4a16_noalloc(p(X), xd, p(Bp), p(S), p(dl), p(Y), yd, M, N, K, gs, stream)


def _problem(wq, seed, M, K, N, adt):
    d = synth.make_inputs(seed, M, K, N, a_dtype=adt)
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), 128)
    X = _cuda(d["A"].view(np.int16)).view(torch.bfloat16) if adt == "bf16" else _cuda(d["A"])
    return d, X, Bp, S, dl


# (300, 1024, 384) and (96, 2048, 256) take the large-M path, whose correction
# columns live in the scratch array; M = 8 takes the weight-streaming kernel,
# which needs no scratch.
@pytest.mark.parametrize("M,K,N,adt", [(300, 1024, 384, "f16"), (96, 2048, 256, "bf16"),
                                       (8, 1024, 256, "f16")])
def test_noalloc_matches_workspace_entry_point(wq, M, K, N, adt):
    lib = wq.load_library()
    d, X, Bp, S, dl = _problem(wq, 1100 + M, M, K, N, adt)
    ws = torch.zeros(max(4096, wq.workspace_size(wq.VARIANT_W4A16, M, N, K, 128)), dtype=torch.uint8,
                     device="cuda")
    ref = wq.gemm_w4a16(X, Bp, S, dl, 128, workspace=ws)
    # another problem of a different shape, run through the same array between the two calls
    M2, K2, N2 = 200, 3072, 512
    _, X2, Bp2, S2, dl2 = _problem(wq, 1190, M2, K2, N2, "f16")
    Y2 = torch.empty((M2, N2), dtype=torch.float16, device="cuda")
    A64 = oracle.activations_to_double(d["A"], adt)
    C = oracle.gemm_asym_plain(A64, d["q"], oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"]), 128)
    torch.cuda.synchronize()
    for i in range(2):
        if i == 1:
            rc = _noalloc(lib, X2, Bp2, S2, dl2, Y2, M2, N2, K2, 128)
            assert rc == 0, lib.wq_last_error()
        Y = torch.full_like(ref, float("nan"))
        rc = _noalloc(lib, X, Bp, S, dl, Y, M, N, K, 128)
        assert rc == 0, lib.wq_last_error()
        torch.cuda.synchronize()
        assert torch.equal(Y, ref), f"call {i}: differs from the workspace entry point"
        err = oracle.rel_fro(Y.double().cpu().numpy(), C)
        assert err <= TOL, (i, err)


def test_noalloc_refuses_problems_beyond_its_scratch(wq):
    lib = wq.load_library()
    M, K, N = 4096, 8192, 65536  # correction columns need (M + N) * 256 * 2 bytes > 16 MiB
    assert lib.wq_workspace_size(wq.VARIANT_W4A16, M, N, K, 128) > 16 << 20
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the call is refused first
    # the arguments are checked before the size: a bad x_dtype is an argument error
    rc = lib.wq_gemm_w4a16_noalloc(fake, 7, fake, fake, fake, fake, 0, M, N, K, 128, None)
    assert rc == 1
    rc = lib.wq_gemm_w4a16_noalloc(fake, 0, fake, fake, fake, fake, 0, M, N, K, 128, None)
    assert rc == 3
    assert b"16777216" in lib.wq_last_error()
