"""The C-ABI library builds, loads and exports every symbol include/wq.h declares;
host-side argument checks return their error codes before any device work.
No GPU needed: nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

import weight_only_int4_g128_gb300 as wq
from weight_only_int4_g128_gb300 import build as wq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")


@pytest.fixture(scope="module")
def lib():
    wq_build.build()
    return wq.load_library()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s*(wq_\w+)\s*\(", text,
                                 re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("wq_pack_w4a16", "wq_pack_w4a8", "wq_unpack_w4", "wq_gemm_w4a16",
                 "wq_gemm_w4a8", "wq_workspace_size", "wq_device_supported", "wq_last_error",
                 "wq_version"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert names
    for name in names:
        assert hasattr(lib, name), name
        assert name in wq.EXPORTS, name
    assert set(wq.EXPORTS) == set(names)


def test_library_links_no_driver_library():
    out = os.popen(f"ldd {wq_build.LIB}").read()
    assert "libcuda.so" not in out


def test_version_and_workspace_queries(lib):
    assert b"sm_103a" in lib.wq_version()
    # decode (M <= 16): W4A16 reads the activations directly and reduces split-K in
    # shared memory (no scratch); W4A8 needs the e4m3 activation components plus one
    # row of per-block sums and factors, padded to [56][K] bytes
    a = lib.wq_workspace_size(wq.VARIANT_W4A16, 16, 4096, 4096, 128)
    b = lib.wq_workspace_size(wq.VARIANT_W4A16_SYM, 1, 4096, 4096, 128)
    c = lib.wq_workspace_size(wq.VARIANT_W4A8, 16, 4096, 4096, 128)
    assert a == b == 0 and c == 56 * 4096
    # large M: the asymmetric variant needs the correction columns, [M + N][kaug] bf16;
    # both variants need room for bf16 activations' scaled fp16 copy [M][K] and its
    # per-token factors [M] fp32 (the query takes no activation type, so it returns
    # the most any type needs)
    a = lib.wq_workspace_size(wq.VARIANT_W4A16, 512, 4096, 4096, 128)
    b = lib.wq_workspace_size(wq.VARIANT_W4A16_SYM, 512, 4096, 4096, 128)
    assert b == 512 * 4096 * 2 + 512 * 4
    assert a == (512 + 4096) * 128 * 2 + b
    assert lib.wq_workspace_size(wq.VARIANT_W4A16, 16, 4096, 4000, 128) == 0  # K % 128
    assert lib.wq_workspace_size(wq.VARIANT_W4A16, 16, 4096, 4096, 64) == 0   # group size
    assert lib.wq_workspace_size(9, 16, 4096, 4096, 128) == 0


def test_shape_and_argument_errors_before_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    # K not a multiple of 128
    rc = lib.wq_gemm_w4a16(fake, 0, fake, fake, fake, fake, 0, 16, 256, 200, 128, fake, 1 << 20, None)
    assert rc == 2 and b"multiples of 128" in lib.wq_last_error()
    # N not a multiple of 128 (the vocab-size projection case, V = 50257)
    rc = lib.wq_gemm_w4a16(fake, 0, fake, fake, fake, fake, 0, 16, 50257, 256, 128, fake, 1 << 20, None)
    assert rc == 2
    # group size other than 128 or K
    rc = lib.wq_gemm_w4a16(fake, 0, fake, fake, fake, fake, 0, 16, 256, 256, 64, fake, 1 << 20, None)
    assert rc == 2
    # bad dtypes
    assert lib.wq_gemm_w4a16(fake, 7, fake, fake, fake, fake, 0, 16, 256, 256, 128, fake, 1, None) == 1
    assert lib.wq_gemm_w4a16(fake, 0, fake, fake, fake, fake, 9, 16, 256, 256, 128, fake, 1, None) == 1
    # null / misaligned pointers
    assert lib.wq_gemm_w4a16(None, 0, fake, fake, fake, fake, 0, 16, 256, 256, 128, fake, 1, None) == 1
    odd = P(0x10008)
    assert lib.wq_gemm_w4a16(odd, 0, fake, fake, fake, fake, 0, 16, 256, 256, 128, fake, 1, None) == 1
    assert lib.wq_gemm_w4a8(None, fake, fake, fake, fake, 0, 16, 256, 256, 128, fake, 1, None) == 1
    # empty problem is a no-op that succeeds
    assert lib.wq_gemm_w4a16(None, 0, None, None, None, None, 0, 0, 256, 256, 128, None, 0, None) == 0
    assert lib.wq_gemm_w4a8(None, None, None, None, None, 0, 0, 256, 256, 128, None, 0, None) == 0
    assert lib.wq_quantize_per_token(None, None, None, 0, 64, None) == 0
    # negative M
    assert lib.wq_gemm_w4a16(fake, 0, fake, fake, fake, fake, 0, -1, 256, 256, 128, fake, 1, None) == 2
    # pack shape checks
    assert lib.wq_pack_w4a16(fake, fake, fake, fake, fake, fake, 100, 256, 128, None) == 2
    assert lib.wq_pack_w4a8(fake, fake, fake, fake, 256, 256, 32, None) == 2
    assert lib.wq_pack_w4a16(None, fake, fake, fake, fake, fake, 256, 256, 128, None) == 1
    assert lib.wq_dequant_w4(fake, fake, fake, 2, 256, 256, 128, None) == 1
    assert lib.wq_debug_wait_probe(0, None) == 1
    assert lib.wq_set_option(99, 1) == 1
    assert lib.wq_set_option(wq.OPTION_WEIGHT_PREFETCH, 2) == 1
    v = ctypes.c_longlong(-1)
    assert lib.wq_get_option(wq.OPTION_WEIGHT_PREFETCH, ctypes.byref(v)) == 0 and v.value == 0
    assert lib.wq_set_option(wq.OPTION_WEIGHT_PREFETCH, 1) == 0
    assert lib.wq_get_option(wq.OPTION_WEIGHT_PREFETCH, ctypes.byref(v)) == 0 and v.value == 1
    assert lib.wq_set_option(wq.OPTION_WEIGHT_PREFETCH, 0) == 0


def test_host_buffer_entry_checks_and_workspace(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    # staging for X [M,K] fp16 and Y [M,N] (256-byte aligned each) ahead of the GEMM's scratch
    for M, N, K, y in ((16, 4096, 4096, 0), (1, 11008, 4096, 1), (512, 4096, 4096, 0), (3, 256, 384, 1)):
        gemm = lib.wq_workspace_size(wq.VARIANT_W4A16, M, N, K, 128)
        al = lambda b: (b + 255) // 256 * 256
        assert lib.wq_host_workspace_size(wq.VARIANT_W4A16, M, N, K, 128, y) == al(M * K * 2) + al(M * N * 2) + gemm
    f32 = lib.wq_host_workspace_size(wq.VARIANT_W4A16, 16, 4096, 4096, 128, 2)
    assert f32 == 16 * 4096 * 2 + 16 * 4096 * 4
    assert lib.wq_host_workspace_size(wq.VARIANT_W4A8, 16, 4096, 4096, 128, 0) == 0  # not a host-entry variant
    assert lib.wq_host_workspace_size(wq.VARIANT_W4A16, 16, 4096, 4000, 128, 0) == 0
    assert lib.wq_host_workspace_size(wq.VARIANT_W4A16, 16, 4096, 4096, 128, 9) == 0
    need = lib.wq_host_workspace_size(wq.VARIANT_W4A16, 16, 256, 256, 128, 0)
    ws = P(0x100000)  # 256-byte aligned, never dereferenced
    h = lib.wq_gemm_w4a16_host
    assert h(fake, 0, fake, fake, fake, fake, 0, 16, 256, 200, 128, ws, need, None) == 2      # K % 128
    assert h(fake, 0, fake, fake, fake, fake, 0, 16, 256, 256, 64, ws, need, None) == 2       # group size
    assert h(fake, 0, fake, fake, fake, fake, 0, -1, 256, 256, 128, ws, need, None) == 2      # M < 0
    assert h(fake, 7, fake, fake, fake, fake, 0, 16, 256, 256, 128, ws, need, None) == 1      # x dtype
    assert h(fake, 0, fake, fake, fake, fake, 9, 16, 256, 256, 128, ws, need, None) == 1      # y dtype
    assert h(None, 0, fake, fake, fake, fake, 0, 16, 256, 256, 128, ws, need, None) == 1      # null X
    assert h(fake, 0, fake, fake, fake, None, 0, 16, 256, 256, 128, ws, need, None) == 1      # null Y
    assert h(fake, 0, P(0x10008), fake, fake, fake, 0, 16, 256, 256, 128, ws, need, None) == 1  # misaligned
    rc = h(fake, 0, fake, fake, fake, fake, 0, 16, 256, 256, 128, ws, need - 1, None)
    assert rc == 3 and b"needed" in lib.wq_last_error()                                          # too small
    assert h(fake, 0, fake, fake, fake, fake, 0, 16, 256, 256, 128, None, need, None) == 3
    assert h(fake, 0, fake, fake, fake, fake, 0, 16, 256, 256, 128, P(0x100010), need, None) == 1  # alignment
    # host X and Y may sit at any address: only the device pointers are checked for alignment
    assert h(None, 0, None, None, None, None, 0, 0, 256, 256, 128, None, 0, None) == 0        # empty


def test_w4a8_zero_point_entry_checks_and_workspace(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    # decode: the same activation-component scratch as W4A8; large M: W4A8's fp16 copy of the
    # int8 rows plus the W4A16 correction columns
    assert lib.wq_workspace_size(wq.VARIANT_W4A8_ASYM, 16, 4096, 4096, 128) == \
        lib.wq_workspace_size(wq.VARIANT_W4A8, 16, 4096, 4096, 128)
    big = lib.wq_workspace_size(wq.VARIANT_W4A8_ASYM, 512, 4096, 4096, 128)
    assert big >= lib.wq_workspace_size(wq.VARIANT_W4A8, 512, 4096, 4096, 128) + (512 + 4096) * 128 * 2
    assert lib.wq_workspace_size(6, 16, 4096, 4096, 128) == 0  # unknown variant
    f = lib.wq_gemm_w4a8_asym
    assert f(fake, fake, fake, fake, fake, fake, 0, 16, 256, 200, 128, fake, 1 << 20, None) == 2  # K % 128
    assert f(fake, fake, fake, fake, fake, fake, 0, 16, 256, 256, 64, fake, 1 << 20, None) == 2   # group
    assert f(fake, fake, fake, fake, fake, fake, 9, 16, 256, 256, 128, fake, 1 << 20, None) == 1  # y dtype
    assert f(None, fake, fake, fake, fake, fake, 0, 16, 256, 256, 128, fake, 1 << 20, None) == 1  # null Xq
    assert f(fake, None, fake, fake, fake, fake, 0, 16, 256, 256, 128, fake, 1 << 20, None) == 1  # x_scale
    assert f(fake, fake, fake, fake, P(0x10008), fake, 0, 16, 256, 256, 128, fake, 1 << 20, None) == 1
    assert f(None, None, None, None, None, None, 0, 0, 256, 256, 128, None, 0, None) == 0        # empty


def test_w4a8_quantize_inside_entry_checks(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    f = lib.wq_gemm_w4a8_fp16
    assert f(fake, fake, fake, None, fake, fake, 0, 16, 256, 200, 128, fake, 1 << 20, None) == 2   # K % 128
    assert f(fake, fake, fake, None, fake, fake, 5, 16, 256, 256, 128, fake, 1 << 20, None) == 1   # y dtype
    assert f(None, fake, fake, None, fake, fake, 0, 16, 256, 256, 128, fake, 1 << 20, None) == 1   # null X
    assert f(fake, fake, fake, None, None, fake, 0, 16, 256, 256, 128, fake, 1 << 20, None) == 1   # x_scale
    assert f(fake, fake, fake, None, P(0x10002), fake, 0, 16, 256, 256, 128, fake, 1 << 20, None) == 1
    assert f(None, None, None, None, None, None, 0, 0, 256, 256, 128, None, 0, None) == 0         # empty


def test_grouped_entry_checks(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    f = lib.wq_gemm_w4a16_grouped
    offs = (ctypes.c_int * 4)(0, 2, 2, 5)
    assert f(fake, 0, fake, fake, fake, fake, 0, offs, 3, 256, 200, 128, None, 0, None) == 2      # K % 128
    assert f(fake, 0, fake, fake, fake, fake, 0, offs, 0, 256, 256, 128, None, 0, None) == 1      # experts
    assert f(fake, 0, fake, fake, fake, fake, 0, offs, 65, 256, 256, 128, None, 0, None) == 1
    assert f(fake, 0, fake, fake, fake, fake, 0, None, 3, 256, 256, 128, None, 0, None) == 1      # offsets
    bad = (ctypes.c_int * 4)(0, 3, 2, 5)
    assert f(fake, 0, fake, fake, fake, fake, 0, bad, 3, 256, 256, 128, None, 0, None) == 1       # decreasing
    nz = (ctypes.c_int * 4)(1, 2, 3, 5)
    assert f(fake, 0, fake, fake, fake, fake, 0, nz, 3, 256, 256, 128, None, 0, None) == 1        # offsets[0]
    empty = (ctypes.c_int * 4)(0, 0, 0, 0)
    assert f(None, 0, None, None, None, None, 0, empty, 3, 256, 256, 128, None, 0, None) == 0     # no tokens
    assert f(fake, 0, P(0x10008), fake, fake, fake, 0, offs, 3, 256, 256, 128, None, 0, None) == 1


def test_grouped_w4a8_entry_checks(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    f = lib.wq_gemm_w4a8_grouped
    offs = (ctypes.c_int * 4)(0, 2, 2, 5)
    assert f(fake, fake, fake, fake, None, fake, 0, offs, 3, 256, 200, 128, None, 0, None) == 2   # K % 128
    assert f(fake, fake, fake, fake, None, fake, 0, offs, 0, 256, 256, 128, None, 0, None) == 1   # experts
    assert f(fake, fake, fake, fake, None, fake, 0, None, 3, 256, 256, 128, None, 0, None) == 1   # offsets
    bad = (ctypes.c_int * 4)(0, 3, 2, 5)
    assert f(fake, fake, fake, fake, None, fake, 0, bad, 3, 256, 256, 128, None, 0, None) == 1    # decreasing
    empty = (ctypes.c_int * 4)(0, 0, 0, 0)
    assert f(None, None, None, None, None, None, 0, empty, 3, 256, 256, 128, None, 0, None) == 0  # no tokens
    assert f(fake, P(0x10002), fake, fake, None, fake, 0, offs, 3, 256, 256, 128, None, 0, None) == 1  # x_scale
    # beyond 8 tokens per expert (one GEMM per expert) every expert's workspace is checked
    # before anything is enqueued
    big = (ctypes.c_int * 4)(0, 2, 2, 15)
    assert f(fake, fake, fake, fake, None, fake, 0, big, 3, 256, 256, 128, None, 0, None) == 3
    # the binding's sizing (the largest per-expert wq_workspace_size) is exactly what the
    # entry checks: one byte less fails the check, that size passes it (then: no device)
    need = max(lib.wq_workspace_size(2, m, 256, 256, 128) for m in (2, 13))
    assert f(fake, fake, fake, fake, None, fake, 0, big, 3, 256, 256, 128, fake, need - 1, None) == 3
    import torch
    if not torch.cuda.is_available():  # with a GPU present this call would launch on fake pointers
        assert f(fake, fake, fake, fake, None, fake, 0, big, 3, 256, 256, 128, fake, need, None) in (4, 5)


def test_swiglu_pair_entry_checks(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    pk = lib.wq_pack_w4a16_pair
    assert pk(fake, fake, fake, fake, fake, fake, fake, fake, fake, 256, 96, 128, None) == 2    # N % 64
    assert pk(fake, fake, fake, fake, fake, fake, fake, fake, fake, 200, 64, 128, None) == 2    # K % 128
    assert pk(fake, fake, fake, None, fake, fake, fake, fake, fake, 256, 64, 128, None) == 1    # null
    f = lib.wq_gemm_w4a16_swiglu
    assert f(fake, 0, fake, fake, fake, fake, 0, 4, 96, 256, 128, None, 0, None) == 2          # N % 64
    assert f(fake, 2, fake, fake, fake, fake, 0, 4, 64, 256, 128, None, 0, None) == 1          # x dtype
    assert f(None, 0, None, None, None, None, 0, 0, 64, 256, 128, None, 0, None) == 0          # empty
    assert f(P(0x10002), 0, fake, fake, fake, fake, 0, 4, 64, 256, 128, None, 0, None) == 1    # alignment
    # beyond the weight-streaming kernel the fp32 pair product needs a workspace
    assert f(fake, 0, fake, fake, fake, fake, 0, 40, 64, 256, 128, None, 0, None) == 3
    ws = lib.wq_workspace_size
    assert ws(4, 4, 64, 256, 128) == 0 and ws(5, 4, 64, 256, 128) == 0
    assert ws(4, 40, 64, 256, 128) >= 40 * 128 * 4
    assert ws(4, 40, 96, 256, 128) == 0  # N % 64


def test_no_device_means_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    P = ctypes.c_void_p
    fake = P(0x10000)
    rc = lib.wq_pack_w4a16(fake, fake, fake, fake, fake, fake, 256, 256, 128, None)
    assert rc in (4, 5)  # WQ_ERR_ARCH or WQ_ERR_CUDA, never success
    assert lib.wq_device_supported(0) == 0


def _chain(*gemms):
    arr = (wq.ChainGemm * len(gemms))()
    for i, g in enumerate(gemms):
        arr[i] = g
    return arr


def test_chain_entry_checks(lib):
    """wq_gemm_w4a16_chain rejects bad lists before touching the device: the list size,
    M beyond 8 rows, the activation type, forward or mismatched producers, shapes, null
    and misaligned pointers, a workspace that is not 256-byte aligned."""
    f = lib.wq_gemm_w4a16_chain
    x, b, s, y = 0x10000, 0x20000, 0x30000, 0x40000

    def g(X=x, src=-1, B=b, S=s, delta=None, Y=y, yd=0, N=256, K=512, gs=128, pair=0):
        return wq.ChainGemm(X, src, B, S, delta, Y, yd, N, K, gs, pair)

    one = _chain(g())
    assert f(one, 0, 4, 0, None, 0, None) == 1                                   # empty list
    assert f(one, 9, 4, 0, None, 0, None) == 1                                   # more than 8 GEMMs
    assert f(one, 1, 9, 0, None, 0, None) == 2                                   # M > 8
    assert f(one, 1, 4, 2, None, 0, None) == 1                                   # x dtype
    assert f(one, 1, 0, 0, None, 0, None) == 0                                   # M == 0: no-op
    assert f(_chain(g(src=0)), 1, 4, 0, None, 0, None) == 1                      # src not earlier
    assert f(_chain(g(), g(X=None, src=0, K=384)), 2, 4, 0, None, 0, None) == 2  # K != producer N
    assert f(_chain(g(yd=2), g(X=None, src=0, K=256)), 2, 4, 0, None, 0, None) == 1  # producer y dtype
    assert f(_chain(g(), g(X=x, src=0, K=256)), 2, 4, 0, None, 0, None) == 1     # X not the producer's Y
    assert f(_chain(g(N=96, pair=1)), 1, 4, 0, None, 0, None) == 2              # pair N % 64
    assert f(_chain(g(pair=2)), 1, 4, 0, None, 0, None) == 1                    # pair flag
    assert f(_chain(g(K=500)), 1, 4, 0, None, 0, None) == 2                     # K % 128
    assert f(_chain(g(gs=64)), 1, 4, 0, None, 0, None) == 2                     # group size
    assert f(_chain(g(B=None)), 1, 4, 0, None, 0, None) == 1                    # null weights
    assert f(_chain(g(X=x + 2)), 1, 4, 0, None, 0, None) == 1                   # misaligned X
    assert f(_chain(g(yd=5)), 1, 4, 0, None, 0, None) == 1                      # y dtype
    assert f(one, 1, 4, 0, ctypes.c_void_p(0x10080), 1 << 20, None) == 1         # workspace alignment
    ws = lib.wq_chain_workspace_size
    assert ws(one, 0, 4, 0) == 0 and ws(one, 1, 9, 0) == 0 and ws(one, 1, 0, 0) == 0


def test_chain_without_a_device_is_an_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    arr = _chain(wq.ChainGemm(0x10000, -1, 0x20000, 0x30000, None, 0x40000, 0, 256, 512, 128, 0))
    assert lib.wq_gemm_w4a16_chain(arr, 1, 4, 0, ctypes.c_void_p(0x100000), 1 << 20, None) in (4, 5)
    assert lib.wq_chain_workspace_size(arr, 1, 4, 0) == 0
