"""The persistent decode chain (wq_gemm_w4a16_chain) against the fp64 oracle.

Each GEMM of a chain is checked on its own: its output against the oracle's product
of the activations it actually read (the chain's input, or the earlier output it was
given, read back).  Bars (relative Frobenius): fp16 outputs 2e-3 (the W4A16 bar);
bf16 outputs 3e-3 (bf16's unit roundoff 2^-8 alone gives up to 2^-8 / sqrt(3) =
2.3e-3 rms relative rounding error); fp32 outputs 1e-4 (no final rounding; the fp32
accumulation of offset codes costs ~3e-5); the gate/up pair's fp16 / bf16 outputs
3e-3 (the W4A16 bar carried through silu(G) * U to first order is 1.45-1.55 times the
GEMM bar on these inputs).  A chain's split tiles are summed in a fixed order, so
repeated calls and graph replays must be bitwise identical.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-3
TOL_BF16 = 3e-3
TOL_F32 = 1e-4
TOL_PAIR = 3e-3


def _bar(Y):
    return {torch.float16: TOL, torch.bfloat16: TOL_BF16, torch.float32: TOL_F32}[Y.dtype]


@pytest.fixture(scope="module")
def wq():
    import weight_only_int4_g128_gb300 as m
    m.load_library(build_if_missing=True)
    assert m.device_supported(torch.cuda.current_device())
    m.device_status(reset=True)
    return m


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _acts(rng, M, K, adt):
    a = rng.standard_normal((M, K))
    if adt == "bf16":
        A = oracle.double_to_bf16(a)
        return _cuda(A.view(np.int16)).view(torch.bfloat16), oracle.bf16_to_double(A)
    A = a.astype(np.float16)
    return _cuda(A), A.astype(np.float64)


def _w(rng, K, N, gs):
    G = K // (K if gs == -1 else gs)
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    s = rng.uniform(0.005, 0.02, size=(G, N)).astype(np.float16)
    z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
    return q, s, z


def _plain(wq, w, gs, sym=False):
    q, s, z = w
    B, S, dl = wq.pack_w4a16(_cuda(q), _cuda(s), _cuda(z), gs)
    return {"B": B, "S": S, "delta": None if sym else dl, "group_size": gs}


def _pair(wq, gate, up, gs, sym=False):
    (qg, sg, zg), (qu, su, zu) = gate, up
    B, S, dl = wq.pack_w4a16_pair(_cuda(qg), _cuda(sg), _cuda(zg), _cuda(qu), _cuda(su), _cuda(zu), gs)
    return {"B": B, "S": S, "delta": None if sym else dl, "group_size": gs, "pair": True}


def _ref_plain(A64, w, gs, sym=False, cols=None):
    q, s, z = w
    if sym:
        return oracle.gemm_asym_identity(A64, q, oracle.half_bits(s), None, gs, cols=cols)
    return oracle.gemm_asym_plain(A64, q, oracle.half_bits(s), oracle.half_bits(z), gs, cols=cols)


def _ref_pair(A64, gate, up, gs, sym=False):
    g = (gate[0], oracle.half_bits(gate[1]), None if sym else oracle.half_bits(gate[2]))
    u = (up[0], oracle.half_bits(up[1]), None if sym else oracle.half_bits(up[2]))
    return oracle.gemm_swiglu_pair(A64, g, u, gs)


def _read(Y):
    if Y.dtype == torch.bfloat16:
        return oracle.bf16_to_double(Y.view(torch.int16).cpu().numpy())
    return Y.double().cpu().numpy()


MLP = [
    # M, K, F (intermediate width), N, group, activations, symmetric
    (1, 512, 384, 640, 128, "f16", False),      # every CTA one k-block: tiles split over kb CTAs
    (3, 1024, 256, 384, -1, "bf16", False),     # one group per column, bf16 rows
    (8, 4096, 1024, 512, 128, "f16", True),     # symmetric weights, all 8 token slots
    (5, 2048, 640, 1024, 128, "bf16", False),
]


@pytest.mark.parametrize("M,K,F,N,gs,adt,sym", MLP)
def test_mlp_chain_parity(wq, M, K, F, N, gs, adt, sym):
    """A decode MLP in one launch: gate/up pair with SwiGLU, then the down projection
    reading the pair's output; each GEMM within its bar of the oracle."""
    rng = np.random.default_rng(9100 + M + K + F)
    X, A64 = _acts(rng, M, K, adt)
    gate, up, down = _w(rng, K, F, gs), _w(rng, K, F, gs), _w(rng, F, N, gs)
    xdt = X.dtype
    Y0, Y1 = wq.gemm_w4a16_chain(X, [dict(_pair(wq, gate, up, gs, sym), out_dtype=xdt),
                                     dict(_plain(wq, down, gs, sym), src=0)])
    torch.cuda.synchronize()
    assert Y0.shape == (M, F) and Y1.shape == (M, N)
    err0 = oracle.rel_fro(_read(Y0), _ref_pair(A64, gate, up, gs, sym))
    assert err0 <= TOL_PAIR, err0
    err1 = oracle.rel_fro(_read(Y1), _ref_plain(_read(Y0), down, gs, sym))
    assert err1 <= _bar(Y1), err1
    assert wq.device_status(reset=True) == 0


def test_mlp_chain_full_size(wq):
    """The decode MLP of the c1 model dimensions (K 4096, two 11008-wide projections,
    down 11008 -> 4096), 4 tokens, fp32 down output: the pair within its bar, the down
    projection within the fp32 bar on its input (a column sample of the oracle)."""
    M, K, F, N, gs = 4, 4096, 11008, 4096, 128
    rng = np.random.default_rng(9200)
    X, A64 = _acts(rng, M, K, "f16")
    gate, up, down = _w(rng, K, F, gs), _w(rng, K, F, gs), _w(rng, F, N, gs)
    Y0, Y1 = wq.gemm_w4a16_chain(X, [_pair(wq, gate, up, gs),
                                     dict(_plain(wq, down, gs), src=0, out_dtype=torch.float32)])
    torch.cuda.synchronize()
    err0 = oracle.rel_fro(_read(Y0), _ref_pair(A64, gate, up, gs))
    assert err0 <= TOL_PAIR, err0
    for n0, n1 in ((0, 160), (1990, 2200), (N - 200, N)):  # column windows across tile edges
        ref1 = _ref_plain(_read(Y0), down, gs, cols=(n0, n1))
        err1 = oracle.rel_fro(_read(Y1)[:, n0:n1], ref1)
        assert err1 <= TOL_F32, (n0, err1)
    assert wq.device_status(reset=True) == 0


def test_independent_gemms_and_a_three_level_chain(wq):
    """Three GEMMs on the same input (attention-style projections), one on a second input,
    and A -> B -> C where each reads the previous output, all in one launch."""
    M, K, gs = 6, 1024, 128
    rng = np.random.default_rng(9300)
    X, A64 = _acts(rng, M, K, "f16")
    X2, A2 = _acts(rng, M, 768, "f16")
    wqkv = [_w(rng, K, n, gs) for n in (512, 256, 384)]
    w4 = _w(rng, 768, 640, gs)
    wa, wb, wc = _w(rng, K, 384, gs), _w(rng, 384, 896, gs), _w(rng, 896, 256, gs)
    steps = [_plain(wq, w, gs) for w in wqkv]
    steps.append(dict(_plain(wq, w4, gs), x=X2, out_dtype=torch.float32))
    steps.append(_plain(wq, wa, gs))
    steps.append(dict(_plain(wq, wb, gs, sym=True), src=4))
    steps.append(dict(_plain(wq, wc, gs), src=5, out_dtype=torch.bfloat16))
    Ys = wq.gemm_w4a16_chain(X, steps)
    torch.cuda.synchronize()
    for Y, w in zip(Ys[:3], wqkv):
        assert oracle.rel_fro(_read(Y), _ref_plain(A64, w, gs)) <= _bar(Y)
    assert oracle.rel_fro(_read(Ys[3]), _ref_plain(A2, w4, gs)) <= _bar(Ys[3])
    assert oracle.rel_fro(_read(Ys[4]), _ref_plain(A64, wa, gs)) <= _bar(Ys[4])
    assert oracle.rel_fro(_read(Ys[5]), _ref_plain(_read(Ys[4]), wb, gs, sym=True)) <= _bar(Ys[5])
    assert oracle.rel_fro(_read(Ys[6]), _ref_plain(_read(Ys[5]), wc, gs)) <= _bar(Ys[6])
    assert wq.device_status(reset=True) == 0


@pytest.mark.parametrize("M,K,N", [
    (1, 256, 77824),    # ranges of 4 k-blocks over 2-k-block tiles: whole tiles stored directly,
                        # windows that cover all of K and wrap
    (8, 4096, 25600),   # 21-22 k-blocks per range, more than one window of 19 at M = 8
])
def test_range_shapes(wq, M, K, N):
    """Stream-K ranges longer than a tile and longer than one activation window."""
    gs = 128
    rng = np.random.default_rng(9400 + M)
    X, A64 = _acts(rng, M, K, "f16")
    w = _w(rng, K, N, gs)
    (Y,) = wq.gemm_w4a16_chain(X, [dict(_plain(wq, w, gs), out_dtype=torch.float32)])
    torch.cuda.synchronize()
    for n0, n1 in ((0, 200), (N // 2 - 100, N // 2 + 300), (N - 260, N)):  # windows across tile edges
        err = oracle.rel_fro(_read(Y)[:, n0:n1], _ref_plain(A64, w, gs, cols=(n0, n1)))
        assert err <= TOL_F32, (n0, err)
    assert wq.device_status(reset=True) == 0


def test_repeat_calls_and_graph_replays_are_bitwise_identical(wq):
    """Calls on one workspace (the generation advances every call) give identical bits; a
    captured call replayed on new activations equals the eager call on them."""
    M, K, F, N, gs = 4, 1024, 512, 384, 128
    rng = np.random.default_rng(9500)
    X, _ = _acts(rng, M, K, "f16")
    gate, up, down = _w(rng, K, F, gs), _w(rng, K, F, gs), _w(rng, F, N, gs)
    steps = [_pair(wq, gate, up, gs), dict(_plain(wq, down, gs), src=0)]
    first = [y.clone() for y in wq.gemm_w4a16_chain(X, steps)]
    for _ in range(3):
        again = wq.gemm_w4a16_chain(X, steps)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    Xg = X.clone()
    outs = [torch.empty_like(first[0]), torch.empty_like(first[1])]
    gsteps = [dict(steps[0], out=outs[0]), dict(steps[1], out=outs[1])]
    ws = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")  # zeroed once, kept by the graph
    wq.gemm_w4a16_chain(Xg, gsteps, workspace=ws)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wq.gemm_w4a16_chain(Xg, gsteps, workspace=ws)
    for r in range(3):
        Xn, _ = _acts(np.random.default_rng(9600 + r), M, K, "f16")
        Xg.copy_(Xn)
        g.replay()
        torch.cuda.synchronize()
        ref = wq.gemm_w4a16_chain(Xn, steps)
        for a, b in zip(outs, ref):
            assert torch.equal(a, b)
    assert wq.device_status(reset=True) == 0


def test_chain_of_one_matches_its_oracle_for_every_output_type(wq):
    """A single GEMM through the chain entry, fp16 / bf16 / fp32 outputs."""
    M, K, N, gs = 7, 640, 256, 128
    rng = np.random.default_rng(9700)
    X, A64 = _acts(rng, M, K, "f16")
    w = _w(rng, K, N, gs)
    ref = _ref_plain(A64, w, gs)
    for dt in (torch.float16, torch.bfloat16, torch.float32):
        (Y,) = wq.gemm_w4a16_chain(X, [dict(_plain(wq, w, gs), out_dtype=dt)])
        torch.cuda.synchronize()
        assert oracle.rel_fro(_read(Y), ref) <= _bar(Y)


def test_one_workspace_serves_different_chains(wq):
    """Chains of different shapes in turn on one workspace (its control words at fixed
    offsets, left consistent by every call): each result equals the same chain on a
    fresh workspace, bit for bit."""
    M, gs = 4, 128
    rng = np.random.default_rng(9800)
    X, _ = _acts(rng, M, 1024, "f16")
    H, _ = _acts(rng, M, 2048, "f16")
    gate, up, down = _w(rng, 1024, 512, gs), _w(rng, 1024, 512, gs), _w(rng, 512, 768, gs)
    big = _w(rng, 2048, 1024, gs)
    mlp = [_pair(wq, gate, up, gs), dict(_plain(wq, down, gs), src=0)]
    single = [_plain(wq, big, gs)]
    ref_mlp = [y.clone() for y in wq.gemm_w4a16_chain(X, mlp, workspace=torch.zeros(8 << 20, dtype=torch.uint8,
                                                                                      device="cuda"))]
    ref_one = wq.gemm_w4a16_chain(H, single, workspace=torch.zeros(8 << 20, dtype=torch.uint8, device="cuda"))[0]
    ws = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        one = wq.gemm_w4a16_chain(H, single, workspace=ws)[0]
        two = wq.gemm_w4a16_chain(X, mlp, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(one, ref_one)
        for a, b in zip(two, ref_mlp):
            assert torch.equal(a, b)
    assert wq.device_status(reset=True) == 0


def test_chain_limits_on_the_device(wq):
    """With a device present: a chain of more than 65536 output tiles and a workspace
    smaller than the query are refused before anything is launched (the placeholder
    pointers below are never dereferenced)."""
    import ctypes
    lib = wq.load_library()
    arr = (wq.ChainGemm * 1)()
    arr[0] = wq.ChainGemm(0x10000, -1, 0x20000, 0x30000, None, 0x40000, 0, 128 * 65537, 128, 128, 0)
    assert lib.wq_chain_workspace_size(arr, 1, 4, 0) == 0
    assert lib.wq_gemm_w4a16_chain(arr, 1, 4, 0, ctypes.c_void_p(0x100000), 1 << 30, None) == 2
    arr[0] = wq.ChainGemm(0x10000, -1, 0x20000, 0x30000, None, 0x40000, 0, 256, 512, 128, 0)
    need = lib.wq_chain_workspace_size(arr, 1, 4, 0)
    assert need > 0
    assert lib.wq_gemm_w4a16_chain(arr, 1, 4, 0, ctypes.c_void_p(0x100000), need - 256, None) == 3
