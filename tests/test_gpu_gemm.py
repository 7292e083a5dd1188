"""GPU GEMM parity against the fp64 oracle, through the C ABI.

Bars: ||Y - C_ref||_F / ||C_ref||_F <= 2e-3 for W4A16 (fp32 accumulate), and
<= 5e-4 for the large-M W4A16 path, whose weights are RN((q - 8) * scale) in fp16
for either activation type (a relative rms rounding error of ~2e-4); W4A8
<= 2e-3 against the oracle over the int8 activations and <= 5 % against the
fp16-activation oracle (the acceptance level of the HyperQwen article, section
"int8 tensor cores: how the numbers were verified").  Special cases whose
result is exact (one-hot rows, integer weights, zero weights) are compared bit
for bit, and repeated runs must be bitwise identical.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_W4A16 = 2e-3
TOL_W4A8 = 2e-3
TOL_W4A8_VS_F16 = 5e-2


@pytest.fixture(scope="module")
def wq():
    import weight_only_int4_g128_gb300 as m
    m.load_library(build_if_missing=True)
    assert m.device_supported(torch.cuda.current_device())
    return m


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _x(d):
    if d["a_dtype"] == "bf16":
        return _cuda(d["A"].view(np.int16)).view(torch.bfloat16)
    return _cuda(d["A"])


def _w4a16(wq, d, out_dtype=torch.float16, sym=False):
    gs = d["group_size"]
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), gs)
    Y = wq.gemm_w4a16(_x(d), Bp, S, None if sym else dl, gs, out_dtype)
    torch.cuda.synchronize()
    return Y, (Bp, S, dl)


def _ref_w4a16(d, sym=False, rows=None, cols=None):
    A = oracle.activations_to_double(d["A"], d["a_dtype"])
    if rows is not None:
        A = A[rows]
    sb = oracle.half_bits(d["scale"])
    if sym:
        return oracle.gemm_asym_identity(A, d["q"], sb, None, d["group_size"], cols=cols)
    return oracle.gemm_asym_plain(A, d["q"], sb, oracle.half_bits(d["zero"]), d["group_size"],
                                  cols=cols)


SMALL = [
    # M, K, N, group, a_dtype        (tiles of 128 columns, token tiles 16..256, ragged M)
    (1, 256, 256, 128, "f16"),
    (16, 256, 256, 128, "f16"),      # the K=256 shape of the small config
    (5, 1024, 384, 128, "f16"),
    (17, 512, 256, 128, "f16"),
    (40, 768, 128, 128, "f16"),
    (100, 384, 256, 128, "f16"),
    (300, 512, 384, 128, "f16"),
    (3, 128, 128, 128, "f16"),       # a single k-block
    (24, 1024, 256, -1, "f16"),      # one group per column
    (9, 640, 256, 128, "bf16"),
    (200, 1280, 256, 128, "bf16"),
    (64, 2048, 256, -1, "bf16"),
    # decode kernel: more k-blocks per CTA than ring stages, bf16, one group per
    # column, 8 tokens
    (2, 5120, 128, 128, "f16"),
    (7, 8192, 256, 128, "bf16"),
    (6, 1024, 256, -1, "f16"),
    (8, 2048, 384, 128, "f16"),
    (4, 640, 256, -1, "bf16"),
]


@pytest.mark.parametrize("M,K,N,gs,adt", SMALL)
def test_w4a16_small_parity(wq, M, K, N, gs, adt):
    d = synth.make_inputs(1000 + M * 7 + K, M, K, N, group_size=gs, a_dtype=adt)
    Y, _ = _w4a16(wq, d)
    ref = _ref_w4a16(d)
    err = oracle.rel_fro(Y.double().cpu().numpy(), ref)
    assert err <= TOL_W4A16, err


@pytest.mark.parametrize("M", [33, 5])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_w4a16_output_dtypes(wq, out_dtype, M):
    d = synth.make_inputs(77, M, 512, 256)
    Y, _ = _w4a16(wq, d, out_dtype)
    assert Y.dtype == out_dtype
    err = oracle.rel_fro(Y.double().cpu().numpy(), _ref_w4a16(d))
    assert err <= (TOL_W4A16 if out_dtype != torch.float32 else 1e-3), err


@pytest.mark.parametrize("M", [4, 130])
def test_w4a16_symmetric_parity(wq, M):
    d = synth.make_inputs(88 + M, M, 512, 256)
    Y, _ = _w4a16(wq, d, torch.float32, sym=True)
    err = oracle.rel_fro(Y.double().cpu().numpy(), _ref_w4a16(d, sym=True))
    assert err <= 1e-3, err


@pytest.mark.parametrize("adt", ["f16", "bf16"])
@pytest.mark.parametrize("K", [128, 256, 1024])
def test_one_hot_rows_give_dequantized_weights_bit_exact(wq, adt, K):
    """X = I_K (one-hot rows, M = K > 16: the large-M kernel): Y[k, :] is the dequantized
    row k, bit for bit.  The large-M kernel feeds RN((q - 8) * scale) in fp16 for both
    activation types (bf16 rows are scaled by a power of two and copied to fp16 exactly,
    and the scale is undone at the store), so with fp32 output the rows are exactly the
    fp16 dequantized weights."""
    N = 256
    d = synth.make_inputs(500 + K, K, K, N, a_dtype=adt)
    eye = np.eye(K, dtype=np.float32)
    if adt == "bf16":
        d["A"] = (eye.view(np.uint32) >> 16).astype(np.uint16)
        Y, _ = _w4a16(wq, d, torch.float32, sym=True)
        want = oracle.dequant_sym_f16(d["q"], oracle.half_bits(d["scale"]), 128).view(np.float16)
        assert np.array_equal(Y.cpu().numpy(), want.astype(np.float32))
    else:
        d["A"] = eye.astype(np.float16)
        Y, _ = _w4a16(wq, d, torch.float16, sym=True)
        got = Y.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, oracle.dequant_sym_f16(d["q"], oracle.half_bits(d["scale"]), 128))


TOL_LARGE_M = 5e-4  # large M: 11-bit weights, expected ~2-3e-4 (see test below)


@pytest.mark.parametrize("M,K,N,gs,adt", [(300, 1024, 384, 128, "bf16"), (64, 2048, 256, -1, "bf16"),
                                          (40, 768, 256, 128, "bf16"), (200, 1280, 256, 128, "f16"),
                                          # K / 8 an odd multiple of 16 (half a warp past the last full
                                          # 32-chunk stride of the bf16 copy), an odd M
                                          (41, 640, 256, 128, "bf16"), (33, 1152, 128, -1, "bf16")])
def test_large_m_precision(wq, M, K, N, gs, adt):
    """Large-M W4A16 against the oracle with fp32 output, within 5e-4 for both activation
    types: the weights are RN((q - 8) * scale) in fp16 (11 significant bits, a relative
    rms rounding error of ~2e-4), bf16 activations reaching the tensor cores unchanged
    through their scaled fp16 copy."""
    d = synth.make_inputs(1500 + M + K, M, K, N, group_size=gs, a_dtype=adt)
    Y, _ = _w4a16(wq, d, torch.float32)
    err = oracle.rel_fro(Y.double().cpu().numpy(), _ref_w4a16(d))
    print(f"\nlarge M {M}x{K}x{N} g{gs} {adt}: rel. error {err:.3e}")
    assert err <= TOL_LARGE_M, err


@pytest.mark.parametrize("M,K,N,gs,adt,odt", [(300, 12288, 10240, 128, "f16", torch.float16),
                                              (280, 13312, 10240, -1, "bf16", torch.float32)])
def test_large_m_last_wave_split_along_k(wq, M, K, N, gs, adt, odt):
    """2 x 80 = 160 tiles of 256 tokens and 96 or more k-blocks: the last wave of 152
    one-CTA slots holds 8 tiles, which run as a second launch split along K (a cluster
    per tile).  Those tiles (rows 256.., the last 8 column tiles) and tiles of the first
    launch are checked against the oracle."""
    d = synth.make_inputs(1700 + M, M, K, N, group_size=gs, a_dtype=adt)
    Y, _ = _w4a16(wq, d, odt)
    got = Y.double().cpu().numpy()
    for c in [(N - 1024, N), (0, 256)]:
        err = oracle.rel_fro(got[:, c[0]:c[1]], _ref_w4a16(d, cols=c))
        assert err <= TOL_LARGE_M, (c, err)


@pytest.mark.parametrize("M,K,N,gs,adt,odt,sym", [
    (600, 1024, 16384, 128, "f16", torch.float16, False),   # 384 tiles, 9 stages per tile (odd)
    (520, 1152, 16384, 128, "bf16", torch.float16, False),  # 9 k-blocks + a correction stage: 10 (even)
    (700, 1024, 12288, -1, "f16", torch.float16, True),     # symmetric, one group per column: 8 stages
])
def test_large_m_several_waves(wq, M, K, N, gs, adt, odt, sym):
    """More than one wave of 256-token tiles (288 or 384 tiles over 152 one-CTA slots),
    odd and even stage counts per tile, the last token tile ragged: column windows at
    the start, middle and end against the oracle, and a repeat call bit-equal."""
    d = synth.make_inputs(1800 + M, M, K, N, group_size=gs, a_dtype=adt)
    Y, _ = _w4a16(wq, d, odt, sym=sym)
    got = Y.double().cpu().numpy()
    for c in [(0, 384), (N // 2 - 128, N // 2 + 128), (N - 384, N)]:
        err = oracle.rel_fro(got[:, c[0]:c[1]], _ref_w4a16(d, sym=sym, cols=c))
        assert err <= TOL_LARGE_M, (c, err)
    Y2, _ = _w4a16(wq, d, odt, sym=sym)
    assert torch.equal(Y, Y2)


def test_bf16_rows_of_any_magnitude(wq):
    """bf16 rows far outside fp16's range (1e30, 1e-30), near its limits (1e4 -> values
    above 65504, 1e-6 -> fp16 subnormals) and all-zero rows: each token row is scaled by
    its own power of two before the fp16 copy, so every row keeps the 5e-4 bar relative
    to its own size, and zero rows give exact zeros."""
    M, K, N = 48, 1024, 256
    d = synth.make_inputs(1600, M, K, N, a_dtype="bf16")
    A = oracle.activations_to_double(d["A"], "bf16")
    mags = np.array([1e30, 1e-30, 1e4, 1e-6, 0.0, 1.0, 3e5, 2e-20])
    f = np.resize(mags, M)
    A32 = (A * f[:, None]).astype(np.float32)
    d["A"] = (A32.view(np.uint32) >> 16).astype(np.uint16)  # truncation: still bf16 values
    Y, _ = _w4a16(wq, d, torch.float32)
    got = Y.double().cpu().numpy()
    ref = _ref_w4a16(d)
    for m in range(M):
        if f[m] == 0.0:
            assert not np.any(got[m]), m
        else:
            err = oracle.rel_fro(got[m:m + 1], ref[m:m + 1])
            assert err <= TOL_LARGE_M, (m, f[m], err)


@pytest.mark.parametrize("M", [4, 8, 16])
@pytest.mark.parametrize("adt", ["f16", "bf16"])
@pytest.mark.parametrize("gs", [128, -1])
def test_one_hot_decode_path_bit_exact(wq, adt, gs, M):
    """M one-hot rows (the decode kernel): Y[m, :] = RN((q - 8) * scale) of row k_m."""
    K, N = 2048, 384
    d = synth.make_inputs(550, M, K, N, group_size=gs, a_dtype=adt)
    ks = np.array([0, 1, 7, 8, 127, 128, 129, 511, 640, 1000, 1023, 1024, 1500, 2000, 2046, 2047])
    if M < 16:
        ks = ks[np.linspace(0, 15, M).astype(int)]
    eye = np.zeros((M, K), np.float32)
    eye[np.arange(M), ks] = 1.0
    if adt == "bf16":
        d["A"] = (eye.view(np.uint32) >> 16).astype(np.uint16)
        out, fn = torch.bfloat16, oracle.dequant_sym_bf16
    else:
        d["A"] = eye.astype(np.float16)
        out, fn = torch.float16, oracle.dequant_sym_f16
    Y, _ = _w4a16(wq, d, out, sym=True)
    got = Y.cpu().view(torch.int16).numpy().view(np.uint16)
    want = fn(d["q"], oracle.half_bits(d["scale"]), gs)[ks]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,K", [(8, 512), (3, 4096), (70, 1024), (257, 256), (16, 4096)])
def test_integer_weights_exact(wq, M, K):
    """scale = 1, zero = -8 (so delta = 0): C = X @ (q - 8) is an exact integer matmul."""
    N = 256
    rng = np.random.Generator(np.random.PCG64(M))
    d = synth.make_inputs(600 + M, M, K, N)
    d["A"] = rng.integers(-3, 4, (M, K)).astype(np.float16)
    d["scale"] = np.ones_like(d["scale"])
    d["zero"] = np.full_like(d["zero"], -8.0)
    Y, _ = _w4a16(wq, d, torch.float32)
    want = d["A"].astype(np.int64) @ (d["q"].astype(np.int64) - 8)
    assert np.array_equal(Y.cpu().numpy().astype(np.int64), want)
    assert np.array_equal(Y.cpu().numpy(), want.astype(np.float32))


def test_zero_weights_give_exact_zero(wq):
    """q == 8 and zero = -8*scale: W == 0, delta == 0, so Y == 0 exactly."""
    d = synth.make_inputs(700, 33, 512, 256)
    d["q"] = np.full_like(d["q"], 8)
    d["zero"] = (-8.0 * d["scale"].astype(np.float64)).astype(np.float16)
    Y, _ = _w4a16(wq, d, torch.float32)
    assert torch.count_nonzero(Y).item() == 0


def test_correction_term_matters(wq):
    """Dropping delta changes the result by exactly the A_group_sum @ delta term."""
    d = synth.make_inputs(701, 16, 1024, 256)
    Ya, (Bp, S, dl) = _w4a16(wq, d, torch.float32)
    Ys = wq.gemm_w4a16(_x(d), Bp, S, None, 128, torch.float32)
    A = oracle.activations_to_double(d["A"], "f16")
    corr = oracle.group_sum(A, 128) @ dl.cpu().double().numpy()
    err = oracle.rel_fro((Ya - Ys).double().cpu().numpy(), corr)
    assert err < 1e-4, err


@pytest.mark.parametrize("M", [1, 16, 100])
def test_repeat_runs_bitwise_identical(wq, M):
    d = synth.make_inputs(800 + M, M, 4096, 512)
    Y1, (Bp, S, dl) = _w4a16(wq, d)
    X = _x(d)
    for _ in range(3):
        Y2 = wq.gemm_w4a16(X, Bp, S, dl, 128)
        assert torch.equal(Y1, Y2)


@pytest.mark.parametrize("M,K,N", [(1, 256, 256), (16, 512, 384), (100, 1024, 256),
                                   (300, 256, 128)])
def test_w4a8_parity(wq, M, K, N):
    d = synth.make_inputs(900 + M, M, K, N, mode="w4a8")
    gXq, gxs = wq.quantize_per_token(_cuda(d["A"]))
    Xq, xs = oracle.quantize_per_token(d["A"])
    assert np.array_equal(gXq.cpu().numpy(), Xq) and np.array_equal(gxs.cpu().numpy(), xs)
    Bp, S = wq.pack_w4a8(_cuda(d["q"]), _cuda(d["scale"]), 128)
    Y = wq.gemm_w4a8(gXq, gxs, Bp, S, 128, torch.float32)
    torch.cuda.synchronize()
    qf, sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), 128)
    ref8 = oracle.gemm_w4a8(Xq, xs, qf, sf, 128)
    y = Y.double().cpu().numpy()
    assert oracle.rel_fro(y, ref8) <= TOL_W4A8
    ref16 = oracle.gemm_asym_identity(oracle.activations_to_double(d["A"], "f16"), qf, sf, None, 128)
    assert oracle.rel_fro(y, ref16) <= TOL_W4A8_VS_F16


def test_w4a8_last_wave_split_along_k(wq):
    """W4A8 over 2 x 80 = 160 tiles of 256 tokens with 96 k-blocks: the last wave runs
    as a K-split second launch whose owners apply the per-token scale at their store;
    the tail tiles and first-launch tiles against the int8 oracle."""
    M, K, N = 300, 12288, 10240
    d = synth.make_inputs(1950, M, K, N, mode="w4a8")
    Xq, xs = oracle.quantize_per_token(d["A"])
    Bp, S = wq.pack_w4a8(_cuda(d["q"]), _cuda(d["scale"]), 128)
    Y = wq.gemm_w4a8(_cuda(Xq), _cuda(xs), Bp, S, 128, torch.float32)
    torch.cuda.synchronize()
    qf, sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), 128)
    y = Y.double().cpu().numpy()
    for c in [(N - 1024, N), (0, 256)]:
        ref8 = oracle.gemm_w4a8(Xq, xs, qf, sf, 128, cols=c)
        assert oracle.rel_fro(y[:, c[0]:c[1]], ref8) <= TOL_W4A8, c


@pytest.mark.parametrize("M,K", [(1, 4096), (5, 1024), (8, 2048), (12, 1024), (40, 1024), (300, 2048)])
def test_w4a8_integer_problems_exact(wq, M, K):
    """Unit scales and unit per-token scales make Y = Xq @ (q - 8), an integer below 2^24:
    every path (the weight-streaming kernel, which stages the int8 rows as exact fp16, for
    M <= 8; the e4m3 tcgen05 kernel for M 9..16; the large-M kernel on exact fp16 rows and
    weights) gives it exactly in fp32, so no low bit of an integer sum is dropped."""
    rng = np.random.default_rng(990 + M)
    N = 256
    Xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    ones = np.ones((K // 128, N), np.float16)
    Bp, S = wq.pack_w4a8(_cuda(q), _cuda(ones), 128)
    Y = wq.gemm_w4a8(_cuda(Xq), _cuda(np.ones(M, np.float32)), Bp, S, 128, torch.float32)
    torch.cuda.synchronize()
    want = Xq.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.array_equal(Y.cpu().numpy().astype(np.int64), want)
    assert np.array_equal(Y.cpu().numpy(), want.astype(np.float32))


def test_w4a8_gpu_quantizer_end_to_end(wq):
    d = synth.make_inputs(950, 24, 1024, 256, mode="w4a8")
    Xq, xs = wq.quantize_per_token(_cuda(d["A"]))
    Bp, S = wq.pack_w4a8(_cuda(d["q"]), _cuda(d["scale"]), 128)
    Y = wq.gemm_w4a8(Xq, xs, Bp, S, 128)
    oXq, oxs = oracle.quantize_per_token(d["A"])
    qf, sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), 128)
    ref8 = oracle.gemm_w4a8(oXq, oxs, qf, sf, 128)
    assert oracle.rel_fro(Y.double().cpu().numpy(), ref8) <= TOL_W4A8


def test_empty_and_error_paths(wq):
    d = synth.make_inputs(960, 64, 256, 256)
    Y, (Bp, S, dl) = _w4a16(wq, d)
    X0 = torch.empty((0, 256), dtype=torch.float16, device="cuda")
    assert wq.gemm_w4a16(X0, Bp, S, dl, 128).shape == (0, 256)
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(wq.WQError) as e:
        wq.gemm_w4a16(_x(d), Bp, S, dl, 128, workspace=small)
    assert e.value.code == 3


def test_bounded_wait_expires_and_context_survives(wq):
    """A wait nothing will complete gives up after its limit and reports it; the
    context stays usable afterwards."""
    wq.device_status(reset=True)
    wq.debug_wait_probe(50_000_000)  # 50 ms
    st = wq.device_status(reset=True)
    assert st & (1 << 4)
    d = synth.make_inputs(970, 16, 256, 256)
    Y, _ = _w4a16(wq, d)
    assert oracle.rel_fro(Y.double().cpu().numpy(), _ref_w4a16(d)) <= TOL_W4A16
    assert wq.device_status(reset=True) == 0


# ---------------------------------------------------------------- full-size configs, sampled
def _sample_cols(N, width=48):
    return [(0, width), (N // 2 - 64, N // 2 - 64 + width), (N - width, N)]


def _sample_rows(M, count=48):
    if M <= count:
        return np.arange(M)
    return np.unique(np.linspace(0, M - 1, count).astype(np.int64))


FULL = [(w, i) for w in ("c0", "c1", "c2", "c3", "c4") for i in range(len(synth.shapes(w)))]


@pytest.mark.parametrize("workload,idx", FULL)
def test_full_size_workloads_sampled(wq, workload, idx, record_property):
    """Every configuration's shapes at full size, in the bench's launch configuration, on
    sampled rows and column windows against the oracle; the largest measured error of
    each shape is recorded (junit property rel_err_max, and printed with -s)."""
    seed, s = synth.shapes(workload)[idx]
    errs = []
    d = synth.make_inputs(seed, **s)
    rows = _sample_rows(s["M"])
    gs = s["group_size"]
    if s["mode"] == "w4a8":
        Xq, xs = wq.quantize_per_token(_cuda(d["A"]))
        Bp, S = wq.pack_w4a8(_cuda(d["q"]), _cuda(d["scale"]), gs)
        Y = wq.gemm_w4a8(Xq, xs, Bp, S, gs)
        torch.cuda.synchronize()
        Xq_h, xs_h = Xq.cpu().numpy(), xs.cpu().numpy()
        oXq, oxs = oracle.quantize_per_token(d["A"][rows])
        assert np.array_equal(Xq_h[rows], oXq) and np.array_equal(xs_h[rows], oxs)
        qf, sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), gs)
        A16 = d["A"][rows].astype(np.float64)  # the fp16 activations before quantization
        for c in _sample_cols(s["N"]):
            ref8 = oracle.gemm_w4a8(oXq, oxs, qf, sf, gs, cols=c)
            # the fp16-activation reference over the same (folded) weights: scale 1 per token
            ref16 = oracle.gemm_asym_identity(A16, qf, sf, None, gs, cols=c)
            got = Y[rows][:, c[0]:c[1]].double().cpu().numpy()
            errs.append(oracle.rel_fro(got, ref8))
            assert errs[-1] <= TOL_W4A8
            assert oracle.rel_fro(got, ref16) <= TOL_W4A8_VS_F16
    else:
        Y, _ = _w4a16(wq, d)
        for c in _sample_cols(s["N"]):
            ref = _ref_w4a16(d, rows=rows, cols=c)
            got = Y[rows][:, c[0]:c[1]].double().cpu().numpy()
            err = oracle.rel_fro(got, ref)
            errs.append(err)
            assert err <= (TOL_LARGE_M if s["M"] > 16 else TOL_W4A16), (c, err)
    record_property("rel_err_max", max(errs))
    print(f"\n{workload}[{idx}] M{s['M']} K{s['K']} N{s['N']}: max sampled rel. error {max(errs):.3e}")


@pytest.mark.parametrize("prefetch", [False, True])
def test_back_to_back_launches_see_their_inputs(wq, prefetch):
    """Decode GEMMs launched back to back (programmatic dependent launch) read activations
    written by the kernel launched just before them, eagerly and inside a CUDA graph, and
    match synchronised runs bit for bit."""
    M, K, N = 4, 2048, 512
    d = synth.make_inputs(980, M, K, N)
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), 128)
    X = _cuda(d["A"])
    refs = []
    for i in range(4):
        Xi = X * (i + 1)
        torch.cuda.synchronize()
        refs.append(wq.gemm_w4a16(Xi, Bp, S, dl, 128))
        torch.cuda.synchronize()
    wq.set_weight_prefetch(prefetch)
    try:
        outs = [wq.gemm_w4a16(X * (i + 1), Bp, S, dl, 128) for i in range(4)]
        torch.cuda.synchronize()
        for Y, R in zip(outs, refs):
            assert torch.equal(Y, R)
        Ys = [torch.empty_like(refs[0]) for _ in range(4)]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(4):
                    wq.gemm_w4a16(X * (i + 1), Bp, S, dl, 128, out=Ys[i])
            for _ in range(3):
                for Y in Ys:
                    Y.zero_()
                g.replay()
        torch.cuda.synchronize()
        for Y, R in zip(Ys, refs):
            assert torch.equal(Y, R)
        sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
        for i, Y in enumerate(Ys):
            A64 = (X * (i + 1)).double().cpu().numpy()  # the fp16 activations the GEMM read
            ref = oracle.gemm_asym_plain(A64, d["q"], sb, zb, 128)
            assert oracle.rel_fro(Y.double().cpu().numpy(), ref) <= TOL_W4A16, i
    finally:
        wq.set_weight_prefetch(False)


@pytest.mark.parametrize("M,K,N,adt,sym,ydt", [
    (4, 2048, 512, "f16", False, torch.float16),      # decode kernel
    (16, 1024, 384, "bf16", True, torch.bfloat16),    # decode kernel, symmetric
    (300, 512, 384, "f16", False, torch.float32),     # large-M kernel with the correction pre-pass
    (130, 1280, 256, "bf16", False, torch.float16),
])
def test_host_buffer_entry_matches_device_entry(wq, M, K, N, adt, sym, ydt):
    """gemm_w4a16_host (host X and Y, copies on the stream) gives the device entry's
    result bit for bit, and the oracle's within the W4A16 tolerance; two calls in a row
    reuse the same staging."""
    d = synth.make_inputs(4100 + M, M, K, N, a_dtype=adt)
    Yd, (Bp, S, dl) = _w4a16(wq, d, out_dtype=ydt, sym=sym)
    delta = None if sym else dl
    hX = _x(d).cpu().pin_memory()
    hY = torch.empty((M, N), dtype=ydt).pin_memory()
    for scale in (2.0, 1.0):
        got = wq.gemm_w4a16_host((hX.float() * scale).to(hX.dtype).pin_memory() if scale != 1.0 else hX,
                                 Bp, S, delta, 128, out=hY)
        torch.cuda.synchronize()
    assert got.data_ptr() == hY.data_ptr() and not hY.is_cuda
    assert torch.equal(hY, Yd.cpu())
    err = oracle.rel_fro(hY.double().numpy(), _ref_w4a16(d, sym=sym))
    assert err <= TOL_W4A16, err
    # a new pinned output when none is given
    Y2 = wq.gemm_w4a16_host(hX, Bp, S, delta, 128, out_dtype=ydt)
    torch.cuda.synchronize()
    assert Y2.is_pinned() and torch.equal(Y2, Yd.cpu())


@pytest.mark.parametrize("M,K,N,adt,ydt", [
    (2500, 1024, 8192, "f16", torch.float16),    # two chunks of 1280 and 1220 rows
    (4096, 512, 4096, "bf16", torch.float32),    # four chunks of 1024 rows
])
def test_host_buffer_entry_pipelined_chunks(wq, M, K, N, adt, ydt):
    """gemm_w4a16_host with M >= 2048 runs row chunks in a pipeline (copies in and out on
    internal streams overlapping the chunk GEMMs): min(4, M / 1024) chunks of rows rounded
    up to 256.  The result equals the device entry called on the same row chunks bit for
    bit (the whole-M device call may tile its last wave differently, so it is compared
    within the large-M bar); sampled rows match the oracle; two calls in a row."""
    d = synth.make_inputs(4200 + M, M, K, N, a_dtype=adt)
    Yfull, (Bp, S, dl) = _w4a16(wq, d, out_dtype=ydt)
    X = _x(d)
    chunks = min(4, M // 1024)
    rows_c = ((M + chunks - 1) // chunks + 255) // 256 * 256
    Yd = torch.cat([wq.gemm_w4a16(X[r0:r0 + rows_c], Bp, S, dl, 128, ydt) for r0 in range(0, M, rows_c)])
    torch.cuda.synchronize()
    assert oracle.rel_fro(Yd.double().cpu().numpy(), Yfull.double().cpu().numpy()) <= TOL_LARGE_M
    hX = X.cpu().pin_memory()
    hY = torch.empty((M, N), dtype=ydt).pin_memory()
    for _ in range(2):
        hY.fill_(float("nan"))
        wq.gemm_w4a16_host(hX, Bp, S, dl, 128, out=hY)
        torch.cuda.synchronize()
        assert torch.equal(hY, Yd.cpu())
    rows = _sample_rows(M)
    cols = (N // 2 - 64, N // 2 + 64)
    ref = _ref_w4a16(d, rows=rows, cols=cols)
    assert oracle.rel_fro(hY[rows][:, cols[0]:cols[1]].double().numpy(), ref) <= TOL_W4A16


@pytest.mark.parametrize("M,K,N,gs,adt", [
    (3, 1408, 256, 128, "f16"),     # 11 k-blocks over 6 segments of 2: the last segment has one
    (2, 256, 20480, 128, "f16"),    # 160 column tiles: one segment, partials stored from registers
    (1, 2560, 19200, 128, "f16"),   # 150 tiles x 2 segments of 10 k-blocks: the 8-deep ring wraps
    (8, 2560, 19200, -1, "bf16"),   # the same with 8 tokens, one group per column, bf16
    (5, 3968, 384, 128, "bf16"),    # 31 k-blocks over 8 segments of 4 (the last 3)
])
def test_weight_streaming_decode_segments(wq, M, K, N, gs, adt):
    """Decode shapes (M <= 8) whose K segmentation exercises a ragged last segment,
    a single segment (no cluster reduction) and a code ring that wraps several
    times; compared with the oracle element by element."""
    d = synth.make_inputs(5300 + M * 13 + K, M, K, N, group_size=gs, a_dtype=adt)
    Y, _ = _w4a16(wq, d)
    ref = _ref_w4a16(d)
    got = Y.double().cpu().numpy()
    err = oracle.rel_fro(got, ref)
    assert err <= TOL_W4A16, err
    assert np.isfinite(got).all()


@pytest.mark.parametrize("M,K,N,gs,odt", [
    (1, 1024, 384, 128, torch.float16),    # M <= 8: weight-streaming kernel on the int8 rows
    (3, 1024, 256, 128, torch.bfloat16),
    (5, 2048, 256, -1, torch.float16),
    (12, 1024, 256, 128, torch.float32),   # M 9..16: e4m3 decode kernel
    (16, 1280, 256, 128, torch.bfloat16),
    (33, 768, 256, 128, torch.float16),    # large-M path (int8 -> fp16, correction columns)
    (200, 1024, 384, 128, torch.float32),
])
def test_w4a8_zero_point_parity(wq, M, K, N, gs, odt):
    """W4A8 with zero-point uint4 weights (packed by pack_w4a16, no fold): against the
    oracle over the int8 rows (2e-3) and against the fp16-activation reference (5 %)."""
    d = synth.make_inputs(6100 + M + K, M, K, N, group_size=gs)
    Xq, xs = oracle.quantize_per_token(d["A"])
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), gs)
    Y = wq.gemm_w4a8_asym(_cuda(Xq), _cuda(xs), Bp, S, dl, gs, out_dtype=odt)
    torch.cuda.synchronize()
    got = Y.double().cpu().numpy()
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    ref8 = oracle.gemm_w4a8_asym(Xq, xs, d["q"], sb, zb, gs)
    err = oracle.rel_fro(got, ref8)
    assert err <= TOL_W4A8, err
    ref16 = oracle.gemm_asym_plain(oracle.activations_to_double(d["A"], "f16"), d["q"], sb, zb, gs)
    assert oracle.rel_fro(got, ref16) <= TOL_W4A8_VS_F16


@pytest.mark.parametrize("M", [4, 40])
def test_w4a8_zero_point_without_delta_is_symmetric(wq, M):
    """delta None: the symmetric product with the scales as given, the same as the W4A8
    reference with those (positive, unfolded) scales."""
    d = synth.make_inputs(6200 + M, M, 512, 256)
    Xq, xs = oracle.quantize_per_token(d["A"])
    Bp, S, _ = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), 128)
    Y = wq.gemm_w4a8_asym(_cuda(Xq), _cuda(xs), Bp, S, None, 128)
    torch.cuda.synchronize()
    ref = oracle.gemm_w4a8(Xq, xs, d["q"], oracle.half_bits(d["scale"]), 128)
    assert oracle.rel_fro(Y.double().cpu().numpy(), ref) <= TOL_W4A8


@pytest.mark.parametrize("M,K,N", [(1, 1024, 256), (7, 2048, 384), (16, 1280, 256), (40, 768, 256), (300, 1024, 384)])
@pytest.mark.parametrize("zero_point", [False, True])
def test_w4a8_quantize_inside_equals_two_steps(wq, M, K, N, zero_point):
    """gemm_w4a8_fp16 (per-token quantization inside the activation pre-pass) gives the
    x_scale of quantize_per_token and the Y of quantize_per_token + the int8 GEMM, bit for
    bit, on every kernel path (M <= 8, M 9..16, large M); and the oracle's value within 2e-3."""
    if zero_point:
        d = synth.make_inputs(6300 + M, M, K, N)
        Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), 128)
    else:
        d = synth.make_inputs(6400 + M, M, K, N, mode="w4a8")
        Bp, S = wq.pack_w4a8(_cuda(d["q"]), _cuda(d["scale"]), 128)
        dl = None
    X = _cuda(d["A"])
    Xq, xs = wq.quantize_per_token(X)
    Y2 = wq.gemm_w4a8_asym(Xq, xs, Bp, S, dl, 128) if zero_point else wq.gemm_w4a8(Xq, xs, Bp, S, 128)
    Y1, xs1 = wq.gemm_w4a8_fp16(X, Bp, S, dl, 128)
    torch.cuda.synchronize()
    assert torch.equal(xs1, xs)
    assert torch.equal(Y1, Y2)
    Xq_o, xs_o = oracle.quantize_per_token(d["A"])
    if zero_point:
        ref = oracle.gemm_w4a8_asym(Xq_o, xs_o, d["q"], oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"]), 128)
    else:
        qf, sfb = oracle.fold(d["q"], oracle.half_bits(d["scale"]), 128)
        ref = oracle.gemm_w4a8(Xq_o, xs_o, qf, sfb, 128)
    assert oracle.rel_fro(Y1.double().cpu().numpy(), ref) <= TOL_W4A8


def _moe_inputs(seed, E, K, N, counts, gs=128, adt="f16", sym=False):
    rng = np.random.default_rng(seed)
    offs = [0] + list(np.cumsum(counts))
    M = int(offs[-1])
    a = rng.standard_normal((M, K))
    if adt == "bf16":
        A = oracle.double_to_bf16(a)  # bits
        X = _cuda(A.view(np.int16)).view(torch.bfloat16)
        A64 = oracle.bf16_to_double(A)
    else:
        A = a.astype(np.float16)
        X = _cuda(A)
        A64 = A.astype(np.float64)
    G = K // (K if gs == -1 else gs)
    q = rng.integers(0, 16, size=(E, K, N)).astype(np.uint8)
    s = rng.uniform(0.005, 0.02, size=(E, G, N)).astype(np.float16)
    z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
    return offs, X, A64, q, s, z


@pytest.mark.parametrize("E,K,N,counts,gs,adt,sym", [
    (8, 256, 7168, (3, 1, 0, 4, 2, 2, 3, 1), 128, "f16", False),   # 16 tokens over 8 experts
    (8, 256, 7168, (2, 2, 2, 2, 2, 2, 2, 2), 128, "bf16", True),
    (4, 1024, 512, (1, 8, 0, 5), -1, "f16", False),                  # per-channel groups
    (3, 512, 384, (12, 0, 40), 128, "f16", False),                   # > 8 tokens: one GEMM per expert
])
def test_grouped_moe_parity(wq, E, K, N, counts, gs, adt, sym):
    """Mixture-of-experts W4A16 against the oracle (each expert's rows times its own
    weights), element by element within 2e-3."""
    offs, X, A64, q, s, z = _moe_inputs(7000 + E + K, E, K, N, counts, gs, adt, sym)
    packs = [wq.pack_w4a16(_cuda(q[e]), _cuda(s[e]), _cuda(z[e]), gs) for e in range(E)]
    Bp = torch.stack([p_[0] for p_ in packs])
    S = torch.stack([p_[1] for p_ in packs])
    dl = None if sym else torch.stack([p_[2] for p_ in packs])
    Y = wq.gemm_w4a16_grouped(X, Bp, S, dl, offs, gs)
    torch.cuda.synchronize()
    sb, zb = oracle.half_bits(s), oracle.half_bits(z)
    ref = oracle.gemm_grouped_asym(A64, offs, q, sb, None if sym else zb, gs)
    err = oracle.rel_fro(Y.double().cpu().numpy(), ref)
    assert err <= TOL_W4A16, err
    # each expert's rows equal that expert's plain GEMM through the single-problem entry
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            Ye = wq.gemm_w4a16(X[r0:r1].contiguous(), Bp[e], S[e], None if sym else dl[e], gs)
            torch.cuda.synchronize()
            assert oracle.rel_fro(Y[r0:r1].double().cpu().numpy(), Ye.double().cpu().numpy()) <= 1e-3


@pytest.mark.parametrize("E,K,N,counts,zero_point", [
    (8, 256, 7168, (3, 1, 0, 4, 2, 2, 3, 1), False),   # the article's case: 16 tokens over 8 experts
    (8, 256, 7168, (2, 2, 2, 2, 2, 2, 2, 2), True),
    (3, 512, 384, (20, 0, 33), True),                   # large-M kernel per expert
    (2, 1024, 256, (0, 5), False),
])
def test_grouped_w4a8_parity(wq, E, K, N, counts, zero_point):
    """Mixture-of-experts W4A8 (folded symmetric or zero-point weights) against the oracle
    within 2e-3; each expert's rows equal that expert's single-problem W4A8 call bit for bit."""
    rng = np.random.default_rng(7100 + E + K)
    offs = [0] + [int(v) for v in np.cumsum(counts)]
    M = offs[-1]
    x = rng.standard_normal((M, K)).astype(np.float16)
    Xq_o, xs_o = oracle.quantize_per_token(x)
    q = rng.integers(0, 16, size=(E, K, N)).astype(np.uint8)
    s = rng.uniform(0.005, 0.02, size=(E, K // 128, N)).astype(np.float16)
    if zero_point:
        z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
        packs = [wq.pack_w4a16(_cuda(q[e]), _cuda(s[e]), _cuda(z[e]), 128) for e in range(E)]
        dl = torch.stack([p_[2] for p_ in packs])
        ref = oracle.gemm_grouped_w4a8(Xq_o, xs_o, offs, q, oracle.half_bits(s), oracle.half_bits(z), 128)
    else:
        s = np.where(rng.random(s.shape) < 0.5, -s, s).astype(np.float16)  # signed scales, folded at pack
        packs = [wq.pack_w4a8(_cuda(q[e]), _cuda(s[e]), 128) for e in range(E)]
        dl = None
        folded = [oracle.fold(q[e], oracle.half_bits(s[e]), 128) for e in range(E)]
        qf = np.stack([f[0] for f in folded])
        sf = np.stack([f[1] for f in folded])
        ref = oracle.gemm_grouped_w4a8(Xq_o, xs_o, offs, qf, sf, None, 128)
    Bp = torch.stack([p_[0] for p_ in packs])
    S = torch.stack([p_[1] for p_ in packs])
    Xq, xs = _cuda(Xq_o), _cuda(xs_o)
    Y = wq.gemm_w4a8_grouped(Xq, xs, Bp, S, dl, offs, 128)
    torch.cuda.synchronize()
    err = oracle.rel_fro(Y.double().cpu().numpy(), ref)
    assert err <= TOL_W4A8, err
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            Xe, xse = Xq[r0:r1].contiguous(), xs[r0:r1].contiguous()
            if zero_point:
                Ye = wq.gemm_w4a8_asym(Xe, xse, Bp[e], S[e], dl[e], 128)
            else:
                Ye = wq.gemm_w4a8(Xe, xse, Bp[e], S[e], 128)
            torch.cuda.synchronize()
            assert torch.equal(Y[r0:r1], Ye)


@pytest.mark.parametrize("idx", range(len(synth.shapes("c4"))))
def test_w4a8_zero_point_and_in_call_quantization_full_size_sampled(wq, idx):
    """The c4 shapes (M 16 / 256 / 2048, K 5120, N 17408) with zero-point weights, through
    the in-call quantization entry, on sampled rows and column windows against the oracle;
    the int8 codes and scales equal the stand-alone quantizer's."""
    seed, s = synth.shapes("c4")[idx]
    d = synth.make_inputs(seed + 900, s["M"], s["K"], s["N"])  # w4a16 recipe: scale + zero point
    X = _cuda(d["A"])
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), 128)
    Y, xs = wq.gemm_w4a8_fp16(X, Bp, S, dl, 128)
    torch.cuda.synchronize()
    Xq_o, xs_o = oracle.quantize_per_token(d["A"])
    assert np.array_equal(xs.cpu().numpy(), xs_o)
    rows = _sample_rows(s["M"])
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    for c in _sample_cols(s["N"]):
        ref = oracle.gemm_w4a8_asym(Xq_o[rows], xs_o[rows], d["q"], sb, zb, 128, cols=c)
        got = Y[rows][:, c[0]:c[1]].double().cpu().numpy()
        assert oracle.rel_fro(got, ref) <= TOL_W4A8, c


@pytest.mark.parametrize("M,K,N,gs,adt", [(3, 1024, 256, -1, "bf16"), (8, 768, 384, 128, "bf16"),
                                          (5, 2048, 256, -1, "f16")])
def test_decode_offset_codes_symmetric(wq, M, K, N, gs, adt):
    """Symmetric weights (no correction) on the M <= 8 decode path: the offset the codes
    carry is removed per block even without delta; fp16 and bf16, one group per column."""
    d = synth.make_inputs(7300 + M + K, M, K, N, group_size=gs, a_dtype=adt)
    Y, _ = _w4a16(wq, d, sym=True)
    ref = _ref_w4a16(d, sym=True)
    assert oracle.rel_fro(Y.double().cpu().numpy(), ref) <= TOL_W4A16


# --------------------------------------------------------------------------- SwiGLU gate/up pair

def _pair_inputs(seed, M, K, N, gs=128, adt="f16", zero_point=True):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K))
    if adt == "bf16":
        A = oracle.double_to_bf16(a)
        X = _cuda(A.view(np.int16)).view(torch.bfloat16)
        A64 = oracle.bf16_to_double(A)
    else:
        A = a.astype(np.float16)
        X = _cuda(A)
        A64 = A.astype(np.float64)
    G = K // (K if gs == -1 else gs)
    ws = []
    for _ in range(2):
        q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
        s = rng.uniform(0.005, 0.02, size=(G, N)).astype(np.float16)
        z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
        ws.append((q, s, z))
    return X, A64, ws


def _swiglu_tol(A64, gate, up, gs):
    """The GEMM bar (2e-3 relative Frobenius on each of G and U) carried to first order
    through Y = silu(G) * U: dY = silu'(G) U dG + silu(G) dU, with each product's error
    spread evenly over its elements (|dG| ~ 2e-3 rms(G), |dU| ~ 2e-3 rms(U), independent).
    On these inputs the factor over the GEMM bar is about 1.45 to 1.55."""
    def product(w):
        q, sb, zb = w
        return (oracle.gemm_asym_identity(A64, q, sb, None, gs) if zb is None
                else oracle.gemm_asym_plain(A64, q, sb, zb, gs))
    G, U = product(gate), product(up)
    sig = 1.0 / (1.0 + np.exp(-np.clip(G, -700, 700)))
    silu, dsilu = G * sig, sig * (1.0 + G * (1.0 - sig))
    rg, ru = np.sqrt(np.mean(G ** 2)), np.sqrt(np.mean(U ** 2))
    amp = np.sqrt((np.sum((dsilu * U) ** 2) * rg ** 2 + np.sum(silu ** 2) * ru ** 2) / np.sum((silu * U) ** 2))
    return TOL_W4A16 * amp


def test_pair_pack_is_the_interleaved_pack(wq):
    """pack_w4a16_pair: codes, scales and deltas of the gate/up pair in the interleaved
    column order, bit for bit (unpack of the packed words, S, delta)."""
    K, N = 256, 192
    _, _, ((qg, sg, zg), (qu, su, zu)) = _pair_inputs(7200, 1, K, N)
    Bp, S, dl = wq.pack_w4a16_pair(_cuda(qg), _cuda(sg), _cuda(zg), _cuda(qu), _cuda(su), _cuda(zu), 128)
    q2 = wq.unpack_w4(Bp, K, 2 * N)
    torch.cuda.synchronize()
    assert np.array_equal(q2.cpu().numpy(), oracle.pair_interleave(qg, qu))
    assert np.array_equal(oracle.half_bits(S.cpu().numpy()),
                          oracle.pair_interleave(oracle.half_bits(sg), oracle.half_bits(su)))
    dg = oracle.delta(oracle.half_bits(sg), oracle.half_bits(zg))
    du = oracle.delta(oracle.half_bits(su), oracle.half_bits(zu))
    assert np.array_equal(dl.cpu().numpy(), oracle.pair_interleave(dg, du))


@pytest.mark.parametrize("M,K,N,gs,adt,zero_point", [
    (1, 128, 192, 128, "f16", True),      # one k-block: no split, SwiGLU in registers
    (3, 1024, 64, 128, "f16", True),      # one column tile, 8 K segments
    (8, 1536, 5504, 128, "f16", True),    # 3 K segments: ownership rounded to 16 rows
    (5, 1280, 3328, 128, "bf16", True),   # 5 K segments, the last owning no rows
    (4, 2048, 320, -1, "f16", False),     # per-channel, symmetric
    (12, 1024, 192, 128, "f16", True),    # M 9..16: tcgen05 decode kernel, then the activation pass
    (40, 768, 320, 128, "bf16", True),    # large M
])
def test_swiglu_pair_parity(wq, M, K, N, gs, adt, zero_point):
    """silu(X @ W_gate) * (X @ W_up) against the oracle, element by element within 2e-3."""
    X, A64, ((qg, sg, zg), (qu, su, zu)) = _pair_inputs(7300 + M + K, M, K, N, gs, adt)
    Bp, S, dl = wq.pack_w4a16_pair(_cuda(qg), _cuda(sg), _cuda(zg), _cuda(qu), _cuda(su), _cuda(zu), gs)
    Y = wq.gemm_w4a16_swiglu(X, Bp, S, dl if zero_point else None, gs)
    torch.cuda.synchronize()
    gate = (qg, oracle.half_bits(sg), oracle.half_bits(zg) if zero_point else None)
    up = (qu, oracle.half_bits(su), oracle.half_bits(zu) if zero_point else None)
    ref = oracle.gemm_swiglu_pair(A64, gate, up, gs)
    assert Y.shape == (M, N)
    err = oracle.rel_fro(Y.double().cpu().numpy(), ref)
    assert err <= _swiglu_tol(A64, gate, up, gs), err
    if M > 16:  # large M: fp16 weights for either activation type, inside the plain GEMM bar
        assert err <= TOL_W4A16, err


def test_swiglu_pair_fp32_output_and_workspace_query(wq):
    """fp32 output (no final rounding) within 1e-4 of the oracle on the fused path (the
    offset codes remove a term of ~1032 times the block sum of x from each block's fp32
    product, which costs about 8 of fp32's 24 bits: ~3e-5 relative, measured 2.9e-5); the
    workspace query is 0 for the fused path and covers the fp32 pair product otherwise."""
    M, K, N = 2, 1024, 256
    X, A64, ((qg, sg, zg), (qu, su, zu)) = _pair_inputs(7400, M, K, N)
    Bp, S, dl = wq.pack_w4a16_pair(_cuda(qg), _cuda(sg), _cuda(zg), _cuda(qu), _cuda(su), _cuda(zu), 128)
    Y = wq.gemm_w4a16_swiglu(X, Bp, S, dl, 128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.gemm_swiglu_pair(A64, (qg, oracle.half_bits(sg), oracle.half_bits(zg)),
                                  (qu, oracle.half_bits(su), oracle.half_bits(zu)), 128)
    assert oracle.rel_fro(Y.double().cpu().numpy(), ref) <= 1e-4
    assert wq.workspace_size(wq.VARIANT_W4A16_SWIGLU, M, N, K, 128) == 0
    assert wq.workspace_size(wq.VARIANT_W4A16_SWIGLU, 40, N, K, 128) >= 40 * 2 * N * 4


def test_every_entry_family_replays_in_a_cuda_graph(wq):
    """Large-M W4A16, in-call-quantized W4A8 (decode and large M), the SwiGLU pair (fused and
    through the fp32 product) and both grouped entries, captured into one CUDA graph with
    caller workspaces and replayed: each result equals its eager call bit for bit (no entry
    allocates or synchronises inside the capture)."""
    K, N = 1024, 256
    d = synth.make_inputs(7500, 64, K, N)
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), 128)
    X = _cuda(d["A"])
    _, _, ((qg, sg, zg), (qu, su, zu)) = _pair_inputs(7501, 1, K, N // 2)
    Bp2, S2, dl2 = wq.pack_w4a16_pair(_cuda(qg), _cuda(sg), _cuda(zg), _cuda(qu), _cuda(su), _cuda(zu), 128)
    Bg, Sg, dg = Bp.unsqueeze(0).repeat(2, 1, 1, 1, 1), S.unsqueeze(0).repeat(2, 1, 1), dl.unsqueeze(0).repeat(2, 1, 1)
    offs = [0, 3, 7]
    Xq, xs = wq.quantize_per_token(X[:7].contiguous())
    ws_bytes = max(wq.workspace_size(v, 64, N, K, 128) for v in (wq.VARIANT_W4A16, wq.VARIANT_W4A8_ASYM))
    ws_bytes = max(ws_bytes, wq.workspace_size(wq.VARIANT_W4A16_SWIGLU, 40, N // 2, K, 128))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    calls = [
        lambda o: wq.gemm_w4a16(X, Bp, S, dl, 128, out=o, workspace=ws),
        lambda o: wq.gemm_w4a8_fp16(X[:5].contiguous(), Bp, S, dl, 128, out=o, workspace=ws)[0],
        lambda o: wq.gemm_w4a8_fp16(X[:40].contiguous(), Bp, S, dl, 128, out=o, workspace=ws)[0],
        lambda o: wq.gemm_w4a16_swiglu(X[:4].contiguous(), Bp2, S2, dl2, 128, out=o, workspace=ws),
        lambda o: wq.gemm_w4a16_swiglu(X[:40].contiguous(), Bp2, S2, dl2, 128, out=o, workspace=ws),
        lambda o: wq.gemm_w4a16_grouped(X[:7].contiguous(), Bg, Sg, dg, offs, 128, out=o, workspace=ws),
        lambda o: wq.gemm_w4a8_grouped(Xq, xs, Bg, Sg, dg, offs, 128, out=o, workspace=ws),
    ]
    shapes = [(64, N), (5, N), (40, N), (4, N // 2), (40, N // 2), (7, N), (7, N)]
    eager = []
    for f, sh in zip(calls, shapes):
        o = torch.empty(sh, dtype=torch.float16, device="cuda")
        f(o)
        torch.cuda.synchronize()
        eager.append(o.clone())
    outs = [torch.empty(sh, dtype=torch.float16, device="cuda") for sh in shapes]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for f, o in zip(calls, outs):
                f(o)
        for _ in range(2):
            for o in outs:
                o.zero_()
            g.replay()
    torch.cuda.synchronize()
    for i, (o, e) in enumerate(zip(outs, eager)):
        assert torch.equal(o, e), i
    # ... and the replayed results against the oracle at each family's bar
    A64 = d["A"].astype(np.float64)
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    W = (d["q"], sb, zb)
    _, A64p, (gate, up) = _pair_inputs(7501, 1, K, N // 2)
    hb = oracle.half_bits
    gate, up = (gate[0], hb(gate[1]), hb(gate[2])), (up[0], hb(up[1]), hb(up[2]))
    Xp = X.double().cpu().numpy()
    refs = [oracle.gemm_asym_plain(A64, *W, 128)]
    for m in (5, 40):
        oXq, oxs = oracle.quantize_per_token(d["A"][:m])
        refs.append(oracle.gemm_w4a8_asym(oXq, oxs, *W, 128))
    refs += [oracle.gemm_swiglu_pair(Xp[:m], gate, up, 128) for m in (4, 40)]
    refs.append(oracle.gemm_asym_plain(A64[:7], *W, 128))  # both experts hold the same weights
    oXq, oxs = oracle.quantize_per_token(d["A"][:7])
    assert np.array_equal(Xq.cpu().numpy(), oXq) and np.array_equal(xs.cpu().numpy(), oxs)
    refs.append(oracle.gemm_w4a8_asym(oXq, oxs, *W, 128))
    tols = [TOL_W4A16, TOL_W4A8, TOL_W4A8, _swiglu_tol(Xp[:4], gate, up, 128),
            _swiglu_tol(Xp[:40], gate, up, 128), TOL_W4A16, TOL_W4A8]
    for i, (o, r, tol) in enumerate(zip(outs, refs, tols)):
        err = oracle.rel_fro(o.double().cpu().numpy(), r)
        assert err <= tol, (i, err, tol)


def test_swiglu_pair_bench_size_sampled(wq):
    """The bench's SwiGLU workload (M 1 and 4, K 4096, two N = 11008 projections), in the
    bench's launch configuration (one launch of the pair instance), on sampled output
    columns against the oracle on the same gate and up columns."""
    d = synth.swiglu_inputs()
    g, u = d["gate"], d["up"]
    Bp, S, dl = wq.pack_w4a16_pair(_cuda(g["q"]), _cuda(g["scale"]), _cuda(g["zero"]),
                                   _cuda(u["q"]), _cuda(u["scale"]), _cuda(u["zero"]), 128)
    N = g["q"].shape[1]
    hb = oracle.half_bits
    for A in d["A"]:
        Y = wq.gemm_w4a16_swiglu(_cuda(A), Bp, S, dl, 128)
        torch.cuda.synchronize()
        A64 = A.astype(np.float64)
        for c0, c1 in _sample_cols(N):
            gate = (np.ascontiguousarray(g["q"][:, c0:c1]), hb(g["scale"][:, c0:c1]), hb(g["zero"][:, c0:c1]))
            up = (np.ascontiguousarray(u["q"][:, c0:c1]), hb(u["scale"][:, c0:c1]), hb(u["zero"][:, c0:c1]))
            ref = oracle.gemm_swiglu_pair(A64, gate, up, 128)
            err = oracle.rel_fro(Y[:, c0:c1].double().cpu().numpy(), ref)
            assert err <= _swiglu_tol(A64, gate, up, 128), (c0, err)
