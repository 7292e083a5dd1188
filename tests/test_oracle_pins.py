"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks one oracle function against a closed form, a library
routine, brute force on tiny inputs, or values the pages print (fixtures
under tests/golden/, each with its citation).  The mutation tests at the end
plant known mistakes in the oracle and check that some pin catches each one.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def _rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------- formats

def test_half_rounding_matches_numpy():
    """Oracle binary16 RNE == numpy's float64->float16 cast (a library routine)."""
    rng = _rng(1)
    parts = [
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24,
                  2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, np.inf, -np.inf]),
    ]
    # exact ties between neighbouring binary16 values
    h = rng.integers(0, 0x7BFF, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    parts.append((lo + hi) / 2)
    x = np.concatenate(parts)
    got = oracle.double_to_half(x)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_half_decode_matches_numpy():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7C00) != 0x7C00
    got = oracle.half_to_double(bits[finite][::7])
    want = bits[finite][::7].view(np.float16).astype(np.float64)
    assert np.array_equal(got, want)


def test_bf16_rounding_matches_torch():
    """Oracle bfloat16 RNE == torch's float32->bfloat16 cast on fp32-exact inputs."""
    rng = _rng(2)
    x32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 2.0 ** -130, 3.0e38], np.float32)
    x32 = np.concatenate([x32, ties])
    got = oracle.double_to_bf16(x32.astype(np.float64))
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    back = oracle.bf16_to_double(got[:500])
    want_back = torch.from_numpy(want[:500].view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(back, want_back)


# --------------------------------------------------------------------------- pack layout

def _word_position(n, w, K):
    """The blocked layout's word position, written out independently of the oracle:
    8 KB blocks of 128 columns x 128 k, row r = n % 128 holds 16 words as four
    16-byte chunks, chunk c stored at slot c ^ ((r // 2) % 4)."""
    block = (n // 128) * (K // 128) + (8 * w) // 128
    r, u = n % 128, w % 16
    c, e = u // 4, u % 4
    return block * 2048 + r * 16 + 4 * (c ^ ((r // 2) % 4)) + e


def test_pack_golden_words():
    """Each golden line: the 8 codes of column 0, k = 0..7 -> their word (the first word)."""
    for row in _golden_rows("pack_layout.txt"):
        codes, word = row.split("->")
        codes = [int(c) for c in codes.split()]
        q = np.zeros((128, 128), np.uint8)
        q[:8, 0] = codes
        assert int(oracle.pack(q).reshape(-1)[_word_position(0, 0, 128)]) == int(word, 16), row


def test_pack_unpack_roundtrip_exhaustive():
    """Every code 0..15 at every nibble position, several column tiles, round trip."""
    K, N = 16 * 8, 256
    q = np.zeros((K, N), np.uint8)
    for k in range(K):
        for n in range(N):
            q[k, n] = (k // 8 + 3 * n + (k % 8)) % 16
    w = oracle.pack(q)
    assert w.shape == (N // 128, K // 128, 128, 16)
    assert np.array_equal(oracle.unpack(w, K, N), q)
    rng = _rng(3)
    q2 = rng.integers(0, 16, (384, 256), dtype=np.uint8)
    assert np.array_equal(oracle.unpack(oracle.pack(q2), 384, 256), q2)


def test_pack_matches_bitwise_definition():
    """Pack == the layout rule written with numpy shifts and the position formula (brute force)."""
    rng = _rng(4)
    K, N = 256, 256
    q = rng.integers(0, 16, (K, N), dtype=np.uint8)
    w = oracle.pack(q).reshape(-1)
    for n in list(range(0, N, 7)) + [1, 2, 3, 127, 128, 255]:
        for kw in range(K // 8):
            word = 0
            for j in range(8):
                word |= int(q[8 * kw + j, n]) << (4 * (j // 2) + 16 * (j % 2))
            assert int(w[_word_position(n, kw, K)]) == word


def test_pack_positions_are_a_permutation():
    """Every (column, word) pair lands on a distinct slot (the layout is a bijection)."""
    K, N = 384, 256
    pos = {_word_position(n, w, K) for n in range(N) for w in range(K // 8)}
    assert len(pos) == N * K // 8 and min(pos) == 0 and max(pos) == N * K // 8 - 1


# --------------------------------------------------------------------------- delta

def test_delta_golden_example():
    s = np.array([[0.5]], np.float16)
    z = np.array([[-3.0]], np.float16)
    d = oracle.delta(oracle.half_bits(s), oracle.half_bits(z))
    for row in _golden_rows("delta_example.txt"):
        qv, wsym, wasym, dv = (float(t) for t in row.split())
        assert d[0, 0] == dv
        A = np.zeros((1, 128))
        A[0, 0] = 1.0
        q = np.full((128, 1), 8, np.uint8)
        q[0, 0] = int(qv)
        c_sym = oracle.gemm_asym_identity(A, q, oracle.half_bits(s), None, 128)
        c_asym = oracle.gemm_asym_plain(A, q, oracle.half_bits(s), oracle.half_bits(z), 128)
        assert c_sym[0, 0] == wsym
        assert c_asym[0, 0] == wasym


def test_delta_is_exact_fp32_of_sum():
    """delta == float32(zero + 8*scale) where the sum is formed exactly (Fraction)."""
    from fractions import Fraction
    d = synth.make_inputs(5, 1, 256, 64)
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    got = oracle.delta(sb, zb)
    s64 = d["scale"].astype(np.float64)
    z64 = d["zero"].astype(np.float64)
    for i in range(0, got.size, 13):
        exact = Fraction(float(z64.flat[i])) + 8 * Fraction(float(s64.flat[i]))
        assert np.float32(float(exact)) == got.flat[i]


# --------------------------------------------------------------------------- GEMM definitions

def _tiny_problem(seed, M, K, N, gs):
    d = synth.make_inputs(seed, M, K, N, group_size=gs)
    A = oracle.activations_to_double(d["A"], "f16")
    return d, A, oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])


@pytest.mark.parametrize("M,K,N,gs", [(1, 128, 8, 128), (3, 256, 16, 128), (5, 384, 24, 128),
                                      (2, 256, 8, -1), (4, 1024, 8, 128)])
def test_identity_equals_plain_definition(M, K, N, gs):
    """C_asym (plain) == C_sym + A_group_sum @ delta, brute force in fp64 (<= 1e-12)."""
    d, A, sb, zb = _tiny_problem(11 + M, M, K, N, gs)
    plain = oracle.gemm_asym_plain(A, d["q"], sb, zb, gs)
    ident = oracle.gemm_asym_identity(A, d["q"], sb, zb, gs)
    assert np.max(np.abs(plain - ident)) <= 1e-12 * np.max(np.abs(plain))


def test_plain_matches_library_matmul():
    """Plain definition == numpy float64 matmul of the dequantized asymmetric weights."""
    M, K, N, gs = 6, 512, 32, 128
    d, A, sb, zb = _tiny_problem(21, M, K, N, gs)
    g = np.arange(K) // gs
    W = (d["q"].astype(np.float64) * d["scale"].astype(np.float64)[g]
         + d["zero"].astype(np.float64)[g])
    ref = A @ W
    got = oracle.gemm_asym_plain(A, d["q"], sb, zb, gs)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-12)


def test_column_window_matches_full():
    M, K, N, gs = 3, 256, 40, 128
    d, A, sb, zb = _tiny_problem(22, M, K, N, gs)
    full = oracle.gemm_asym_plain(A, d["q"], sb, zb, gs)
    part = oracle.gemm_asym_plain(A, d["q"], sb, zb, gs, cols=(7, 29))
    assert np.array_equal(full[:, 7:29], part)


def test_integer_special_case_exact():
    """scale = 1, zero = -8  =>  W = q - 8 and delta = 0: C is an integer matmul."""
    rng = _rng(7)
    M, K, N, gs = 4, 256, 16, 128
    q = rng.integers(0, 16, (K, N), dtype=np.uint8)
    A = rng.integers(-3, 4, (M, K)).astype(np.float64)
    s = np.ones((K // gs, N), np.float16)
    z = np.full((K // gs, N), -8.0, np.float16)
    want = (A.astype(np.int64) @ (q.astype(np.int64) - 8)).astype(np.float64)
    got = oracle.gemm_asym_plain(A, q, oracle.half_bits(s), oracle.half_bits(z), gs)
    got2 = oracle.gemm_asym_identity(A, q, oracle.half_bits(s), oracle.half_bits(z), gs)
    assert np.array_equal(got, want) and np.array_equal(got2, want)
    assert np.all(oracle.delta(oracle.half_bits(s), oracle.half_bits(z)) == 0)


def test_zero_weights_give_zero():
    """q == 8 and zero = -8*scale  =>  W == 0 exactly, so C == 0 (tests the correction sign)."""
    d, A, sb, _ = _tiny_problem(8, 3, 256, 16, 128)
    q = np.full_like(d["q"], 8)
    z = (-8.0 * d["scale"].astype(np.float64)).astype(np.float16)
    zb = oracle.half_bits(z)
    assert np.all(oracle.gemm_asym_plain(A, q, sb, zb, 128) == 0)
    assert np.max(np.abs(oracle.gemm_asym_identity(A, q, sb, zb, 128))) == 0


def test_per_channel_closed_form():
    """One group per column: C = s[n] * (A @ (q - 8)) + rowsum(A) * delta[n]."""
    d, A, sb, zb = _tiny_problem(9, 3, 512, 12, -1)
    s = d["scale"].astype(np.float64)[0]
    z = d["zero"].astype(np.float64)[0]
    want = s * (A @ (d["q"].astype(np.float64) - 8)) + A.sum(1, keepdims=True) * (z + 8 * s)
    got = oracle.gemm_asym_plain(A, d["q"], sb, zb, -1)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_group_sum_matches_numpy():
    d, A, _, _ = _tiny_problem(10, 5, 640, 8, 128)
    got = oracle.group_sum(A, 128)
    want = A.reshape(5, 5, 128).sum(-1)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-13)


# --------------------------------------------------------------------------- dequant spec

def test_dequant_f16_matches_numpy_cast():
    """fp16_RN((q-8)*s): the product is exact in fp64, numpy's cast rounds it once."""
    d = synth.make_inputs(12, 1, 512, 64)
    w = oracle.dequant_sym_f16(d["q"], oracle.half_bits(d["scale"]), 128)
    g = np.arange(512) // 128
    exact = (d["q"].astype(np.float64) - 8) * d["scale"].astype(np.float64)[g]
    assert np.array_equal(w, exact.astype(np.float16).view(np.uint16))


def test_dequant_bf16_matches_torch_cast():
    d = synth.make_inputs(13, 1, 512, 64)
    w = oracle.dequant_sym_bf16(d["q"], oracle.half_bits(d["scale"]), 128)
    g = np.arange(512) // 128
    exact = ((d["q"].astype(np.float64) - 8) * d["scale"].astype(np.float64)[g]).astype(np.float32)
    want = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(w, want)


# --------------------------------------------------------------------------- fold

def test_fold_golden_table():
    K, N = 128, 16
    q = np.repeat(np.arange(16, dtype=np.uint8)[:, None], N, 1)
    q = np.tile(q, (K // 16, 1))
    s = np.full((1, N), -1.0, np.float16)
    qf, sf = oracle.fold(q, oracle.half_bits(s), 128)
    assert np.all(sf == oracle.half_bits(np.ones((1, N), np.float16)))
    table = {}
    for row in _golden_rows("fold_table.txt"):
        v, vf, val, valf = (int(t) for t in row.split())
        table[v] = (vf, val, valf)
    for k in range(16):
        v = int(q[k, 0])
        vf, val, valf = table[v]
        assert int(qf[k, 0]) == vf
        assert (v - 8) * -1 == val and (int(qf[k, 0]) - 8) == valf


def test_fold_equivalence_except_minus8():
    """Folded dequant == original for every code except v=0 in a negative group,
    which differs by exactly |s|; groups with a positive scale are untouched."""
    d = synth.make_inputs(14, 1, 512, 48, mode="w4a8")
    sb = oracle.half_bits(d["scale"])
    qf, sfb = oracle.fold(d["q"], sb, 128)
    g = np.arange(512) // 128
    s = d["scale"].astype(np.float64)[g]
    sf = sfb.view(np.float16).astype(np.float64)[g]
    w = (d["q"].astype(np.float64) - 8) * s
    wf = (qf.astype(np.float64) - 8) * sf
    neg = s < 0
    assert np.all(sf >= 0)
    assert np.array_equal(qf[~neg], d["q"][~neg])
    keep = ~(neg & (d["q"] == 0))
    assert np.array_equal(w[keep], wf[keep])
    bad = neg & (d["q"] == 0)
    assert bad.any()
    assert np.array_equal(w[bad] - wf[bad], np.abs(s[bad]))


# --------------------------------------------------------------------------- W4A8

def test_w4a8_matches_integer_closed_form():
    """C = x_scale[m] * sum_g s[g,n] * (Xq_g @ (q_g - 8)), with exact int64 partials."""
    d = synth.make_inputs(15, 3, 384, 16, mode="w4a8")
    Xq, xs = oracle.quantize_per_token(d["A"])
    qf, sfb = oracle.fold(d["q"], oracle.half_bits(d["scale"]), 128)
    sf = sfb.view(np.float16).astype(np.float64)
    want = np.zeros((3, 16))
    for g in range(3):
        part = Xq[:, 128 * g:128 * (g + 1)].astype(np.int64) @ (
            qf[128 * g:128 * (g + 1)].astype(np.int64) - 8)
        want += part.astype(np.float64) * sf[g]
    want *= xs.astype(np.float64)[:, None]
    got = oracle.gemm_w4a8(Xq, xs, qf, sfb, 128)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)


def test_quantize_per_token_properties():
    rng = _rng(16)
    x = rng.standard_normal((6, 512)).astype(np.float16)
    x[3] = 0
    Xq, xs = oracle.quantize_per_token(x)
    amax = np.abs(x.astype(np.float64)).max(1)
    assert np.array_equal(xs, (amax / 127.0).astype(np.float32))
    assert Xq.min() >= -127 and Xq.max() <= 127
    assert np.all(Xq[3] == 0) and xs[3] == 0
    for m in (0, 1, 2, 4, 5):
        i = np.argmax(np.abs(x[m].astype(np.float64)))
        assert abs(int(Xq[m, i])) == 127
    # ties round half to even: amax = 127 -> x_scale = 1, x = k + 0.5
    t = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.25, -2.75]], np.float16)
    tq, ts = oracle.quantize_per_token(t)
    assert ts[0] == 1.0
    assert tq.tolist() == [[127, 0, 2, 2, 0, -2, 3, -3]]


def test_error_magnitudes_match_printed_numbers():
    """The pages print 0.26 % (bf16 W4A16) and 0.9-1.05 % (W4A8 int8 activations) relative
    error on random int4 g128 weights at the model shapes.  The oracle's roundings, run on a
    slice of the same recipe (K = 5120), reproduce both magnitudes."""
    vals = dict(r.split() for r in _golden_rows("page_numbers.txt"))
    M, K, N = 8, 5120, 256
    # bf16 activations, bf16 dequantized weights, bf16 output (the W4A16 path on the page)
    d = synth.make_inputs(17, M, K, N, a_dtype="bf16")
    A = oracle.activations_to_double(d["A"], "bf16")
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    ref = oracle.gemm_asym_plain(A, d["q"], sb, zb, 128)
    wbits = oracle.dequant_sym_bf16(d["q"], sb, 128)
    wbf = (wbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dl = oracle.delta(sb, zb).astype(np.float64)
    c = A @ wbf + oracle.group_sum(A, 128) @ dl
    cb = (oracle.double_to_bf16(c).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    e16 = oracle.rel_fro(cb, ref)
    assert 0.5 * float(vals["w4a16_bf16_rel_err"]) < e16 < 1.6 * float(vals["w4a16_bf16_rel_err"])
    # W4A8: int8 per-token activations vs the fp16-activation reference, same folded weights
    d8 = synth.make_inputs(18, M, K, N, mode="w4a8")
    qf, sfb = oracle.fold(d8["q"], oracle.half_bits(d8["scale"]), 128)
    Xq, xs = oracle.quantize_per_token(d8["A"])
    c8 = oracle.gemm_w4a8(Xq, xs, qf, sfb, 128)
    A16 = oracle.activations_to_double(d8["A"], "f16")
    c16 = oracle.gemm_asym_identity(A16, qf, sfb, None, 128)
    e8 = oracle.rel_fro(c8, c16)
    assert 0.6 * float(vals["w4a8_rel_err_low"]) < e8 < 1.5 * float(vals["w4a8_rel_err_high"])
    assert e8 < float(vals["w4a8_acceptance"])


# --------------------------------------------------------------------------- W4A8, zero-point weights

def test_w4a8_asym_integer_closed_form():
    """Unit scales and integer zero points make every weight the integer q + z, so C is
    x_scale[m] times an exact int64 matmul (a textbook integer product)."""
    rng = _rng(40)
    M, K, N = 3, 384, 24
    Xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    xs = rng.uniform(0.01, 0.05, size=M).astype(np.float32)
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    G = K // 128
    zi = rng.integers(-12, 5, size=(G, N))
    sb = oracle.half_bits(np.ones((G, N), np.float16))
    zb = oracle.half_bits(zi.astype(np.float16))
    W = q.astype(np.int64) + np.repeat(zi, 128, axis=0)
    want = (Xq.astype(np.int64) @ W).astype(np.float64) * xs.astype(np.float64)[:, None]
    got = oracle.gemm_w4a8_asym(Xq, xs, q, sb, zb, 128)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("gs", [128, -1])
def test_w4a8_asym_equals_identity_form_on_int8_rows(gs):
    """x_scale * (Xq @ W_sym + group_sum(Xq) @ delta): the W4A16 identity form (pinned above)
    applied to the int8 rows as exact fp64 values, then scaled per token."""
    d = synth.make_inputs(41, 4, 512, 32, group_size=gs)
    Xq, xs = oracle.quantize_per_token(d["A"])
    sb, zb = oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"])
    got = oracle.gemm_w4a8_asym(Xq, xs, d["q"], sb, zb, gs)
    ident = oracle.gemm_asym_identity(Xq.astype(np.float64), d["q"], sb, zb, gs) * xs.astype(np.float64)[:, None]
    assert oracle.rel_fro(got, ident) <= 1e-12


def test_w4a8_asym_reduces_to_symmetric_when_zero_is_minus_8_scale():
    """zero = -8 scale (delta = 0) turns q*s + z into (q - 8)*s: the symmetric W4A8
    reference with the same (positive, so unfolded) scales, exactly."""
    d = synth.make_inputs(42, 2, 256, 16)
    Xq, xs = oracle.quantize_per_token(d["A"])
    sb = oracle.half_bits(d["scale"])
    z = (-8.0 * d["scale"].astype(np.float64)).astype(np.float16)  # exact: times a power of two
    got = oracle.gemm_w4a8_asym(Xq, xs, d["q"], sb, oracle.half_bits(z), 128)
    want = oracle.gemm_w4a8(Xq, xs, d["q"], sb, 128)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------- grouped (mixture of experts)

def _grouped_case(seed, E=4, K=256, N=32, counts=(3, 0, 5, 2)):
    rng = _rng(seed)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(offs[-1])
    A = rng.standard_normal((M, K)).astype(np.float16).astype(np.float64)
    q = rng.integers(0, 16, size=(E, K, N)).astype(np.uint8)
    s = rng.uniform(0.005, 0.02, size=(E, K // 128, N)).astype(np.float16)
    z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
    return A, offs, q, oracle.half_bits(s), oracle.half_bits(z)


def test_grouped_equals_block_diagonal_gemm():
    """The grouped product equals one plain GEMM of block-expanded rows (expert e's rows
    occupy columns e*K .. (e+1)*K, zeros elsewhere) against the experts' weights stacked
    along K: the zero blocks add exactly nothing, so the two agree bit for bit."""
    A, offs, q, sb, zb = _grouped_case(50)
    E, K, N = q.shape
    M = A.shape[0]
    Ablk = np.zeros((M, E * K))
    for e in range(E):
        Ablk[offs[e]:offs[e + 1], e * K:(e + 1) * K] = A[offs[e]:offs[e + 1]]
    qcat = q.reshape(E * K, N)
    want = oracle.gemm_asym_plain(Ablk, qcat, sb.reshape(-1, N), zb.reshape(-1, N), 128)
    got = oracle.gemm_grouped_asym(A, offs, q, sb, zb, 128)
    assert np.array_equal(got, want)


def test_grouped_with_one_expert_is_the_plain_gemm():
    A, _, q, sb, zb = _grouped_case(51, E=1, counts=(6,))
    got = oracle.gemm_grouped_asym(A, [0, 6], q, sb, zb, 128)
    assert np.array_equal(got, oracle.gemm_asym_plain(A, q[0], sb[0], zb[0], 128))


@pytest.mark.parametrize("zero_point", [False, True])
def test_grouped_w4a8_equals_block_diagonal_gemm(zero_point):
    """Grouped W4A8 (folded symmetric or zero-point weights): the int8 rows expanded
    block-diagonally along K against the experts' weights stacked along K give the same
    per-token-scaled product bit for bit (the zero blocks add exact zeros)."""
    rng = _rng(52 + zero_point)
    E, K, N, counts = 3, 256, 24, (2, 4, 0)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(offs[-1])
    Xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    xs = rng.uniform(0.01, 0.05, size=M).astype(np.float32)
    q = rng.integers(0, 16, size=(E, K, N)).astype(np.uint8)
    s = rng.uniform(0.005, 0.02, size=(E, K // 128, N)).astype(np.float16)
    z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
    sb, zb = oracle.half_bits(s), (oracle.half_bits(z) if zero_point else None)
    Xblk = np.zeros((M, E * K), np.int8)
    for e in range(E):
        Xblk[offs[e]:offs[e + 1], e * K:(e + 1) * K] = Xq[offs[e]:offs[e + 1]]
    qcat, scat = q.reshape(E * K, N), sb.reshape(-1, N)
    if zero_point:
        want = oracle.gemm_w4a8_asym(Xblk, xs, qcat, scat, zb.reshape(-1, N), 128)
    else:
        want = oracle.gemm_w4a8(Xblk, xs, qcat, scat, 128)
    got = oracle.gemm_grouped_w4a8(Xq, xs, offs, q, sb, zb, 128)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------- SwiGLU gate/up pair

def _pair_weights(rng, K, N, zero_point=True):
    ws = []
    for _ in range(2):
        q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
        s = rng.uniform(0.005, 0.02, size=(K // 128, N)).astype(np.float16)
        z = (-s.astype(np.float64) * rng.uniform(6, 10, size=s.shape)).astype(np.float16)
        ws.append((q, s, z if zero_point else None))
    return ws


def _weight_values(q, s, z):
    """W[k, n] = q * s + z (or (q - 8) * s), fp64, one group of 128 along K."""
    sr = np.repeat(s.astype(np.float64), 128, axis=0)
    if z is None:
        return (q.astype(np.float64) - 8.0) * sr
    return q.astype(np.float64) * sr + np.repeat(z.astype(np.float64), 128, axis=0)


@pytest.mark.parametrize("zero_point", [True, False])
def test_swiglu_one_hot_rows_equal_library_sigmoid(zero_point):
    """A row with a single 1 at k selects row k of each weight, so the pair gives
    W_gate[k] * sigmoid(W_gate[k]) * W_up[k]; the sigmoid here is scipy's expit, not the
    oracle's formula.  Swapping gate and up fails this (silu is not symmetric)."""
    special = pytest.importorskip("scipy.special")
    rng = _rng(60 + zero_point)
    K, N = 256, 40
    (qg, sg, zg), (qu, su, zu) = _pair_weights(rng, K, N, zero_point)
    ks = np.array([0, 5, 127, 128, 255])
    A = np.zeros((len(ks), K))
    A[np.arange(len(ks)), ks] = 1.0
    gate = (qg, oracle.half_bits(sg), None if zg is None else oracle.half_bits(zg))
    up = (qu, oracle.half_bits(su), None if zu is None else oracle.half_bits(zu))
    got = oracle.gemm_swiglu_pair(A, gate, up, 128)
    Wg, Wu = _weight_values(qg, sg, zg)[ks], _weight_values(qu, su, zu)[ks]
    want = Wg * special.expit(Wg) * Wu
    assert np.allclose(got, want, rtol=1e-14, atol=0)


def test_swiglu_zero_gate_and_large_gate():
    """silu(0) = 0: a gate weight of exact zeros (q = 8, zero = -8 scale) gives Y = 0 for any
    rows; a large positive gate (all activations 1, K = 1024, weights near +0.1) makes
    sigmoid = 1 to fp64 precision, so Y = G * U."""
    rng = _rng(62)
    K, N = 1024, 24
    A = rng.standard_normal((3, K))
    (qg, sg, zg), up = _pair_weights(rng, K, N)
    up = (up[0], oracle.half_bits(up[1]), oracle.half_bits(up[2]))
    q8 = np.full((K, N), 8, np.uint8)
    z8 = (-8.0 * sg.astype(np.float64)).astype(np.float16)  # exact: times a power of two
    y0 = oracle.gemm_swiglu_pair(A, (q8, oracle.half_bits(sg), oracle.half_bits(z8)), up, 128)
    assert np.all(y0 == 0.0)
    ones = np.ones((2, K))
    qh = np.full((K, N), 12, np.uint8)
    sh = np.full((K // 128, N), 0.025, np.float16)
    zh = np.zeros_like(sh)  # w = 12 * 0.025 = 0.3 each, G = 1024 * 0.3 ~ 307
    gate = (qh, oracle.half_bits(sh), oracle.half_bits(zh))
    G = oracle.gemm_asym_plain(ones, qh, oracle.half_bits(sh), oracle.half_bits(zh), 128)
    U = oracle.gemm_asym_plain(ones, up[0], up[1], up[2], 128)
    assert np.array_equal(oracle.gemm_swiglu_pair(ones, gate, up, 128), G * U)


def test_pair_interleave_is_a_paired_permutation():
    """The pair layout holds every gate and every up column exactly once, and gate column j
    sits 8 columns before up column j inside one 16-column group."""
    N = 64
    gate = np.arange(N)[None, :]
    up = 1000 + np.arange(N)[None, :]
    c = oracle.pair_interleave(gate, up)[0]
    assert sorted(c.tolist()) == list(range(N)) + list(range(1000, 1000 + N))
    pos = {v: i for i, v in enumerate(c.tolist())}
    for j in range(N):
        assert pos[1000 + j] == pos[j] + 8 and pos[j] // 16 == pos[1000 + j] // 16


# --------------------------------------------------------------------------- pin sensitivity

def _pins_pass():
    try:
        test_delta_golden_example()
        test_identity_equals_plain_definition(3, 256, 16, 128)
        test_fold_golden_table()
        test_fold_equivalence_except_minus8()
        test_w4a8_matches_integer_closed_form()
        test_zero_weights_give_zero()
        test_w4a8_asym_integer_closed_form()
        test_grouped_equals_block_diagonal_gemm()
        test_grouped_w4a8_equals_block_diagonal_gemm(True)
        test_swiglu_one_hot_rows_equal_library_sigmoid(True)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("mid", [1, 2, 3, 4, 5, 6, 7, 8])
def test_planted_mistakes_are_caught(mid):
    """A plausible mistake planted in the oracle (wrong delta sign, wrong clamp, wrong
    offset, dropped correction, dropped activation scale, dropped W4A8 zero point, rows
    multiplied by the wrong expert, the SwiGLU activation on the up projection) fails at
    least one pin."""
    assert _pins_pass()
    with oracle.mutation(mid):
        assert not _pins_pass()
    assert _pins_pass()
