"""GPU pack / unpack / fold / dequant / per-token quantization against the oracle,
bit for bit (integer and byte work; dequantized weights rounded once)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wq():
    import weight_only_int4_g128_gb300 as m
    m.load_library(build_if_missing=True)
    assert m.device_supported(torch.cuda.current_device())
    return m


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("K,N,gs", [(256, 256, 128), (384, 640, 128), (1024, 128, -1),
                                    (4096, 384, 128)])
def test_pack_w4a16_bit_exact(wq, K, N, gs):
    d = synth.make_inputs(100 + K + N, 1, K, N, group_size=gs)
    Bp, S, dl = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), gs)
    torch.cuda.synchronize()
    want = oracle.pack(d["q"])
    assert np.array_equal(Bp.cpu().numpy().view(np.uint32), want)
    assert np.array_equal(_u16(S), oracle.half_bits(d["scale"]))
    want_d = oracle.delta(oracle.half_bits(d["scale"]), oracle.half_bits(d["zero"]))
    assert np.array_equal(dl.cpu().numpy().view(np.uint32), want_d.view(np.uint32))
    q2 = wq.unpack_w4(Bp, K, N)
    assert np.array_equal(q2.cpu().numpy(), d["q"])


def test_pack_every_code_every_position(wq):
    K, N = 128, 128
    q = np.zeros((K, N), np.uint8)
    for k in range(K):
        q[k] = (np.arange(N) + k * 7 + k // 8) % 16
    s = np.full((1, N), 0.01, np.float16)
    z = np.full((1, N), -0.08, np.float16)
    Bp, _, _ = wq.pack_w4a16(_cuda(q), _cuda(s), _cuda(z), 128)
    assert np.array_equal(Bp.cpu().numpy().view(np.uint32), oracle.pack(q))


@pytest.mark.parametrize("K,N", [(256, 256), (1024, 384)])
def test_pack_w4a8_fold_bit_exact(wq, K, N):
    d = synth.make_inputs(200 + K, 1, K, N, mode="w4a8")
    Bp, S = wq.pack_w4a8(_cuda(d["q"]), _cuda(d["scale"]), 128)
    torch.cuda.synchronize()
    qf, sf = oracle.fold(d["q"], oracle.half_bits(d["scale"]), 128)
    assert np.array_equal(Bp.cpu().numpy().view(np.uint32), oracle.pack(qf))
    assert np.array_equal(_u16(S), sf)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("gs", [128, -1])
def test_dequant_bit_exact(wq, dtype, gs):
    K, N = 512, 384
    d = synth.make_inputs(300, 1, K, N, group_size=gs)
    Bp, S, _ = wq.pack_w4a16(_cuda(d["q"]), _cuda(d["scale"]), _cuda(d["zero"]), gs)
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    W = wq.dequant_w4(Bp, S, K, N, gs, tdt)
    sb = oracle.half_bits(d["scale"])
    want = (oracle.dequant_sym_f16 if dtype == "f16" else oracle.dequant_sym_bf16)(d["q"], sb, gs)
    assert np.array_equal(_u16(W), want)


def test_dequant_extreme_scales_bit_exact(wq):
    """Scales across the binary16 range (subnormal to large) still round once."""
    K, N = 128, 256
    rng = np.random.Generator(np.random.PCG64(7))
    q = rng.integers(0, 16, (K, N), dtype=np.uint8)
    bits = rng.integers(0, 0x7BFF, (1, N)).astype(np.uint16)
    bits[0, :4] = [0x0001, 0x03FF, 0x0400, 0x7BFF]
    s = bits.view(np.float16)
    z = np.zeros_like(s)
    Bp, S, _ = wq.pack_w4a16(_cuda(q), _cuda(s), _cuda(z), 128)
    for dtype, fn in ((torch.float16, oracle.dequant_sym_f16),
                      (torch.bfloat16, oracle.dequant_sym_bf16)):
        W = wq.dequant_w4(Bp, S, K, N, 128, dtype)
        assert np.array_equal(_u16(W), fn(q, bits, 128))


@pytest.mark.parametrize("M,K", [(1, 64), (7, 5120), (64, 300)])
def test_quantize_per_token_bit_exact(wq, M, K):
    x = synth.make_activations(400 + M, M, K)
    if M > 2:
        x[2] = 0
    Xq, xs = wq.quantize_per_token(_cuda(x))
    wXq, wxs = oracle.quantize_per_token(x)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), wxs.view(np.uint32))
    assert np.array_equal(Xq.cpu().numpy(), wXq)


def test_quantize_ties_round_half_even(wq):
    t = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.25, -2.75]], np.float16)
    Xq, xs = wq.quantize_per_token(_cuda(t))
    assert xs.item() == 1.0
    assert Xq.cpu().numpy().tolist() == [[127, 0, 2, 2, 0, -2, 3, -3]]
