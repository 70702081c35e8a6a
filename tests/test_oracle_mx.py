"""Pins of the oracle's format variants: MXFP4 (blocks of 32, E8M0 scales; the
bitsofall "NVFP4" section contrasts NVFP4 with MXFP4's 32-value power-of-two
scaled blocks; the block-scale rule is the OCP MX one) and the linear forward
with FP32 LoRA adapters (the same page's LoRA paragraph: adapters in higher
precision, e.g. FP32).  Each check uses something other than the oracle's own
formula: exact powers of two, a brute-force nearest-grid search, numpy."""
import math

import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_quantize_gb300 import synth

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_block_of_32_shares_one_scale():
    """The page's MXFP4 block size (golden fixture): a large value at position 31
    sets the scale of positions 0..31 (so the small ones there round to zero),
    while positions 32..63 get their own scale and keep their small values."""
    from conftest import golden
    bs = int(golden("nvfp4_format.txt")["mxfp4_block_size"])
    w = np.full((1, 2 * bs), 0.1, np.float32)
    w[0, bs - 1] = 100.0
    rc, qc, qs = oracle.mxfp4_quantize(bf16_bits(w))
    assert rc == 0 and qs.shape == (1, 2)
    codes = np.zeros(2 * bs, np.int64)
    codes[0::2] = qc[0] & 15
    codes[1::2] = qc[0] >> 4
    assert np.all(codes[:bs - 1] == 0) and codes[bs - 1] == 7
    assert np.all(codes[bs:] != 0)
    assert qs[0, 0] > qs[0, 1]


def test_e8m0_decoder_every_byte():
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.e8m0_value(255))


@pytest.mark.parametrize("e", [-127, -100, -3, 0, 5, 60, 125])
def test_round_trip_every_code(e):
    """Blocks of values code * 2^e with one element at +-6 * 2^e come back as the
    same codes and the scale byte e + 127 (negative zero as code 0)."""
    rng = np.random.default_rng(e + 200)
    N, K = 16, 64
    codes = rng.integers(0, 16, size=(N, K))
    codes[:, 0] = 7
    codes[:, 32] = 15
    vals = np.array([GRID[c & 7] * (-1.0 if c & 8 else 1.0) for c in codes.ravel()]).reshape(N, K)
    W = bf16_bits(np.ldexp(vals, e))
    rc, qc, qs = oracle.mxfp4_quantize(W)
    assert rc == 0
    assert np.all(qs == e + 127)
    expect = np.where(codes == 8, 0, codes)
    got = np.zeros((N, K), np.int64)
    got[:, 0::2] = qc & 15
    got[:, 1::2] = qc >> 4
    assert np.array_equal(got, expect)


def _nearest_code(q):
    """Brute force: the grid value nearest |q| (ties to the even code), sign bit."""
    a = abs(q)
    best, bi = None, 0
    for i, g in enumerate(GRID):
        d = abs(a - g)
        if best is None or d < best or (d == best and i % 2 == 0 and bi % 2 == 1):
            best, bi = d, i
    if bi == 0:
        return 0
    return bi | (8 if q < 0 else 0)


def test_brute_force_codes_and_scale_rule():
    W = synth.weight(8, 96, 31)
    Wb = synth.bits(W)
    rc, qc, qs = oracle.mxfp4_quantize(Wb)
    assert rc == 0
    w = W.float().numpy().astype(np.float64)
    for n in range(8):
        for b in range(3):
            blk = w[n, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            e = math.floor(math.log2(amax)) - 2
            assert qs[n, b] == e + 127
            assert 4.0 <= amax / 2.0 ** e < 8.0
            for i in range(32):
                k = 32 * b + i
                c = (qc[n, k // 2] >> (4 * (k % 2))) & 15
                assert c == _nearest_code(blk[i] / 2.0 ** e), (n, k)


def test_dequantize_and_error_bound():
    W = synth.weight(32, 128, 32)
    Wb = synth.bits(W)
    rc, qc, qs = oracle.mxfp4_quantize(Wb)
    assert rc == 0
    wh = oracle.mxfp4_dequantize(qc, qs, 32, 128)
    codes = np.zeros((32, 128), np.int64)
    codes[:, 0::2] = qc & 15
    codes[:, 1::2] = qc >> 4
    mag = np.array(GRID)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    scale = np.ldexp(1.0, np.repeat(qs.astype(np.int64) - 127, 32, axis=1))
    assert np.array_equal(wh, mag * scale)
    w = W.float().numpy().astype(np.float64)
    q = np.abs(w) / scale
    step = np.select([q < 2, q < 4], [0.5, 1.0], 2.0)  # grid spacing around |q|
    inside = q <= 6
    assert np.all(np.abs(wh - w)[inside] <= 0.5 * step[inside] * scale[inside] + 1e-300)
    assert np.all(np.abs(wh)[~inside] == 6.0 * scale[~inside])


def test_zero_block_and_errors():
    Wb = np.zeros((2, 64), np.uint16)
    rc, qc, qs = oracle.mxfp4_quantize(Wb)
    assert rc == 0 and np.all(qc == 0) and np.all(qs == 0)
    assert oracle.mxfp4_quantize(np.zeros((2, 48), np.uint16))[0] == 2  # K % 32 != 0
    bad = np.zeros((2, 64), np.uint16)
    bad[1, 5] = 0x7F80  # +inf
    assert oracle.mxfp4_quantize(bad)[0] == 4


def test_mx_linear_against_numpy():
    M, K, N, r = 5, 128, 48, 4
    Wb = synth.bits(synth.weight(N, K, 33))
    rc, qc, qs = oracle.mxfp4_quantize(Wb)
    x = synth.bits(synth.activations(M, K, 34))
    A = synth.bits(synth.lora_A(r, K, 35))
    B = synth.bits(synth.lora_B(N, r, 36))
    y, t = oracle.mxfp4_lora_linear_fwd(x, qc, qs, A, B, 2.0, want_t=True)
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wh = oracle.mxfp4_dequantize(qc, qs, N, K)
    tr = f(x) @ f(A).T
    assert np.allclose(t, tr, rtol=1e-12, atol=1e-12)
    assert np.allclose(y, f(x) @ wh.T + 2.0 * tr @ f(B).T, rtol=1e-12, atol=1e-12)


def test_f32_adapters_reduce_to_bf16_and_match_numpy():
    M, K, N, r = 4, 64, 40, 8
    Wb = synth.bits(synth.weight(N, K, 37))
    rc, qc, qs, st = oracle.nvfp4_quantize(Wb)
    x = synth.bits(synth.activations(M, K, 38))
    Ab = synth.bits(synth.lora_A(r, K, 39))
    Bb = synth.bits(synth.lora_B(N, r, 40))
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    # bf16-representable FP32 adapters give exactly the bf16-adapter forward
    y16 = oracle.lora_linear_fwd(x, qc, qs, st, Ab, Bb, 2.0)
    y32 = oracle.lora_linear_fwd_f32ab(x, qc, qs, st, f(Ab), f(Bb), 2.0)
    assert np.array_equal(y16, y32)
    # arbitrary FP32 adapters against numpy on the oracle's dequantized weight
    rng = np.random.default_rng(3)
    A = (rng.standard_normal((r, K)) / 8).astype(np.float32)
    B = (rng.standard_normal((N, r)) / 100).astype(np.float32)
    y, t = oracle.lora_linear_fwd_f32ab(x, qc, qs, st, A, B, 2.0, want_t=True)
    wh = oracle.nvfp4_dequantize(qc, qs, st, N, K)
    xf = f(x).astype(np.float64)
    assert np.allclose(t, xf @ A.astype(np.float64).T, rtol=1e-12, atol=1e-12)
    assert np.allclose(y, xf @ wh.T + 2.0 * t @ B.astype(np.float64).T, rtol=1e-12, atol=1e-12)
