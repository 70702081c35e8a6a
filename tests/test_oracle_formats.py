"""Pins of the oracle's NVFP4 number formats and quantizer against what the pages
and independent libraries fix (CPU only)."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden
from nvfp4_weight_only_quantize_gb300 import synth

G = golden("nvfp4_format.txt")
# All 256 E4M3 byte values decoded by torch's float8_e4m3fn (a library that is run).
TORCH_E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decoder_matches_torch_on_all_bytes():
    for b in range(256):
        v = oracle.e4m3_value(b)
        if math.isnan(TORCH_E4M3[b]):
            assert math.isnan(v), b
        else:
            assert v == TORCH_E4M3[b], (b, v, TORCH_E4M3[b])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e2m1_decoder_is_the_golden_grid():
    mags = [float(v) for v in G["e2m1_magnitudes"].split(",")]
    assert [oracle.e2m1_value(c) for c in range(8)] == mags
    assert [oracle.e2m1_value(8 + c) for c in range(8)] == [-m for m in mags]


def test_format_size_facts():
    # 4 bits per code + one 8-bit scale per block of 16 = 4.5 bits/value; ratios vs FP16/FP8.
    bits = 4 + 8 / int(G["block_size"])
    assert bits == float(G["bits_per_value"])
    assert 16 / bits == pytest.approx(float(G["ratio_vs_fp16"]), abs=0.1)  # about 3.5 times
    assert 8 / bits == pytest.approx(float(G["ratio_vs_fp8"]), abs=0.05)  # about 1.8 times


def _threshold_code(q: float) -> int:
    """E2M1 rounding written as explicit midpoints (a different formulation from the
    oracle's nearest-value scan): ties .25,1.25,2.5,5 go down, .75,1.75,3.5 go up."""
    a = abs(q)
    c = (a > 0.25) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5) + (a >= 3.5) + (a > 5.0)
    return (c | 8) if (c and q < 0) else c


def test_e2m1_rounding_exhaustive_over_bf16():
    pats = np.arange(65536, dtype=np.uint32)
    vals = (pats << 16).view(np.float32)
    for q in vals:
        if not np.isfinite(q):
            continue
        assert oracle.e2m1_round(float(q)) == _threshold_code(float(q)), q


def test_e2m1_ties_and_saturation():
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 1e30: 7,
             -0.25: 0, -0.2: 0, -0.3: 9, -7.0: 15, 0.0: 0, -0.0: 0}
    for q, c in cases.items():
        assert oracle.e2m1_round(q) == c, (q, oracle.e2m1_round(q), c)


def _e4m3_up_by_torch(t: np.float32) -> int:
    """Smallest finite E4M3 >= t from torch's RNE conversion: RNE lands on a
    neighbour of t, so it is either the answer or the value just below it."""
    if not t > 0:
        return 0
    if t > 448:
        return 0x7E
    b = int(torch.tensor([float(t)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
    if TORCH_E4M3[b] >= t:
        return b
    return b + 1


def test_e4m3_round_up_against_torch():
    rng = np.random.default_rng(1)
    ts = list(rng.uniform(0, 460, 2000).astype(np.float32)) + list((2.0 ** rng.uniform(-14, 9, 3000)).astype(np.float32))
    for b in range(127):  # every finite value and its float32 neighbours
        v = np.float32(TORCH_E4M3[b])
        ts += [v, np.nextafter(v, np.float32(1e9)), np.nextafter(v, np.float32(0))]
    ts += [np.float32(0), np.float32(448.0), np.float32(448.01), np.float32(1e-30)]
    for t in ts:
        assert oracle.e4m3_round_up(float(t)) == _e4m3_up_by_torch(t), t


def test_e4m3_round_nearest_even_against_torch():
    rng = np.random.default_rng(2)
    ts = np.concatenate([rng.uniform(0, 447.9, 2000), 2.0 ** rng.uniform(-12, 8.7, 2000)]).astype(np.float32)
    mids = [(TORCH_E4M3[b] + TORCH_E4M3[b + 1]) / 2 for b in range(126)]  # exact ties
    ts = np.concatenate([ts, np.array(mids, np.float32)])
    got = np.array([oracle.e4m3_round_rne(float(t)) for t in ts])
    ref = torch.from_numpy(ts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, ref)


def _bf16_bits(vals) -> np.ndarray:
    v = torch.tensor(np.asarray(vals, np.float64), dtype=torch.float64)
    assert torch.equal(v.to(torch.bfloat16).to(torch.float64), v), "not exactly representable in bf16"
    return synth.bits(v.to(torch.bfloat16))


def test_round_trip_every_code_and_scale():
    """Blocks built as e2m1(code) * e4m3(scale) * 2^k round-trip to the same bytes:
    s_t is forced to 2^k by a global amax of 2688 * 2^k, and every block carries a
    +-6 element so its scale is found exactly."""
    k = -10
    codes_cycle = [c for c in range(16) if c != 8]  # 0x8 (-0) is never emitted
    rows, want_codes, want_scales = [], [], []
    for sb in range(1, 127):
        sc = TORCH_E4M3[sb]
        blk_codes = codes_cycle + [7]  # 15 codes + one more +6
        rows.append([oracle.e2m1_value(c) * sc * 2.0 ** k for c in blk_codes])
        want_codes.append(blk_codes)
        want_scales.append(sb)
    W = _bf16_bits(rows)
    rc, codes, scales, st = oracle.nvfp4_quantize(W)
    assert rc == 0 and st == np.float32(2.0 ** k)
    assert list(scales[:, 0]) == want_scales
    for i, blk in enumerate(want_codes):
        got = [(codes[i, j // 2] >> (4 * (j % 2))) & 15 for j in range(16)]
        assert got == blk, (i, got, blk)


def _unpack(codes):
    lo, hi = codes & 15, codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


@pytest.mark.parametrize("shape", [(64, 256), (33, 48), (1, 16)])
def test_quantizer_invariants_on_synthetic_weights(shape):
    N, K = shape
    W = synth.weight(N, K, seed=synth.seed_of(0, 0, synth.T_W))
    Wb = synth.bits(W)
    w = W.to(torch.float64).numpy()
    rc, codes, scales, st = oracle.nvfp4_quantize(Wb)
    assert rc == 0
    assert st == np.float32(np.float32(np.abs(w).max()) / np.float32(2688.0))
    c = _unpack(codes)
    assert not np.any(c == 8), "negative zero emitted"
    assert np.all(scales < 0x7F)
    what = oracle.nvfp4_dequantize(codes, scales, st, N, K)
    blocks = np.abs(w).reshape(N, K // 16, 16)
    cb = (c & 7).reshape(N, K // 16, 16)
    sc = TORCH_E4M3[scales]
    for n in range(N):
        for b in range(K // 16):
            if scales[n, b] >= 8:  # E4M3-normal scale: block amax maps to magnitude 6
                assert cb[n, b, np.argmax(blocks[n, b])] == 7
    # |w_hat - w| <= half the widest E2M1 gap (1.0) * scale * s_t
    err = np.abs(what - w)
    bound = np.repeat(sc * float(st), 16, axis=1) * 1.0 + 1e-30
    assert np.all(err <= bound)
    # the global-amax element is reproduced to E2M1 resolution: |w_hat| within 1/8 of amax
    i = np.argmax(np.abs(w))
    assert abs(abs(what.flat[i]) - abs(w.flat[i])) <= abs(w.flat[i]) / 8
    # storage: 4 bits/code + 8 bits per 16 = 0.5625 bytes/weight
    assert (codes.nbytes + scales.nbytes) / (N * K) == 0.5625


def test_quantizer_zero_and_nonfinite_and_shape():
    rc, codes, scales, st = oracle.nvfp4_quantize(np.zeros((2, 32), np.uint16))
    assert rc == 0 and st == 1.0 and not codes.any() and not scales.any()
    bad = np.zeros((2, 32), np.uint16)
    bad[1, 5] = 0x7F80  # +Inf
    assert oracle.nvfp4_quantize(bad)[0] == oracle.ORC_ERR_NONFINITE
    bad[1, 5] = 0x7FC1  # NaN
    assert oracle.nvfp4_quantize(bad)[0] == oracle.ORC_ERR_NONFINITE
    assert oracle.nvfp4_quantize(np.zeros((2, 24), np.uint16))[0] == oracle.ORC_ERR_SHAPE


def test_quantizer_matches_brute_force_codes_on_tiny_input():
    """Brute force over all 16 codes: for each element the emitted code minimises
    |e2m1(c) - w/(scale*s_t)| (ties to the even code) among all 16 codes."""
    W = synth.weight(4, 32, seed=7)
    Wb = synth.bits(W)
    rc, codes, scales, st = oracle.nvfp4_quantize(Wb)
    w = W.to(torch.float32).numpy()
    c = _unpack(codes)
    for n in range(4):
        for k in range(32):
            denom = np.float32(np.float32(TORCH_E4M3[scales[n, k // 16]]) * st)
            q = np.float32(w[n, k] / denom)
            d = [abs(oracle.e2m1_value(cc) - float(q)) for cc in range(16)]
            best = min(d)
            cands = [cc for cc in range(16) if d[cc] == best and cc != 8]
            even = [cc for cc in cands if cc % 2 == 0]
            pick = (even or cands)
            if oracle.e2m1_value(pick[0]) == 0:
                pick = [0]
            assert c[n, k] in pick, (n, k, q, c[n, k], pick)
