"""Pins of the oracle's AQN noise, RMSNorm and sigma schedule (CPU only)."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from nvfp4_weight_only_quantize_gb300 import synth

MASK = (1 << 64) - 1


def _numpy_philox(ctr, key):
    """Philox4x64-10 block from numpy's bit generator (a library that is run).
    numpy advances its 256-bit counter before producing each block, so the block
    for counter c is the first output after seeding with c - 1; the test below
    also shows the counter words are little-endian."""
    c = sum(int(v) << (64 * i) for i, v in enumerate(ctr))
    c = (c - 1) % (1 << 256)
    words = np.array([(c >> (64 * i)) & MASK for i in range(4)], dtype=np.uint64)
    g = np.random.Philox(counter=words, key=np.array(key, dtype=np.uint64))
    return g.random_raw(4).astype(np.uint64)


@pytest.mark.parametrize("ctr,key", [
    ([0, 0, 0, 0], [0, 0]),
    ([1, 0, 0, 0], [5, 7]),
    ([123456, 42, 0, 0], [0x0123456789ABCDEF, 3]),
    ([MASK, 9, 0, 0], [MASK, MASK]),
    ([7, 0, 11, 13], [1, 2]),
])
def test_philox_matches_numpy(ctr, key):
    ours = oracle.philox4x64_10(np.array(ctr, np.uint64), np.array(key, np.uint64))
    np.testing.assert_array_equal(ours, _numpy_philox(ctr, key))


def test_noise_words_follow_counter_layout():
    H, seed, step, layer = 37, 1234, 17, 5
    z, raw = oracle.aqn_noise(H, seed, step, layer, want_raw=True)
    for c in range(H):
        blk = _numpy_philox([c // 4, step, 0, 0], [seed, layer])
        assert raw[c] == blk[c % 4]
    # Box-Muller on (w0, w1) and (w2, w3) of each block
    for c in range(0, H - 1, 2):
        blk = _numpy_philox([c // 4, step, 0, 0], [seed, layer])
        p = (c % 4) // 2
        u1 = ((int(blk[2 * p]) >> 11) + 1) * 2.0 ** -53
        u2 = (int(blk[2 * p + 1]) >> 11) * 2.0 ** -53
        rad = np.sqrt(-2 * np.log(u1))
        assert z[c] == pytest.approx(rad * np.cos(2 * np.pi * u2), abs=1e-14)
        assert z[c + 1] == pytest.approx(rad * np.sin(2 * np.pi * u2), abs=1e-14)


def test_noise_is_standard_normal_and_depends_on_every_key():
    z = oracle.aqn_noise(1_000_000, 42, 3, 1)
    assert abs(z.mean()) < 4e-3 and abs(z.var() - 1) < 6e-3
    assert stats.kstest(z[:200_000], "norm").pvalue > 1e-3
    base = oracle.aqn_noise(64, 42, 3, 1)
    for args in [(43, 3, 1), (42, 4, 1), (42, 3, 2)]:
        assert not np.allclose(base, oracle.aqn_noise(64, *args))
    np.testing.assert_array_equal(base, oracle.aqn_noise(64, 42, 3, 1))


def test_rmsnorm_sigma_zero_is_torch_rms_norm():
    x = synth.activations(6, 40, 3)
    g = synth.norm_gamma(40, 4)
    y = oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, 0.0, 1, 2, 3)
    ref = torch.nn.functional.rms_norm(x.double(), (40,), weight=g.double(), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12)


def test_rmsnorm_constant_row_closed_form():
    H = 32
    for bits_c, c in [(0x4000, 2.0), (0xBE80, -0.25)]:
        x = np.full((1, H), bits_c, np.uint16)
        g = synth.norm_gamma(H, 9)
        y = oracle.aqn_rmsnorm(x, synth.bits(g), 1e-6, 0.0, 0, 0, 0)
        ref = g.double().numpy() * np.sign(c) / np.sqrt(1 + 1e-6 / c ** 2)
        np.testing.assert_allclose(y[0], ref, rtol=1e-14)


def test_rmsnorm_noise_enters_the_scale_additively():
    x = synth.activations(3, 24, 5)
    g = synth.norm_gamma(24, 6)
    sigma = 0.01
    y = oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, sigma, 11, 12, 13)
    z = oracle.aqn_noise(24, 11, 12, 13)
    ref = torch.nn.functional.rms_norm(x.double(), (24,), weight=g.double() + sigma * torch.from_numpy(z),
                                       eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12)


def test_rmsnorm_noise_scales_the_scale_multiplicatively():
    """The other reading of noise in the norm's scale: y = rms_norm(x) with
    weight gamma * (1 + sigma z), against torch's rms_norm; with gamma = 1 the
    two readings coincide, and with sigma = 0 both are plain RMSNorm."""
    x = synth.activations(3, 24, 5)
    g = synth.norm_gamma(24, 6)
    sigma = 0.01
    y = oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, sigma, 11, 12, 13, multiplicative=True)
    z = torch.from_numpy(oracle.aqn_noise(24, 11, 12, 13))
    ref = torch.nn.functional.rms_norm(x.double(), (24,), weight=g.double() * (1 + sigma * z), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12)
    ones = np.full(24, 0x3F80, np.uint16)
    np.testing.assert_array_equal(oracle.aqn_rmsnorm(synth.bits(x), ones, 1e-6, sigma, 1, 2, 3, multiplicative=True),
                                  oracle.aqn_rmsnorm(synth.bits(x), ones, 1e-6, sigma, 1, 2, 3))
    np.testing.assert_array_equal(oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, 0.0, 1, 2, 3,
                                                     multiplicative=True),
                                  oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, 0.0, 1, 2, 3))


def test_sigma_schedule():
    s0, s1, S, T = 1e-2, 5e-4, 10, 1000
    vals = [oracle.aqn_sigma(t, T, s0, s1, S) for t in range(T)]
    assert vals[0] == pytest.approx(s0) and vals[-1] == pytest.approx(s1)
    stages = sorted(set(vals), reverse=True)
    assert len(stages) == S
    ratios = [stages[i + 1] / stages[i] for i in range(S - 1)]
    assert max(ratios) == pytest.approx(min(ratios), rel=1e-12)  # exponential: constant ratio
    assert ratios[0] == pytest.approx((s1 / s0) ** (1 / (S - 1)))
    assert all(vals[i] >= vals[i + 1] for i in range(T - 1))
    assert oracle.aqn_sigma(5, 10, s0, s1, 1) == s0 and oracle.aqn_sigma(T + 50, T, s0, s1, S) == pytest.approx(s1)
