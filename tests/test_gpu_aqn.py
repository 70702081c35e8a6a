"""GPU parity of the AQN noise and AQN-RMSNorm against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import NORM_TOL, Z_TOL, assert_rel_rms, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,seed,step,layer", [(3584, 0, 0, 0), (5120, 12345, 77, 63), (37, 2 ** 63 + 5, 2 ** 40, 7)])
def test_noise_words_bit_exact_and_values(H, seed, step, layer):
    z, raw = q.qerl_aqn_noise(H, seed, step, layer, want_raw=True)
    oz, oraw = oracle.aqn_noise(H, seed, step, layer, want_raw=True)
    np.testing.assert_array_equal(raw.cpu().numpy().view(np.uint64), oraw)
    np.testing.assert_allclose(z.double().cpu().numpy(), oz, rtol=0, atol=Z_TOL)


@pytest.mark.parametrize("M,H,sigma", [(1, 3584, 1e-2), (8, 3584, 5e-4), (64, 3584, 0.0), (3, 100, 0.05),
                                       (5, 5120, 1e-2), (2, 8, 0.3)])
def test_rmsnorm_parity(M, H, sigma):
    x = synth.activations(M, H, 3 * M + H).cuda()
    g = synth.norm_gamma(H, H + 1).cuda()
    y = q.qerl_aqn_rmsnorm(x, g, 1e-6, sigma, seed=7, step=3, layer_id=2)
    ref = oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, sigma, 7, 3, 2)
    assert_rel_rms(f64(y), ref, NORM_TOL, "aqn_rmsnorm", bf16_out=True)


def test_rmsnorm_prefill_size_sampled_rows():
    """Qwen2.5-14B prefill: [4096, 5120], sigma 1e-2, checked on 64 sampled rows."""
    M, H = 4096, 5120
    x = synth.activations(M, H, synth.seed_of(2, 0, synth.T_X), "cuda")
    g = synth.norm_gamma(H, synth.seed_of(2, 0, synth.T_GAMMA), "cuda")
    y = q.qerl_aqn_rmsnorm(x, g, 1e-6, 1e-2, seed=2, step=5, layer_id=0)
    rows = np.sort(np.random.default_rng(0).choice(M, 64, replace=False))
    ref = oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, 1e-2, 2, 5, 0, rows=rows)
    assert_rel_rms(f64(y)[rows], ref, NORM_TOL, "aqn_rmsnorm prefill", bf16_out=True)


def test_rmsnorm_empty_batch():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = synth.norm_gamma(64, 1).cuda()
    y = q.qerl_aqn_rmsnorm(x, g, 1e-6, 0.1, 0, 0, 0)
    assert y.shape == (0, 64)


@pytest.mark.parametrize("M,H,sigma", [(1, 3584, 1e-2), (64, 3584, 5e-2), (3, 100, 0.05), (2, 20000, 1e-2)])
def test_rmsnorm_multiplicative_noise_parity(M, H, sigma):
    """The multiplicative reading, gamma (1 + sigma z), through the one-launch
    path (H <= 16384) and the two-kernel path (H = 20000); the additive mode
    of the same entry point equals qerl_aqn_rmsnorm bit for bit."""
    x = synth.activations(M, H, 5 * M + H).cuda()
    g = synth.norm_gamma(H, H + 3).cuda()
    y = q.qerl_aqn_rmsnorm(x, g, 1e-6, sigma, seed=9, step=4, layer_id=1, noise_mode=q.AQN_NOISE_MUL)
    ref = oracle.aqn_rmsnorm(synth.bits(x), synth.bits(g), 1e-6, sigma, 9, 4, 1, multiplicative=True)
    assert_rel_rms(f64(y), ref, NORM_TOL, "aqn_rmsnorm multiplicative", bf16_out=True)
    ya = q.qerl_aqn_rmsnorm(x, g, 1e-6, sigma, seed=9, step=4, layer_id=1, noise_mode=q.AQN_NOISE_ADD)
    yd = q.qerl_aqn_rmsnorm(x, g, 1e-6, sigma, seed=9, step=4, layer_id=1)
    torch.cuda.synchronize()
    assert torch.equal(ya, yd)
    assert not torch.equal(ya, y)


def test_rmsnorm_mode_rejects_unknown_mode():
    x = torch.zeros(1, 16, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QerlError):
        q.qerl_aqn_rmsnorm(x, g, 1e-6, 0.1, seed=1, step=1, layer_id=1, noise_mode=2)
