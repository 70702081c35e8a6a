"""Shared helpers of the parity tests: seeded inputs on both sides and the
tolerance checks.  Tolerances:
  - quantized codes, scale bytes, tensor scale, Philox words: bit-exact;
  - linear outputs (y, dx, dA, dB): |got - ref| <= 1e-2 * (|ref| + rms(ref))
    elementwise, rms over the checked outputs;
  - AQN-RMSNorm: |got - ref| <= 2e-3 * (|ref| + rms(ref)) + ulp_bf16(ref) / 2; the
    half ulp is the rounding of the bf16 result itself (up to 2^-8 relative), which
    no bf16 output can avoid and which is larger than 2e-3 in the low part of a
    binade; noise z: 1e-5 absolute (FP32 Box-Muller against the fp64 oracle:
    the log, the sine/cosine and the FP32 forms of u1 and u2 each err by about
    one part in 2^24 of values up to 8.6, a few 1e-6 at most).
"""
import numpy as np
import torch

import oracle
from nvfp4_weight_only_quantize_gb300 import synth

LIN_TOL = 1e-2
_QUANT_CACHE = {}  # the oracle's quantization of the 8 most recent weights
NORM_TOL = 2e-3
Z_TOL = 1e-5


def half_ulp_bf16(ref):
    """Half the spacing of bf16 numbers at |ref| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(ref, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def assert_rel_rms(got, ref, tol, what="", bf16_out=False):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = tol * (np.abs(ref) + rms)
    if bf16_out:
        bound = bound + half_ulp_bf16(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tol {tol}; worst at {i}: "
                             f"got {got[i]}, ref {ref[i]}, rms {rms}")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class LinearCase:
    """One seeded linear (W quantized by the oracle AND by the GPU, which must agree)."""

    def __init__(self, M, K, N, r, config=0, layer=0, idx=0, device="cuda", lora_scale=2.0, dy_std=1e-2):
        base = synth.seed_of(config, layer, 16 * idx)
        self.seed = base
        self.M, self.K, self.N, self.r, self.s = M, K, N, r, lora_scale
        gen_dev = device if N * K > 4_000_000 else "cpu"
        self.W = synth.weight(N, K, base + synth.T_W, gen_dev).to(device)
        self.x = synth.activations(M, K, base + synth.T_X, gen_dev).to(device)
        self.A = synth.lora_A(r, K, base + synth.T_A, gen_dev).to(device)
        self.B = synth.lora_B(N, r, base + synth.T_B, gen_dev).to(device)
        self.dy = synth.activations(M, N, base + synth.T_DY, gen_dev, std=dy_std).to(device)

    def quantize_gpu(self):
        import nvfp4_weight_only_quantize_gb300 as q
        self.codes, self.scales, self.ts = q.qerl_nvfp4_quantize(self.W)
        return self

    def oracle_quant(self):
        key = (self.N, self.K, self.seed)
        if key not in _QUANT_CACHE:
            rc, codes, scales, st = oracle.nvfp4_quantize(synth.bits(self.W))
            assert rc == 0
            if len(_QUANT_CACHE) >= 8:
                _QUANT_CACHE.pop(next(iter(_QUANT_CACHE)))
            _QUANT_CACHE[key] = (codes, scales, st)
        return _QUANT_CACHE[key]
