"""GPU parity of the format variants against the oracle: the MXFP4 quantizer
(codes and E8M0 scale bytes bit for bit), the forward with an MXFP4 weight and
the forward with FP32 LoRA adapters (linear tolerance)."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(1, 32), (37, 96), (256, 512), (18944, 3584)])
def test_mxfp4_quantize_bit_exact(N, K):
    W = synth.weight(N, K, 50 + N, "cuda" if N * K > 4_000_000 else "cpu").cuda()
    codes, scales = q.qerl_mxfp4_quantize(W)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rc, oc, osc = oracle.mxfp4_quantize(synth.bits(W))
    assert rc == 0
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy(), osc)


def test_mxfp4_quantize_special_blocks():
    """All-zero blocks, tiny and huge magnitudes, exact powers of two."""
    vals = np.zeros((4, 64), np.float32)
    vals[1, :32] = 2.0 ** -130
    vals[1, 32:] = np.linspace(-3e38, 3e38, 32)
    vals[2, :] = 2.0 ** np.arange(-20, 44)
    vals[3, :] = np.tile([0.25, -0.75, 1.25, 5.0], 16)
    W = torch.tensor(vals).to(torch.bfloat16).cuda()
    codes, scales = q.qerl_mxfp4_quantize(W)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rc, oc, osc = oracle.mxfp4_quantize(synth.bits(W))
    assert np.array_equal(codes.cpu().numpy(), oc) and np.array_equal(scales.cpu().numpy(), osc)


@pytest.mark.parametrize("M,K,N,r", [(1, 32, 1, 1), (5, 96, 37, 4), (64, 3584, 512, 32), (17, 1024, 384, 16)])
def test_mxfp4_linear(M, K, N, r):
    W = synth.weight(N, K, 60 + N).cuda()
    x = synth.activations(M, K, 61).cuda()
    A = synth.lora_A(r, K, 62).cuda()
    B = synth.lora_B(N, r, 63).cuda()
    codes, scales = q.qerl_mxfp4_quantize(W)
    t = torch.empty(M, r, dtype=torch.float32, device="cuda")
    y = q.qerl_mxfp4_lora_linear_fwd(x, codes, scales, A, B, 2.0, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rc, oc, osc = oracle.mxfp4_quantize(synth.bits(W))
    ref, tref = oracle.mxfp4_lora_linear_fwd(synth.bits(x), oc, osc, synth.bits(A), synth.bits(B), 2.0, want_t=True)
    assert_rel_rms(f64(y), ref, LIN_TOL, "y")
    assert_rel_rms(f64(t), tref, 1e-5, "t")


@pytest.mark.parametrize("M,K,N,r", [(3, 48, 33, 5), (64, 3584, 512, 32), (8, 2048, 2048, 64)])
def test_f32_adapters(M, K, N, r):
    c = LinearCase(M, K, N, r, config=15, idx=M).quantize_gpu()
    rng = np.random.default_rng(M + K)
    A = torch.tensor((rng.standard_normal((r, K)) / np.sqrt(K)).astype(np.float32)).cuda()
    B = torch.tensor((rng.standard_normal((N, r)) * 0.01).astype(np.float32)).cuda()
    t = torch.empty(M, r, dtype=torch.float32, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd_f32ab(c.x, c.codes, c.scales, c.ts, A, B, 2.0, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    oc, osc, ost = c.oracle_quant()
    ref, tref = oracle.lora_linear_fwd_f32ab(synth.bits(c.x), oc, osc, ost, A.cpu().numpy(), B.cpu().numpy(), 2.0,
                                             want_t=True)
    assert_rel_rms(f64(y), ref, LIN_TOL, "y")
    assert_rel_rms(f64(t), tref, 1e-5, "t")
