"""Tensor-core rank products against the oracle: t = x A^T of the many-token
forward (alone and for up to three linears sharing one pass over x), and v = dy B,
t = x A^T of the backward (checked through dA = s v^T x and dB = s dy^T t).
Token counts around the 128-token tile, reductions that are not a multiple of
the 64-wide stage, ranks on both sides of the 32/64 padding and of the 4-wide
vector stores, and reductions long enough for many splits."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N,r", [(65, 256, 128, 1), (128, 512, 64, 5), (129, 256, 200, 31), (300, 1280, 136, 33),
                                     (1000, 768, 128, 64), (65, 16384, 128, 32), (300, 512, 136, 128),
                                     (130, 256, 64, 100), (200, 512, 72, 65)])
def test_forward_t_many_tokens(M, K, N, r):
    c = LinearCase(M, K, N, r, config=9, idx=M + r).quantize_gpu()
    t = torch.empty(M, r, dtype=torch.float32, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_out=t)
    y0 = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    assert torch.equal(y, y0)  # t requested or not: the same down-projection
    oc, osc, ost = c.oracle_quant()
    ref, tref = oracle.lora_linear_fwd(synth.bits(c.x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s,
                                       want_t=True)
    assert_rel_rms(f64(t), tref, 1e-5, "t")
    assert_rel_rms(f64(y), ref, LIN_TOL, "y")


@pytest.mark.parametrize("M,K,N,r", [(1, 80, 64, 1), (127, 80, 24, 5), (128, 208, 200, 32), (129, 1040, 136, 33),
                                     (700, 64, 1000, 63), (300, 16, 8, 64), (2000, 4096, 64, 16)])
# (300, 16, 8, 64): reductions shorter than one stage keep the CUDA-core kernel
def test_backward_rank_products(M, K, N, r):
    c = LinearCase(M, K, N, r, config=9, idx=3 * M + r).quantize_gpu()
    dx, dA, dB = q.qerl_nvfp4_lora_linear_bwd(c.dy, c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    oc, osc, ost = c.oracle_quant()
    rdx, rdA, rdB = oracle.lora_linear_bwd(synth.bits(c.dy), synth.bits(c.x), oc, osc, ost, synth.bits(c.A),
                                           synth.bits(c.B), c.s)
    assert_rel_rms(f64(dx), rdx, LIN_TOL, "dx")
    assert_rel_rms(f64(dA), rdA, LIN_TOL, "dA")
    assert_rel_rms(f64(dB), rdB, LIN_TOL, "dB")


def test_backward_rank_matches_cuda_cores():
    """The tensor-core and CUDA-core rank products give the same weight
    gradients dA = s v^T x and dB = s dy^T t to 5e-5: the tensor-core wide
    products take the FP32 v and t as a bf16 pair hi + lo, exact to 2^-18
    relative per term, so over ~25k outputs the worst one strays about
    4 x 2^-18 = 1.5e-5 of the rms, plus the FP32 summation order.  dx is only
    held to the oracle tolerance here: the tensor-core dx takes its LoRA term
    through a bf16 copy of v, the CUDA-core dx through the FP32 v."""
    c = LinearCase(515, 1024, 320, 24, config=9, idx=11).quantize_gpu()
    outs = {}
    try:
        for algo in (q.ALGO_AUTO, q.ALGO_SIMT):
            q.set_linear_algo(algo)
            outs[algo] = q.qerl_nvfp4_lora_linear_bwd(c.dy, c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
            torch.cuda.synchronize()
            assert q.get_error() == 0
    finally:
        q.set_linear_algo(q.ALGO_AUTO)
    assert_rel_rms(f64(outs[q.ALGO_AUTO][0]), f64(outs[q.ALGO_SIMT][0]), LIN_TOL, "dx")
    for name, a, b in zip(("dA", "dB"), outs[q.ALGO_AUTO][1:], outs[q.ALGO_SIMT][1:]):
        assert_rel_rms(f64(a), f64(b), 5e-5, name)


@pytest.mark.parametrize("M,Ns,r", [(200, [128, 256, 64], 12), (130, [136, 72], 40), (1000, [256, 128, 128], 32),
                                    (200, [128, 256, 64], 96)])
def test_grouped_t_many_tokens(M, Ns, r):
    """r = 96 pads to 128 ranks per group: two groups per pass over x, then one."""
    K = 512
    cases = [LinearCase(M, K, N, r, config=9, idx=40 + i).quantize_gpu() for i, N in enumerate(Ns)]
    x = cases[0].x
    gs = [(c.codes, c.scales, c.ts, c.A, c.B) for c in cases]
    t_outs = [torch.empty(M, r, dtype=torch.float32, device="cuda") for _ in Ns]
    ys = q.qerl_nvfp4_lora_linear_fwd_grouped(x, gs, 2.0, t_outs=t_outs)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    for i, c in enumerate(cases):
        oc, osc, ost = c.oracle_quant()
        ref, tref = oracle.lora_linear_fwd(synth.bits(x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), 2.0,
                                           want_t=True)
        assert_rel_rms(f64(t_outs[i]), tref, 1e-5, f"t[{i}]")
        assert_rel_rms(f64(ys[i]), ref, LIN_TOL, f"y[{i}]")
