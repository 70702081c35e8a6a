"""GPU parity of the decoder-layer glue (residual add, SwiGLU) and of a decoder
layer run as a sequence of this library's calls.

The glue against plain references: bf16(h + y) bit for bit against torch's FP32
sum rounded to bf16 (the sum of two bf16 values is exact in FP32 here), and
bf16(silu(g) u) within one bf16 unit of the fp64 value.

The layer: N1(h0) -> q|k|v (one grouped call); h1 = h0 + o(attn); N2(h1) ->
gate, up; m = silu(g) u; h2 = h1 + down(m), every activation carried in bf16,
against the oracle chain with the textbook norm (the norm's output rounded to
bf16 before the linears), the reading these calls implement.  The chain test
module provides the seeded layers and that oracle chain."""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, assert_rel_rms, f64
from test_gpu_chain_layers import EPS, Chain, assert_resid, to_bits, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,offset", [(1, 0), (7, 0), (4096, 0), (64 * 27648, 0), (1000, 1)])
def test_residual_add_bit_exact(n, offset):
    h = synth.activations(1, n + offset, 500).cuda().view(-1)[offset:]
    y = (synth.activations(1, n + offset, 501).cuda().view(-1)[offset:] * 0.1).to(torch.bfloat16)
    out = q.qerl_residual_add(h, y)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    assert torch.equal(out, (h.float() + y.float()).to(torch.bfloat16))
    h2 = h.clone()
    q.qerl_residual_add(h2, y, out=h2)  # in place
    assert torch.equal(h2, out)


@pytest.mark.parametrize("n,offset", [(3, 0), (4096, 0), (64 * 27648, 0), (1001, 1)])
def test_swiglu_within_one_unit(n, offset):
    g = (synth.activations(1, n + offset, 502).cuda().view(-1)[offset:] * 4.0).to(torch.bfloat16)
    u = synth.activations(1, n + offset, 503).cuda().view(-1)[offset:]
    out = q.qerl_swiglu(g, u)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    gd, ud = f64(g), f64(u)
    ref = gd / (1.0 + np.exp(-gd)) * ud
    err = np.abs(f64(out) - ref)
    assert (err <= ulp_bf16(ref) + 1e-30).all(), np.max(err / ulp_bf16(ref))


def test_swiglu_extremes():
    """Large negative g (e^-g overflows FP32: silu -> -0), large positive g (silu
    = g), zeros and signs."""
    g = torch.tensor([-200.0, -90.0, -1.0, 0.0, 1.0, 90.0, 200.0, 3.0e38], dtype=torch.bfloat16, device="cuda")
    u = torch.tensor([1.0, 2.0, -3.0, 5.0, 0.5, -1.0, 1.0, 0.0], dtype=torch.bfloat16, device="cuda")
    out = f64(q.qerl_swiglu(g, u))
    torch.cuda.synchronize()
    gd, ud = f64(g), f64(u)
    with np.errstate(over="ignore"):
        ref = gd / (1.0 + np.exp(-gd)) * ud
    assert np.all(np.abs(out - ref) <= ulp_bf16(ref)), (out, ref)


def per_linear_layer(ch, l, h, sigma, seed, step):
    """Decoder layer l of `ch` (noise keys 2l, 2l + 1) on h [M, H] bf16 through
    the library's calls; returns h2 and leaves q, k, v in the layer's buffers."""
    Ly, M = ch.layers[l], ch.M
    ws_norm = q.workspace(q.OP_AQN_RMSNORM, M, 0, ch.H, 0)
    n1 = q.qerl_aqn_rmsnorm(h, Ly["gamma_attn"], EPS, sigma, seed, step, 2 * l, ws=ws_norm)
    q.qerl_nvfp4_lora_linear_fwd_grouped(n1, [Ly[nm] for nm in ("q", "k", "v")], 2.0, packed=True,
                                         ys=[Ly[nm + "_out"] for nm in ("q", "k", "v")])
    o = q.qerl_nvfp4_lora_linear_fwd_packed(Ly["attn"], *Ly["o"], 2.0)
    h1 = q.qerl_residual_add(h, o)
    n2 = q.qerl_aqn_rmsnorm(h1, Ly["gamma_mlp"], EPS, sigma, seed, step, 2 * l + 1, ws=ws_norm)
    g = q.qerl_nvfp4_lora_linear_fwd_packed(n2, *Ly["gate"], 2.0)
    u = q.qerl_nvfp4_lora_linear_fwd_packed(n2, *Ly["up"], 2.0)
    m = q.qerl_swiglu(g, u)
    d = q.qerl_nvfp4_lora_linear_fwd_packed(m, *Ly["down"], 2.0)
    return q.qerl_residual_add(h1, d, out=h1)


def check_per_linear(ch, rows, sigma, seed, step):
    """Each layer, fed the oracle chain's input of that layer on the sampled
    rows, against the textbook-norm oracle layer."""
    hb = synth.bits(ch.x)[rows]
    for l in range(ch.L):
        x = ch.x.clone()
        x[torch.as_tensor(rows)] = torch.from_numpy(hb.astype(np.int16)).view(torch.bfloat16).to(x.device)
        out = per_linear_layer(ch, l, x, sigma, seed, step)
        torch.cuda.synchronize()
        assert q.get_error() == 0
        ref = ch.oracle_layer(l, hb, rows, sigma, seed, step, fused=False)
        for nm in ("q", "k", "v"):
            assert_rel_rms(f64(ch.layers[l][nm + "_out"])[rows], ref[nm], LIN_TOL, f"layer {l} {nm}")
        assert_resid(f64(out)[rows], ref["h"], ref["d"], f"layer {l} h")
        hb = to_bits(ref["h"])


def test_per_linear_layers_small():
    """Three small layers, every token."""
    ch = Chain(3, 17, 512, 512, 128, 768, 16, cfg=21)
    check_per_linear(ch, np.arange(17), 1e-2, 7, 3)


def test_per_linear_layer_qwen32b():
    """One Qwen2.5-32B decoder layer (hidden 5120, kv 1024, intermediate 27648),
    M = 64, r = 64, on sampled rows: the shapes of the 64-layer stack's
    per-linear path."""
    ch = Chain(1, 64, 5120, 5120, 1024, 27648, 64, cfg=3)
    check_per_linear(ch, np.array([0, 63]), 1e-2, 3, 1)
