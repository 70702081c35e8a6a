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


@pytest.fixture(params=[q.ALGO_AUTO, q.ALGO_SIMT], ids=["tcgen05", "cuda_cores"])
def algo(request):
    """The variant forwards on the tensor-core kernel (AUTO, where K % 256 == 0)
    and on the CUDA-core GEMM."""
    q.set_linear_algo(request.param)
    yield request.param
    q.set_linear_algo(q.ALGO_AUTO)


# K = 32 and 96 are CUDA-core shapes under either selection; the others cover
# the tensor-core kernel's token tiles (16 .. 256), split-K launches (N = 256,
# K = 4096), ragged N, ranks over one 64-wide LoRA step (96, 256) and, above
# 64 tokens, the down-projection on tensor cores.
VARIANT_SHAPES = [(1, 32, 1, 1), (5, 96, 37, 4), (1, 512, 300, 8), (64, 3584, 512, 32), (17, 1024, 384, 16),
                  (8, 4096, 256, 32), (5, 512, 130, 96), (3, 256, 128, 256), (200, 1024, 384, 32)]


@pytest.mark.parametrize("M,K,N,r", VARIANT_SHAPES)
def test_mxfp4_linear(M, K, N, r, algo):
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


@pytest.mark.parametrize("k", [-100, 12, 60])
def test_mxfp4_linear_scale_range(k, algo):
    """Weights (and B) scaled by 2^k: E8M0 bytes near 20, 132 and 180, below and
    above 128, where the tensor-core dequantizer's second factor takes over."""
    M, K, N, r = 16, 512, 256, 16
    W = (synth.weight(N, K, 70).float() * 2.0 ** k).to(torch.bfloat16).cuda()
    x = synth.activations(M, K, 71).cuda()
    A = synth.lora_A(r, K, 72).cuda()
    B = (synth.lora_B(N, r, 73).float() * 2.0 ** k).to(torch.bfloat16).cuda()
    codes, scales = q.qerl_mxfp4_quantize(W)
    y = q.qerl_mxfp4_lora_linear_fwd(x, codes, scales, A, B, 2.0)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rc, oc, osc = oracle.mxfp4_quantize(synth.bits(W))
    assert np.array_equal(scales.cpu().numpy(), osc)
    b = osc.astype(np.int64)
    assert (b.max() < 128) if k < 0 else (b.min() > 128), (b.min(), b.max())
    ref = oracle.mxfp4_lora_linear_fwd(synth.bits(x), oc, osc, synth.bits(A), synth.bits(B), 2.0)
    assert np.isfinite(f64(y)).all()
    assert_rel_rms(f64(y), ref, LIN_TOL, "y")


def test_mxfp4_linear_gate_proj_sampled(algo):
    """Qwen2.5-7B gate_proj (18944 x 3584) at M = 8, r = 32, the bench's format
    workload; tokens 0 and 7 against the oracle."""
    if algo == q.ALGO_SIMT:
        pytest.skip("the CUDA-core GEMM is covered at smaller sizes")
    M, K, N, r = 8, 3584, 18944, 32
    W = synth.weight(N, K, 80, "cuda")
    x = synth.activations(M, K, 81).cuda()
    A = synth.lora_A(r, K, 82).cuda()
    B = synth.lora_B(N, r, 83).cuda()
    codes, scales = q.qerl_mxfp4_quantize(W)
    y = q.qerl_mxfp4_lora_linear_fwd(x, codes, scales, A, B, 2.0)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rc, oc, osc = oracle.mxfp4_quantize(synth.bits(W.cpu()))
    assert rc == 0 and np.array_equal(scales.cpu().numpy(), osc)
    rows = np.array([0, 7])
    ref = oracle.mxfp4_lora_linear_fwd(synth.bits(x), oc, osc, synth.bits(A), synth.bits(B), 2.0, rows=rows)
    assert_rel_rms(f64(y)[rows], ref, LIN_TOL, "y")


def _f32_adapters(r, K, N, seed):
    rng = np.random.default_rng(seed)
    A = torch.tensor((rng.standard_normal((r, K)) / np.sqrt(K)).astype(np.float32)).cuda()
    B = torch.tensor((rng.standard_normal((N, r)) * 0.01).astype(np.float32)).cuda()
    return A, B


@pytest.mark.parametrize("M,K,N,r", [(3, 48, 33, 5)] + VARIANT_SHAPES[2:] + [(8, 2048, 2048, 64)])
def test_f32_adapters(M, K, N, r, algo):
    c = LinearCase(M, K, N, r, config=15, idx=M).quantize_gpu()
    A, B = _f32_adapters(r, K, N, M + K)
    t = torch.empty(M, r, dtype=torch.float32, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd_f32ab(c.x, c.codes, c.scales, c.ts, A, B, 2.0, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    oc, osc, ost = c.oracle_quant()
    ref, tref = oracle.lora_linear_fwd_f32ab(synth.bits(c.x), oc, osc, ost, A.cpu().numpy(), B.cpu().numpy(), 2.0,
                                             want_t=True)
    assert_rel_rms(f64(y), ref, LIN_TOL, "y")
    assert_rel_rms(f64(t), tref, 1e-5, "t")


@pytest.mark.parametrize("M,K,N,r", [(8, 512, 384, 32), (64, 256, 200, 96)])
def test_f32_adapters_lora_term_precision(M, K, N, r, algo):
    """A zero weight leaves y = bf16(s t B^T): both paths must round the LoRA
    term as the fp64 oracle's value rounds, up to the term's own error (bf16
    B or u would move a third or more of the outputs by an ulp; the hi/lo
    products, about 2^-16 of the term, and the FP32 GEMM leave well under 2 %),
    and stay within an ulp plus 2^-14 of the outputs' rms."""
    x = synth.activations(M, K, 90).cuda()
    codes = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.full((N, K // 16), 0x38, dtype=torch.uint8, device="cuda")  # e4m3 1.0
    ts = torch.ones(1, dtype=torch.float32, device="cuda")
    A, B = _f32_adapters(r, K, N, 91)
    B = B * 100.0  # a LoRA term of order one
    y = q.qerl_nvfp4_lora_linear_fwd_f32ab(x, codes, scales, ts, A, B, 2.0)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    ref = oracle.lora_linear_fwd_f32ab(synth.bits(x), codes.cpu().numpy(), scales.cpu().numpy(), 1.0,
                                       A.cpu().numpy(), B.cpu().numpy(), 2.0)
    ref_bf16 = torch.tensor(ref).to(torch.bfloat16).to(torch.float64).numpy()
    got = f64(y)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * np.sqrt(np.mean(ref ** 2))
    assert (np.abs(got - ref) <= bound).all(), np.max(np.abs(got - ref) / bound)
    assert (got != ref_bf16).mean() < 0.02, (got != ref_bf16).mean()


@pytest.mark.parametrize("chained", [True, False], ids=["chained", "serialised"])
def test_variants_back_to_back_share_one_workspace(chained):
    """Two MXFP4 forwards and two FP32-adapter forwards issued back to back on one
    stream, each pair through one workspace, with no synchronisation between:
    each call rewrites the workspace (the expanded scales, u) that the call before
    it reads, so each output must still match its own oracle, with launches
    chained (each kernel may start before its predecessor ends) and serialised."""
    q.set_launch_chaining(chained)
    try:
        M, K, N, r = 8, 2048, 1024, 32
        x = synth.activations(M, K, 100).cuda()
        A = synth.lora_A(r, K, 101).cuda()
        B = synth.lora_B(N, r, 102).cuda()
        Ws = [synth.weight(N, K, 103 + i).cuda() * (2.0 ** (8 * i)) for i in range(2)]
        mx = [q.qerl_mxfp4_quantize(W.to(torch.bfloat16)) for W in Ws]
        ws = q.workspace(q.OP_MXFP4_FWD, M, N, K, r)
        ys = [q.qerl_mxfp4_lora_linear_fwd(x, c, s, A, B, 2.0, ws=ws) for c, s in mx]
        cases = [LinearCase(M, K, N, r, config=16, idx=i).quantize_gpu() for i in range(2)]
        Af, Bf = _f32_adapters(r, K, N, 104)
        wsf = q.workspace(q.OP_LINEAR_FWD_F32AB, M, N, K, r)
        yf = [q.qerl_nvfp4_lora_linear_fwd_f32ab(c.x, c.codes, c.scales, c.ts, Af, Bf, 2.0, ws=wsf) for c in cases]
        torch.cuda.synchronize()
        assert q.get_error() == 0
        for W, y in zip(Ws, ys):
            rc, oc, osc = oracle.mxfp4_quantize(synth.bits(W.to(torch.bfloat16)))
            ref = oracle.mxfp4_lora_linear_fwd(synth.bits(x), oc, osc, synth.bits(A), synth.bits(B), 2.0)
            assert_rel_rms(f64(y), ref, LIN_TOL, "y (MXFP4)")
        for c, y in zip(cases, yf):
            oc, osc, ost = c.oracle_quant()
            ref = oracle.lora_linear_fwd_f32ab(synth.bits(c.x), oc, osc, ost, Af.cpu().numpy(), Bf.cpu().numpy(), 2.0)
            assert_rel_rms(f64(y), ref, LIN_TOL, "y (FP32 adapters)")
    finally:
        q.set_launch_chaining(True)
