"""GPU parity of the CUDA-core GEMV forward (one or two tokens) against the fp64
oracle: ragged shapes (N not a multiple of the rows per warp, K not a multiple
of a full batch of chunks, ranks 1 to 256), both code layouts, t output, the
grouped entry point, the full Qwen2.5-7B sizes on sampled rows, run-to-run
determinism, and the selection rules (AUTO, GEMV, fallback when M > 2)."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu


@pytest.fixture
def gemv():
    q.set_linear_algo(q.ALGO_GEMV)
    yield
    q.set_linear_algo(q.ALGO_AUTO)


def _check(c, y, t=None, rows=None):
    oc, osc, ost = c.oracle_quant()
    ref, tref = oracle.lora_linear_fwd(synth.bits(c.x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s,
                                       rows=rows, want_t=True)
    got = f64(y) if rows is None else f64(y)[rows]
    assert_rel_rms(got, ref, LIN_TOL, "y")
    if t is not None:
        assert_rel_rms(f64(t) if rows is None else f64(t)[rows], tref, 1e-5, "t")


# K = 32 (one chunk), 96, 4128 (129 chunks: a second, mostly empty batch),
# 4160; N = 1, 3, 33 (odd: a warp's second row past N), 77; r = 1 .. 256.
@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,N,r", [(32, 1, 1), (96, 33, 5), (256, 3, 8), (4128, 77, 32), (4160, 40, 256),
                                   (1024, 300, 64)])
def test_ragged(gemv, M, K, N, r):
    c = LinearCase(M, K, N, r, config=10, idx=K + N + r).quantize_gpu()
    t = torch.empty(M, r, dtype=torch.float32, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    _check(c, y, t)
    y2 = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)  # t in the workspace
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("M", [1, 2])
def test_packed_equals_standard(gemv, M):
    c = LinearCase(M, 2048, 515, 16, config=10, idx=7).quantize_gpu()
    packed = q.qerl_nvfp4_pack_codes(c.codes)
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    yp = q.qerl_nvfp4_lora_linear_fwd_packed(c.x, packed, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    assert torch.equal(y, yp)
    _check(c, yp)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("name", ["k_proj", "gate_proj", "down_proj"])
def test_qwen7b_full_size_sampled(gemv, M, name):
    """Qwen2.5-7B linears at their sizes (down_proj: K = 18944, x staged at
    76 / 152 KB), 48 sampled output features checked against the oracle."""
    wl = synth.WORKLOADS[1]
    _, N, K = next(l for l in wl.linears if l[0] == name)
    c = LinearCase(M, K, N, wl.r, config=1, idx=3).quantize_gpu()
    packed = q.qerl_nvfp4_pack_codes(c.codes)
    t = torch.empty(M, wl.r, dtype=torch.float32, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd_packed(c.x, packed, c.scales, c.ts, c.A, c.B, c.s, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rng = np.random.default_rng(N + K + M)
    cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 46, replace=False)]))
    oc, osc, ost = c.oracle_quant()
    xb = synth.bits(c.x)
    ref, tref = oracle.lora_linear_fwd(xb, oc[cols], osc[cols], ost, synth.bits(c.A), synth.bits(c.B)[cols], c.s,
                                       want_t=True)
    assert_rel_rms(f64(y)[:, cols], ref, LIN_TOL, "y")
    assert_rel_rms(f64(t), tref, 1e-5, "t")


def test_auto_takes_gemv_and_matches_tensor_cores():
    """AUTO at M = 1 on a small weight runs the GEMV (the launch count grows by
    its two kernels); the tensor-core path on the same call agrees with it
    within the tolerance."""
    c = LinearCase(1, 3584, 1000, 32, config=10, idx=11).quantize_gpu()
    q.set_linear_algo(q.ALGO_AUTO)
    n0 = q.lib().qerl_launch_count()
    y_auto = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.lib().qerl_launch_count() - n0 == 2  # down-projection + GEMV
    q.set_linear_algo(q.ALGO_GEMV)
    y_gemv = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    q.set_linear_algo(q.ALGO_TCGEN05)
    try:
        y_tc = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    finally:
        q.set_linear_algo(q.ALGO_AUTO)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    assert torch.equal(y_auto, y_gemv)
    _check(c, y_gemv)
    _check(c, y_tc)


def test_auto_keeps_tensor_cores_for_large_weights_and_two_tokens():
    """Above 24M weight values, and at two tokens, AUTO runs the tensor-core
    kernel (its output is bit-identical to the TCGEN05 selection's)."""
    for M, N, K in ((1, 7000, 4096), (2, 1000, 3584)):  # 28.7M weights; two tokens
        c = LinearCase(M, K, N, 16, config=10, idx=15 + M).quantize_gpu()
        ys = {}
        try:
            for algo in (q.ALGO_AUTO, q.ALGO_TCGEN05, q.ALGO_GEMV):
                q.set_linear_algo(algo)
                ys[algo] = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
        finally:
            q.set_linear_algo(q.ALGO_AUTO)
        torch.cuda.synchronize()
        assert q.get_error() == 0
        assert torch.equal(ys[q.ALGO_AUTO], ys[q.ALGO_TCGEN05])
        _check(c, ys[q.ALGO_AUTO])
        _check(c, ys[q.ALGO_GEMV])


def test_gemv_selection_falls_back_beyond_two_tokens(gemv):
    c = LinearCase(3, 512, 130, 8, config=10, idx=12).quantize_gpu()
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    _check(c, y)


def test_k_not_multiple_of_32_falls_back(gemv):
    c = LinearCase(1, 48, 20, 4, config=10, idx=13).quantize_gpu()
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    _check(c, y)


@pytest.mark.parametrize("algo", ["auto", "gemv"])
def test_grouped_qkv_at_one_token(algo):
    """q|k|v through the grouped entry point at M = 1: one tensor-core launch
    under AUTO, one GEMV per group when the GEMV is selected."""
    q.set_linear_algo(q.ALGO_GEMV if algo == "gemv" else q.ALGO_AUTO)
    wl = synth.WORKLOADS[1]
    cases = [LinearCase(1, K, N, wl.r, config=1, idx=20 + i).quantize_gpu() for i, (_, N, K) in
             enumerate(wl.linears[:3])]
    x = cases[0].x
    for c in cases:
        c.x = x
    try:
        ys = q.qerl_nvfp4_lora_linear_fwd_grouped(x, [(c.codes, c.scales, c.ts, c.A, c.B) for c in cases], 2.0)
    finally:
        q.set_linear_algo(q.ALGO_AUTO)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    for c, y in zip(cases, ys):
        rows = np.arange(0, c.N, 7)
        oc, osc, ost = c.oracle_quant()
        ref = oracle.lora_linear_fwd(synth.bits(x), oc[rows], osc[rows], ost, synth.bits(c.A),
                                     synth.bits(c.B)[rows], 2.0)
        assert_rel_rms(f64(y)[:, rows], ref, LIN_TOL, "y")


def test_deterministic(gemv):
    c = LinearCase(2, 3584, 2000, 32, config=10, idx=14).quantize_gpu()
    ys = [q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s) for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(ys[0], y) for y in ys[1:])


@pytest.mark.parametrize("M,K", [(1, 50944), (2, 25344), (2, 25600)])
def test_shared_memory_limit(gemv, M, K):
    """x staged in up to 200 KiB of shared memory: M * (K + r) * 4 bytes at the
    limit (1 x 50944 and 2 x 25344 take the GEMV), and just past it for two
    tokens (2 x 25600 falls back to the tensor-core kernel); every output
    checked on a narrow weight."""
    r = 16
    c = LinearCase(M, K, 40, r, config=10, idx=K + M).quantize_gpu()
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    _check(c, y)
