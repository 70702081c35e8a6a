"""Pins of the oracle's LoRA linear forward/backward (CPU only): closed forms,
numpy matmul of the dequantized weight, and adjoint identities."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_quantize_gb300 import synth


def _case(M=5, K=48, N=24, r=4, seed=3):
    W = synth.weight(N, K, seed)
    x = synth.activations(M, K, seed + 1)
    A = synth.lora_A(r, K, seed + 2)
    B = synth.lora_B(N, r, seed + 3)
    rc, codes, scales, st = oracle.nvfp4_quantize(synth.bits(W))
    assert rc == 0
    return dict(x=synth.bits(x), A=synth.bits(A), B=synth.bits(B), codes=codes, scales=scales, st=st,
                xf=x.double().numpy(), Af=A.double().numpy(), Bf=B.double().numpy(), M=M, K=K, N=N, r=r)


def test_forward_matches_numpy_matmul():
    c = _case()
    what = oracle.nvfp4_dequantize(c["codes"], c["scales"], c["st"], c["N"], c["K"])
    y = oracle.lora_linear_fwd(c["x"], c["codes"], c["scales"], c["st"], c["A"], c["B"], 2.0)
    ref = c["xf"] @ what.T + 2.0 * (c["xf"] @ c["Af"].T) @ c["Bf"].T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_forward_zero_adapter_is_plain_gemm_and_basis_vectors_pick_columns():
    c = _case(M=3, K=32, N=8, r=2)
    what = oracle.nvfp4_dequantize(c["codes"], c["scales"], c["st"], 8, 32)
    zeroA = np.zeros_like(c["A"])
    y = oracle.lora_linear_fwd(c["x"], c["codes"], c["scales"], c["st"], zeroA, c["B"], 2.0)
    np.testing.assert_allclose(y, c["xf"] @ what.T, rtol=1e-13)
    # x = e_k picks column k of w_hat (bf16 1.0 = 0x3F80)
    for k in (0, 5, 31):
        e = np.zeros((1, 32), np.uint16)
        e[0, k] = 0x3F80
        yk = oracle.lora_linear_fwd(e, c["codes"], c["scales"], c["st"], zeroA, c["B"], 2.0)
        np.testing.assert_array_equal(yk[0], what[:, k])


def test_forward_row_subset_and_t():
    c = _case(M=6)
    rows = np.array([4, 1], np.int64)
    y_all, t_all = oracle.lora_linear_fwd(c["x"], c["codes"], c["scales"], c["st"], c["A"], c["B"], 2.0,
                                          want_t=True)
    y_s, t_s = oracle.lora_linear_fwd(c["x"], c["codes"], c["scales"], c["st"], c["A"], c["B"], 2.0,
                                      rows=rows, want_t=True)
    np.testing.assert_array_equal(y_s, y_all[rows])
    np.testing.assert_allclose(t_all, c["xf"] @ c["Af"].T, rtol=1e-13)
    np.testing.assert_array_equal(t_s, t_all[rows])


def test_constant_code_weight_gives_row_sums():
    # every weight equal -> every block identical -> y[m, n] = w * sum_k x[m, k]
    K, N = 32, 4
    W = np.full((N, K), 0x3C00, np.uint16)  # bf16 0.0078125
    rc, codes, scales, st = oracle.nvfp4_quantize(W)
    x = synth.activations(3, K, 11)
    A = np.zeros((1, K), np.uint16)
    B = np.zeros((N, 1), np.uint16)
    y = oracle.lora_linear_fwd(synth.bits(x), codes, scales, st, A, B, 2.0)
    what = oracle.nvfp4_dequantize(codes, scales, st, N, K)
    assert np.all(what == what[0, 0]) and what[0, 0] == pytest.approx(0.0078125, rel=1e-6)
    ref = what[0, 0] * x.double().numpy().sum(1)
    np.testing.assert_allclose(y, np.repeat(ref[:, None], N, 1), rtol=1e-12)


def _fwd(c, x=None, A=None, B=None):
    return oracle.lora_linear_fwd(c["x"] if x is None else x, c["codes"], c["scales"], c["st"],
                                  c["A"] if A is None else A, c["B"] if B is None else B, 2.0)


def test_backward_adjoint_identities():
    c = _case(M=7, K=48, N=32, r=4)
    dy = synth.activations(7, 32, 99, std=0.01)
    dyb, dyf = synth.bits(dy), dy.double().numpy()
    dx, dA, dB = oracle.lora_linear_bwd(dyb, c["x"], c["codes"], c["scales"], c["st"], c["A"], c["B"], 2.0)
    # y is linear in x: <dy, y(x')> = <dx, x'> for any x'
    xp = synth.bits(synth.activations(7, 48, 5))
    xpf = synth.activations(7, 48, 5).double().numpy()
    assert np.sum(dyf * _fwd(c, x=xp)) == pytest.approx(np.sum(dx * xpf), rel=1e-10)
    # y is affine in A and in B: <dy, y(A') - y(0)> = <dA, A'>, same for B
    Ap = synth.lora_A(4, 48, 6)
    lin_A = np.sum(dyf * (_fwd(c, A=synth.bits(Ap)) - _fwd(c, A=np.zeros_like(c["A"]))))
    assert lin_A == pytest.approx(np.sum(dA * Ap.double().numpy()), rel=1e-10)
    Bp = synth.lora_B(32, 4, 7)
    lin_B = np.sum(dyf * (_fwd(c, B=synth.bits(Bp)) - _fwd(c, B=np.zeros_like(c["B"]))))
    assert lin_B == pytest.approx(np.sum(dB * Bp.double().numpy()), rel=1e-10)


def test_backward_subsets_match_full():
    c = _case(M=6, K=32, N=16, r=3)
    dy = synth.bits(synth.activations(6, 16, 12, std=0.01))
    full = oracle.lora_linear_bwd(dy, c["x"], c["codes"], c["scales"], c["st"], c["A"], c["B"], 2.0)
    rows, cols, nrows = np.array([5, 0]), np.array([31, 2, 7]), np.array([15, 3])
    sub = oracle.lora_linear_bwd(dy, c["x"], c["codes"], c["scales"], c["st"], c["A"], c["B"], 2.0,
                                 dx_rows=rows, dA_cols=cols, dB_rows=nrows)
    np.testing.assert_array_equal(sub[0], full[0][rows])
    np.testing.assert_array_equal(sub[1], full[1][:, cols])
    np.testing.assert_array_equal(sub[2], full[2][nrows])


def test_threaded_forward_equals_single_threaded():
    """Threads take whole output features; every element is summed in the same
    order, so the threaded forward equals the single-threaded one bit for bit."""
    rng = np.random.default_rng(5)
    N, K, M, r = 96, 64, 3, 4
    W = synth.bits(synth.weight(N, K, 71))
    rc, codes, scales, st = oracle.nvfp4_quantize(W)
    assert rc == 0
    x = synth.bits(synth.activations(M, K, 72))
    A = synth.bits(synth.lora_A(r, K, 73))
    B = synth.bits(synth.lora_B(N, r, 74))
    y1, t1 = oracle.lora_linear_fwd(x, codes, scales, st, A, B, 2.0, want_t=True)
    try:
        oracle.set_threads(4)
        y4, t4 = oracle.lora_linear_fwd(x, codes, scales, st, A, B, 2.0, want_t=True)
    finally:
        oracle.set_threads(1)
    assert np.array_equal(y1, y4) and np.array_equal(t1, t4)
    del rng
