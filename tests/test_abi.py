"""The C-ABI library loads, exports every symbol include/qerl.h declares, and
rejects bad arguments on the host before any CUDA call (CPU only)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import nvfp4_weight_only_quantize_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    q.build()
    return q.lib()


def test_header_symbols_are_exported(L):
    src = open(os.path.join(ROOT, "include", "qerl.h")).read()
    declared = set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(qerl_\w+)\s*\(", src, re.M))
    assert declared == set(q.EXPORTED), declared ^ set(q.EXPORTED)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings_and_workspace(L):
    for s in range(9):
        assert q.status_string(s)
    assert q.workspace_bytes(q.OP_QUANTIZE, 0, 10, 32, 0) >= 4096
    assert q.workspace_bytes(q.OP_AQN_RMSNORM, 4, 0, 3584, 0) >= 3584 * 4
    assert q.workspace_bytes(q.OP_LINEAR_FWD, 64, 3584, 3584, 32) >= 64 * 32 * 4
    assert q.workspace_bytes(q.OP_LINEAR_BWD, 64, 3584, 3584, 32) >= 2 * 64 * 32 * 4


def test_argument_errors_return_before_any_launch(L):
    fake = C.c_void_p(1 << 20)  # never dereferenced: every case fails its host check first
    ws = C.c_void_p(1 << 20)
    # quantize: K % 16, null pointers, misaligned row stride, bad rounding flag
    assert L.qerl_nvfp4_quantize(fake, 4, 24, 24, fake, fake, fake, None, ws, 4096, None) == 2
    assert L.qerl_nvfp4_quantize(None, 4, 32, 32, fake, fake, fake, None, ws, 4096, None) == 1
    assert L.qerl_nvfp4_quantize(fake, 4, 32, 36, fake, fake, fake, None, ws, 4096, None) == 3
    assert L.qerl_nvfp4_quantize(C.c_void_p((1 << 20) + 2), 4, 32, 32, fake, fake, fake, None, ws, 4096,
                                 None) == 3
    bad_opts = q._QuantOpts(7)
    assert L.qerl_nvfp4_quantize(fake, 4, 32, 32, fake, fake, fake, C.byref(bad_opts), ws, 4096, None) == 1
    assert L.qerl_nvfp4_quantize(fake, 4, 32, 32, fake, fake, fake, None, None, 0, None) == 8
    # linear: r out of range, K % 16, misaligned x, missing workspace
    args = lambda x, K, r, wsb: (x, 8, K, 16, fake, fake, fake, fake, fake, r, 2.0, fake, None, ws, wsb, None)
    assert L.qerl_nvfp4_lora_linear_fwd(*args(fake, 32, 0, 1 << 20)) == 2
    assert L.qerl_nvfp4_lora_linear_fwd(*args(fake, 32, 257, 1 << 20)) == 2
    assert L.qerl_nvfp4_lora_linear_fwd(*args(fake, 40, 4, 1 << 20)) == 2
    assert L.qerl_nvfp4_lora_linear_fwd(*args(C.c_void_p((1 << 20) + 8), 32, 4, 1 << 20)) == 3
    assert L.qerl_nvfp4_lora_linear_fwd(*args(fake, 32, 4, 0)) == 8
    bargs = (fake, fake, 8, 32, 16, fake, fake, fake, fake, fake, 4, 2.0, None, fake, fake, fake, 0, ws)
    assert L.qerl_nvfp4_lora_linear_bwd(*bargs, 0, None) == 8
    assert L.qerl_nvfp4_lora_linear_bwd(None, *bargs[1:], 1 << 20, None) == 1
    # AQN
    assert L.qerl_aqn_rmsnorm(fake, 4, 0, fake, 1e-6, 0.0, 0, 0, 0, fake, ws, 1 << 20, None) == 1
    assert L.qerl_aqn_rmsnorm(fake, 4, 64, fake, 1e-6, 0.1, 0, 0, 0, fake, None, 0, None) == 8
    assert L.qerl_aqn_rmsnorm_mode(fake, 4, 64, fake, 1e-6, 0.1, 0, 0, 0, 2, fake, ws, 1 << 20, None) == 1
    assert L.qerl_aqn_rmsnorm_mode(fake, 4, 64, fake, 1e-6, 0.1, 0, 0, 0, 1, fake, None, 0, None) == 8
    assert L.qerl_aqn_noise(0, 0, 0, 0, fake, None, None) == 1
    assert L.qerl_set_linear_algo(9) == 1
    assert L.qerl_set_linear_algo(4) == 1
    # decoder-layer glue: NULL pointers, negative length; an empty call launches nothing
    assert L.qerl_residual_add(None, fake, 8, fake, None) == 1
    assert L.qerl_swiglu(fake, fake, -1, fake, None) == 1
    assert L.qerl_swiglu(fake, fake, 0, fake, None) == 0
    # format variants: K % 32 (MXFP4) / K % 16, r, missing or short workspace
    vargs = lambda K, r, wsp, wsb: (fake, 8, K, 16, fake, fake, fake, fake, r, 2.0, fake, None, wsp, wsb, None)
    assert L.qerl_mxfp4_lora_linear_fwd(*vargs(48, 4, ws, 1 << 20)) == 2
    assert L.qerl_mxfp4_lora_linear_fwd(*vargs(64, 0, ws, 1 << 20)) == 2
    assert L.qerl_mxfp4_lora_linear_fwd(*vargs(64, 4, None, 0)) == 8
    need = q.workspace_bytes(q.OP_MXFP4_FWD, 8, 16, 256, 4)
    assert L.qerl_mxfp4_lora_linear_fwd(*vargs(256, 4, ws, need - 1)) == 8
    fargs = lambda K, r, wsb: (fake, 8, K, 16, fake, fake, fake, fake, fake, r, 2.0, fake, None, ws, wsb, None)
    assert L.qerl_nvfp4_lora_linear_fwd_f32ab(*fargs(40, 4, 1 << 20)) == 2
    need = q.workspace_bytes(q.OP_LINEAR_FWD_F32AB, 8, 16, 256, 4)
    assert L.qerl_nvfp4_lora_linear_fwd_f32ab(*fargs(256, 4, need - 1)) == 8


def test_grouped_argument_errors_return_before_any_launch(L):
    fake = 1 << 20  # never dereferenced
    g = q._Group(16, fake, fake, fake, fake, fake, fake, None)
    arr = (q._Group * 2)(g, g)
    ptr = C.cast(arr, C.c_void_p)

    def call(x, K, r, groups, n, packed, wsb):
        return L.qerl_nvfp4_lora_linear_fwd_grouped(x, 8, K, r, 2.0, groups, n, packed, fake, wsb, None)
    assert call(fake, 32, 4, None, 2, 0, 1 << 30) == 1      # no group array
    assert call(fake, 32, 4, ptr, 0, 0, 1 << 30) == 1       # n_groups outside 1..8
    assert call(fake, 32, 4, ptr, 9, 0, 1 << 30) == 1
    assert call(fake, 32, 4, ptr, 2, 2, 1 << 30) == 1       # packed flag
    assert call(fake, 32, 0, ptr, 2, 0, 1 << 30) == 2       # r outside 1..256
    assert call(fake, 40, 4, ptr, 2, 0, 1 << 30) == 2       # K % 16
    assert call(fake + 8, 32, 4, ptr, 2, 0, 1 << 30) == 3   # misaligned x
    assert call(fake, 32, 4, ptr, 2, 0, 0) == 8             # short workspace
    bad = (q._Group * 2)(g, q._Group(16, fake + 4, fake, fake, fake, fake, fake, None))
    assert call(fake, 32, 4, C.cast(bad, C.c_void_p), 2, 0, 1 << 30) == 3  # misaligned codes of group 1


def test_workspace_covers_every_region(L):
    """Lower bounds from the regions each call keeps in its workspace."""
    M, K, r = 4096, 5120, 32
    Ns = [5120, 1024, 1024]
    # grouped forward above 64 tokens: u per group (bf16 [M, 64]) + one partial slice per group
    assert q.grouped_ws_bytes(M, K, r, Ns) >= 3 * M * 64 * 2 + 3 * M * r * 4
    assert q.grouped_ws_bytes(M, K, 128, Ns) >= 3 * M * 128 * 2 + 3 * M * 128 * 4
    # backward: v and t (FP32), v' (bf16 [M, 64]), B^T (bf16 [r, N]), hi/lo pair (bf16 [M, 64]), partials
    M, N, K = 8192, 3584, 3584
    assert q.workspace_bytes(q.OP_LINEAR_BWD, M, N, K, r) >= 2 * M * r * 4 + M * 64 * 2 + r * N * 2 + M * 64 * 2
    # format variants on tensor cores: MXFP4 keeps one scale byte per 16 values (and the 2^-7 tensor scale)
    # beside u (bf16 [M, 64]); FP32 adapters keep u_hi | u_lo | u_hi (bf16 [M, 3 * 64]); the CUDA-core
    # GEMM (K % 256 != 0) keeps t (FP32 [M, r])
    M, N, K = 8, 18944, 3584
    assert q.workspace_bytes(q.OP_MXFP4_FWD, M, N, K, r) >= N * K // 16 + 4 + M * 64 * 2
    assert q.workspace_bytes(q.OP_LINEAR_FWD_F32AB, M, N, K, r) >= M * 3 * 64 * 2
    assert q.workspace_bytes(q.OP_MXFP4_FWD, M, N, 96, r) >= M * r * 4
    assert q.workspace_bytes(q.OP_LINEAR_FWD_F32AB, M, N, 48, r) >= M * r * 4
    assert q.workspace_bytes(q.OP_MXFP4_FWD, M, N, 48, r) == 0  # K % 32 != 0: no MXFP4 call


def test_sigma_schedule_matches_oracle(L):
    for S in (1, 2, 5, 10):
        for T in (1, 7, 1000):
            for t in (0, 1, T // 3, T - 1, T, 5 * T):
                got = q.qerl_aqn_sigma(t, T, 1e-2, 5e-4, S)
                assert got == pytest.approx(oracle.aqn_sigma(t, T, 1e-2, 5e-4, S), rel=1e-6)
    assert q.qerl_aqn_sigma(3, 10, 0.0, 1e-3, 4) == 0.0
