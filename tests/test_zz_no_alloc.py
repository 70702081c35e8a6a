"""The no-allocation forward, qerl_nvfp4_lora_linear_fwd_noalloc.

Some callers cannot call cudaMalloc: a host framework that owns every device
byte through its own memory pool and refuses allocations from outside it, or
code that must not allocate mid-step because cudaMalloc can synchronize the
device.  This entry point runs the same forward with a fixed scratch buffer in
the library's own device memory.  These tests call it through the C ABI twice
in a row and compare each result with the workspace entry point's output.

This file is named so that pytest collects it last: a run that stops at the
first failure has run every other test before it.  It passes on its own in a
fresh process too (the first call on a device sets up the scratch address).
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu


def _noalloc(L, c, y, t_out=None):
    s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: None if t is None else C.c_void_p(t.data_ptr())
    return L.qerl_nvfp4_lora_linear_fwd_noalloc(p(c.x), c.M, c.K, c.N, p(c.codes), p(c.scales), p(c.ts), p(c.A),
                                                p(c.B), c.r, C.c_float(c.s), p(y), p(t_out), s)


# Qwen2.5-7B decode shapes (split-K partial tiles and the LoRA u/t regions in
# the scratch), a prefill-sized M, and a shape the tensor-core path does not
# cover (K % 64 != 0: CUDA-core path).
@pytest.mark.parametrize("M,K,N,r", [(64, 3584, 3584, 32), (8, 3584, 512, 32), (1, 3584, 18944, 32),
                                     (4096, 2048, 2048, 16), (5, 48, 40, 4)])
def test_noalloc_matches_workspace_entry_point_twice(M, K, N, r):
    """Both entry points launch the same kernels in the same order; only where
    the scratch lives differs, so y and t must be identical bit for bit.  Each
    call starts from NaN-filled outputs, so a stale or unwritten scratch region
    shows up as a mismatch.  t is also checked against the fp64 oracle."""
    L = q.lib()
    c = LinearCase(M, K, N, r, config=7, idx=M + N).quantize_gpu()
    t_ref = torch.empty(M, r, dtype=torch.float32, device="cuda")
    ref = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_out=t_ref)
    torch.cuda.synchronize()
    rows = np.arange(M) if M <= 64 else np.array([0, 1, M // 2, M - 1])
    oc, osc, ost = c.oracle_quant()
    y_orc, t_orc = oracle.lora_linear_fwd(synth.bits(c.x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s,
                                          rows=rows, want_t=True)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        t = torch.full((M, r), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(L, c, y, t) == 0
        torch.cuda.synchronize()
        assert q.get_error() == 0
        assert torch.equal(y, ref), f"noalloc call {call}: y differs from the workspace entry point"
        assert torch.equal(t, t_ref), f"noalloc call {call}: t differs from the workspace entry point"
        assert_rel_rms(f64(y)[rows], y_orc, LIN_TOL, f"noalloc call {call}: y against the oracle")
        assert_rel_rms(f64(t)[rows], t_orc, 1e-5, f"noalloc call {call}: t against the oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    L = q.lib()
    # M * r_pad * 2 bytes of LoRA scratch alone exceed the 8 MiB buffer.
    M, K, N, r = 1 << 17, 64, 64, 32
    assert q.workspace_bytes(q.OP_LINEAR_FWD, M, N, K, r) > q.NOALLOC_SCRATCH_BYTES
    fake = C.c_void_p(1 << 20)
    st = L.qerl_nvfp4_lora_linear_fwd_noalloc(fake, M, K, N, fake, fake, fake, fake, fake, r, C.c_float(2.0), fake,
                                              None, None)
    assert st == 9 and "no-allocation" in q.status_string(st)
