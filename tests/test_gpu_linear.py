"""GPU parity of the NVFP4 LoRA linear forward/backward against the fp64 oracle,
for every kernel path, from tiny ragged shapes to the full Qwen2.5 sizes."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu

ALGOS = [q.ALGO_SIMT, q.ALGO_AUTO]


@pytest.fixture(params=ALGOS, ids=["simt", "auto"])
def algo(request):
    q.set_linear_algo(request.param)
    yield request.param
    q.set_linear_algo(q.ALGO_AUTO)


def _fwd_check(c: LinearCase, rows=None, want_t=True):
    t = torch.empty(c.M, c.r, dtype=torch.float32, device="cuda") if want_t else None
    y = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    oc, osc, ost = oracle_q = c.oracle_quant()
    ref, tref = oracle.lora_linear_fwd(synth.bits(c.x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s,
                                       rows=rows, want_t=True)
    got = f64(y) if rows is None else f64(y)[rows]
    assert_rel_rms(got, ref, LIN_TOL, "y")
    if want_t:
        tg = f64(t) if rows is None else f64(t)[rows]
        assert_rel_rms(tg, tref, 1e-5, "t")
    return y


def _bwd_check(c: LinearCase, dx_rows=None, dA_cols=None, dB_rows=None, t_saved=None, accumulate=False):
    dA0 = torch.randn(c.r, c.K, device="cuda") if accumulate else None
    dB0 = torch.randn(c.N, c.r, device="cuda") if accumulate else None
    dx, dA, dB = q.qerl_nvfp4_lora_linear_bwd(c.dy, c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_saved=t_saved,
                                              dA=None if dA0 is None else dA0.clone(),
                                              dB=None if dB0 is None else dB0.clone(), accumulate=accumulate)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    oc, osc, ost = c.oracle_quant()
    rdx, rdA, rdB = oracle.lora_linear_bwd(synth.bits(c.dy), synth.bits(c.x), oc, osc, ost, synth.bits(c.A),
                                           synth.bits(c.B), c.s, dx_rows=dx_rows, dA_cols=dA_cols,
                                           dB_rows=dB_rows)
    gdx, gdA, gdB = f64(dx), f64(dA), f64(dB)
    if accumulate:
        gdA -= f64(dA0)
        gdB -= f64(dB0)
    assert_rel_rms(gdx if dx_rows is None else gdx[dx_rows], rdx, LIN_TOL, "dx")
    assert_rel_rms(gdA if dA_cols is None else gdA[:, dA_cols], rdA, LIN_TOL, "dA")
    assert_rel_rms(gdB if dB_rows is None else gdB[dB_rows], rdB, LIN_TOL, "dB")


def test_config0_full(algo):
    """Qwen2.5-3B q_proj 2048x2048, 16 tokens, r=16, every output."""
    c = LinearCase(16, 2048, 2048, 16, config=0).quantize_gpu()
    _fwd_check(c)
    _bwd_check(c)


@pytest.mark.parametrize("M,K,N,r", [(1, 16, 1, 1), (3, 48, 33, 5), (17, 256, 200, 8), (64, 1024, 384, 32),
                                     (130, 512, 136, 16), (257, 2048, 520, 64), (9, 4096, 128, 256),
                                     (20, 192, 100, 4), (70, 320, 257, 12), (200, 768, 192, 24), (129, 256, 64, 256),
                                     (5, 512, 128, 64)])
def test_ragged_shapes(algo, M, K, N, r):
    c = LinearCase(M, K, N, r, config=9, idx=M + N).quantize_gpu()
    _fwd_check(c)
    _bwd_check(c)


def test_bwd_with_saved_t_and_accumulate(algo):
    c = LinearCase(40, 512, 256, 16, config=9, idx=3).quantize_gpu()
    t = torch.empty(c.M, c.r, dtype=torch.float32, device="cuda")
    q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_out=t)
    _bwd_check(c, t_saved=t, accumulate=True)


def test_empty_batch(algo):
    c = LinearCase(1, 64, 32, 4, config=9).quantize_gpu()
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd(x, c.codes, c.scales, c.ts, c.A, c.B, 2.0)
    assert y.shape == (0, 32)
    dy = torch.empty(0, 32, dtype=torch.bfloat16, device="cuda")
    dx, dA, dB = q.qerl_nvfp4_lora_linear_bwd(dy, x, c.codes, c.scales, c.ts, c.A, c.B, 2.0,
                                              dA=torch.ones(4, 64, device="cuda"), dB=torch.ones(32, 4, device="cuda"))
    torch.cuda.synchronize()
    assert float(dA.abs().max()) == 0 and float(dB.abs().max()) == 0


QWEN7B = synth.WORKLOADS[1]


@pytest.mark.parametrize("M", [1, 8, 64])
@pytest.mark.parametrize("lin", range(7), ids=[l[0] for l in QWEN7B.linears])
def test_qwen7b_decode_full_size(M, lin):
    """Qwen2.5-7B decoder-layer linears at full size in the decode launch shape;
    checked on up to 4 sampled token rows (all outputs of each)."""
    name, N, K = QWEN7B.linears[lin]
    c = LinearCase(M, K, N, QWEN7B.r, config=1, idx=lin).quantize_gpu()
    rows = np.arange(M) if M <= 4 else np.sort(np.random.default_rng(lin).choice(M, 4, replace=False))
    _fwd_check(c, rows=rows)


@pytest.mark.parametrize("lin", [0, 1, 4, 6], ids=["q_proj", "k_proj", "gate_proj", "down_proj"])
def test_qwen14b_prefill_full_size(lin):
    """Qwen2.5-14B prefill linears, M = 4096, checked on 3 sampled rows."""
    wl = synth.WORKLOADS[2]
    name, N, K = wl.linears[lin]
    c = LinearCase(4096, K, N, wl.r, config=2, idx=lin).quantize_gpu()
    _fwd_check(c, rows=np.array([0, 1777, 4095]))


def test_qwen32b_stack_layer_shapes():
    """Qwen2.5-32B decode stack, M = 64, r = 64: the largest linear (gate_proj
    27648 x 5120) and down_proj (5120 x 27648) of one layer, 2 sampled rows."""
    wl = synth.WORKLOADS[3]
    for lin in (4, 6):
        name, N, K = wl.linears[lin]
        c = LinearCase(64, K, N, wl.r, config=3, layer=63, idx=lin).quantize_gpu()
        _fwd_check(c, rows=np.array([0, 63]))


@pytest.mark.parametrize("lin", [0, 6], ids=["q_proj", "down_proj"])
def test_qwen7b_backward_full_size(lin):
    """Qwen2.5-7B training backward, M = 8192, r = 32: dx on 2 rows, dA on 8
    columns, dB on 8 rows (each an exact sum over all 8192 tokens)."""
    wl = synth.WORKLOADS[4]
    name, N, K = wl.linears[lin]
    c = LinearCase(8192, K, N, wl.r, config=4, idx=lin).quantize_gpu()
    rng = np.random.default_rng(lin)
    _bwd_check(c, dx_rows=np.array([0, 8191]), dA_cols=np.sort(rng.choice(K, 8, replace=False)),
               dB_rows=np.sort(rng.choice(N, 8, replace=False)))


@pytest.mark.parametrize("M,K,N,r", [(1, 256, 128, 1), (8, 512, 1024, 8), (64, 3584, 3584, 32), (37, 1024, 384, 16),
                                     (64, 18944, 512, 32), (16, 2048, 18944, 32), (33, 768, 200, 5)])
def test_forward_without_t(M, K, N, r):
    """Decode shapes with no t output take the fused down-projection path."""
    c = LinearCase(M, K, N, r, config=9, idx=M * 7 + r).quantize_gpu()
    _fwd_check(c, rows=None if M * N <= 200_000 else np.arange(min(M, 4)), want_t=False)
