"""Grouped forward (linears sharing x) against the oracle, group by group: the
one-launch tensor-core path (fused and unfused down-projection, decode and
many-token tiles, packed and standard codes, ragged N) and the
one-after-the-other fallback."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu


def _groups(M, K, Ns, r, packed, seed):
    cases = [LinearCase(M, K, N, r, config=9, idx=seed + i).quantize_gpu() for i, N in enumerate(Ns)]
    x = cases[0].x
    gs = []
    for c in cases:
        codes = q.qerl_nvfp4_pack_codes(c.codes) if packed else c.codes
        gs.append((codes, c.scales, c.ts, c.A, c.B))
    return cases, x, gs


def _check(cases, x, ys, rows=None, t_outs=None):
    for i, c in enumerate(cases):
        oc, osc, ost = c.oracle_quant()
        ref, tref = oracle.lora_linear_fwd(synth.bits(x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s,
                                           rows=rows, want_t=True)
        got = f64(ys[i]) if rows is None else f64(ys[i])[rows]
        assert_rel_rms(got, ref, LIN_TOL, f"y[{i}]")
        if t_outs is not None and t_outs[i] is not None:
            tg = f64(t_outs[i]) if rows is None else f64(t_outs[i])[rows]
            assert_rel_rms(tg, tref, 1e-5, f"t[{i}]")


@pytest.mark.parametrize("packed", [False, True], ids=["standard", "packed"])
@pytest.mark.parametrize("M,K,Ns,r", [(13, 512, [200, 72, 384], 5), (64, 1024, [512, 128], 32), (1, 256, [128, 256, 64], 16),
                                      (40, 768, [1000], 8)])
def test_grouped_matches_oracle(packed, M, K, Ns, r):
    cases, x, gs = _groups(M, K, Ns, r, packed, seed=len(Ns) * 10 + M)
    ys = q.qerl_nvfp4_lora_linear_fwd_grouped(x, gs, 2.0, packed=packed)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    # (each case has its own x in LinearCase; the groups share the first one)
    for c in cases:
        c.x = x
    _check(cases, x, ys)


def test_grouped_with_t_outputs():
    M, K, Ns, r = 24, 512, [256, 136], 12
    cases, x, gs = _groups(M, K, Ns, r, True, seed=77)
    for c in cases:
        c.x = x
    t_outs = [torch.empty(M, r, device="cuda"), None]
    ys = q.qerl_nvfp4_lora_linear_fwd_grouped(x, gs, 2.0, packed=True, t_outs=t_outs)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    _check(cases, x, ys, t_outs=t_outs)


@pytest.mark.parametrize("M,Ns", [(100, [256, 128]), (300, [136, 256, 64]), (8, [128, 128, 128, 256]),
                                  (200, [128, 256, 64]), (1000, [256, 128, 128]), (256, [256, 256]),
                                  (512, [512, 128, 128])])
def test_grouped_many_tokens_and_many_groups(M, Ns):
    """More than 64 tokens: one launch, one down-projection pass for all groups;
    more than three groups: the groups run one after the other.  Group tile
    counts of 1 + 2 + 1 check that every CTA picks its own group's maps."""
    K, r = 512, 8
    cases, x, gs = _groups(M, K, Ns, r, False, seed=5)
    for c in cases:
        c.x = x
    ys = q.qerl_nvfp4_lora_linear_fwd_grouped(x, gs, 2.0)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    _check(cases, x, ys)


QWEN7B = synth.WORKLOADS[1]


@pytest.mark.parametrize("names", [("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj")], ids=["qkv", "gate_up"])
@pytest.mark.parametrize("M", [1, 64])
def test_grouped_qwen7b_decode(names, M):
    lins = {n: (N, K) for n, N, K in QWEN7B.linears}
    K = lins[names[0]][1]
    cases = [LinearCase(M, K, lins[n][0], QWEN7B.r, config=1, idx=i).quantize_gpu() for i, n in enumerate(names)]
    x = cases[0].x
    for c in cases:
        c.x = x
    gs = [(q.qerl_nvfp4_pack_codes(c.codes), c.scales, c.ts, c.A, c.B) for c in cases]
    ys = q.qerl_nvfp4_lora_linear_fwd_grouped(x, gs, QWEN7B.lora_scale, packed=True)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rows = np.arange(M) if M <= 2 else np.array([0, 31, 63])
    _check(cases, x, ys, rows=rows)
