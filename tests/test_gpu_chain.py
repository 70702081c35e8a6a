"""Chained launches: a sequence of calls where each input is the previous call's
output (norm -> linears -> norm -> linear) gives bit-identical results with
chaining on and off, including a weight quantized and packed right before its
first chained use."""
import pytest
import torch

import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth

pytestmark = pytest.mark.gpu

H, I, M, R = 512, 1536, 16, 16


def _weights(seed):
    out = []
    for i, (N, K) in enumerate([(H, H), (I, H), (H, I), (H, H)]):
        W = synth.weight(N, K, seed + 10 * i, "cuda")
        out.append((W, synth.lora_A(R, K, seed + 10 * i + 1, "cuda"), synth.lora_B(N, R, seed + 10 * i + 2, "cuda")))
    return out


def _sequence(weights, x, gamma, packed):
    fwd = q.qerl_nvfp4_lora_linear_fwd_packed if packed else q.qerl_nvfp4_lora_linear_fwd
    outs = []
    qw = []
    for W, A, B in weights:  # quantize (and pack) right before use, on the same stream
        codes, scales, ts = q.qerl_nvfp4_quantize(W)
        if packed:
            q.qerl_nvfp4_pack_codes(codes, out=codes)
        qw.append((codes, scales, ts, A, B))
    h = q.qerl_aqn_rmsnorm(x, gamma, 1e-6, 1e-2, 7, 3, 0)
    outs.append(h)
    a = fwd(h, *qw[0], 2.0)
    g = fwd(h, *qw[1], 2.0)
    d = fwd(g, *qw[2], 2.0)  # input written by the previous call
    h2 = q.qerl_aqn_rmsnorm(d, gamma, 1e-6, 1e-2, 7, 3, 1)
    e = fwd(h2, *qw[3], 2.0)
    outs += [a, g, d, h2, e]
    torch.cuda.synchronize()
    assert q.get_error() == 0
    return outs


@pytest.mark.parametrize("packed", [False, True], ids=["standard", "packed"])
def test_chained_matches_unchained(packed):
    weights = _weights(100)
    x = synth.activations(M, H, 5, "cuda")
    gamma = synth.norm_gamma(H, 6, "cuda")
    try:
        q.set_launch_chaining(False)
        ref = _sequence(weights, x, gamma, packed)
        q.set_launch_chaining(True)
        for _ in range(3):
            got = _sequence(weights, x, gamma, packed)
            for r_, g_ in zip(ref, got):
                assert torch.equal(r_, g_)
    finally:
        q.set_launch_chaining(True)


def test_chained_in_a_cuda_graph():
    weights = _weights(200)
    x = synth.activations(M, H, 8, "cuda")
    gamma = synth.norm_gamma(H, 9, "cuda")
    qw = []
    for W, A, B in weights:
        codes, scales, ts = q.qerl_nvfp4_quantize(W)
        qw.append((q.qerl_nvfp4_pack_codes(codes), scales, ts, A, B))
    torch.cuda.synchronize()
    bufs = [torch.empty(M, n, dtype=torch.bfloat16, device="cuda") for n in (H, H, I, H, H, H)]
    ws = q.workspace(q.OP_LINEAR_FWD, M, I, I, R)
    wsn = q.workspace(q.OP_AQN_RMSNORM, M, 0, H, 0)

    def step():
        q.qerl_aqn_rmsnorm(x, gamma, 1e-6, 1e-2, 7, 3, 0, y=bufs[0], ws=wsn)
        q.qerl_nvfp4_lora_linear_fwd_packed(bufs[0], *qw[0], 2.0, y=bufs[1], ws=ws)
        q.qerl_nvfp4_lora_linear_fwd_packed(bufs[0], *qw[1], 2.0, y=bufs[2], ws=ws)
        q.qerl_nvfp4_lora_linear_fwd_packed(bufs[2], *qw[2], 2.0, y=bufs[3], ws=ws)
        q.qerl_aqn_rmsnorm(bufs[3], gamma, 1e-6, 1e-2, 7, 3, 1, y=bufs[4], ws=wsn)
        q.qerl_nvfp4_lora_linear_fwd_packed(bufs[4], *qw[3], 2.0, y=bufs[5], ws=ws)

    q.set_launch_chaining(False)
    step()
    torch.cuda.synchronize()
    ref = [b.clone() for b in bufs]
    q.set_launch_chaining(True)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(5):
        for b in bufs:
            b.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert q.get_error() == 0
        for r_, b in zip(ref, bufs):
            assert torch.equal(r_, b)
