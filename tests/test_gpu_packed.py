"""The packed code layout: the permutation against the table the header states,
its inverse, and the forward/backward on packed codes against the oracle (which
reads the standard layout) and against the standard-layout entry points."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, LinearCase, assert_rel_rms, f64

pytestmark = pytest.mark.gpu

# The header's table: magnitude bits (m, e0, e1) of the even element of pair p
# start at MAG[p], its sign sits at SIGN[p]; the odd element adds 16.
MAG = [6, 3, 0, 9]
SIGN = [15, 12, 13, 14]


def pack_reference(codes: np.ndarray) -> np.ndarray:
    """Bit-by-bit restatement of the layout on little-endian 32-bit words."""
    w = codes.reshape(-1).view("<u4").astype(np.uint64)
    out = np.zeros_like(w)
    for i in range(8):
        p, hi = i // 2, 16 * (i % 2)
        nib = (w >> np.uint64(4 * i)) & np.uint64(15)
        for b in range(3):
            out |= ((nib >> np.uint64(b)) & np.uint64(1)) << np.uint64(MAG[p] + b + hi)
        out |= ((nib >> np.uint64(3)) & np.uint64(1)) << np.uint64(SIGN[p] + hi)
    return out.astype("<u4").view(np.uint8).reshape(codes.shape)


def test_layout_table_is_a_permutation():
    pos = sorted([MAG[p] + b + 16 * h for p in range(4) for b in range(3) for h in range(2)] +
                 [SIGN[p] + 16 * h for p in range(4) for h in range(2)])
    assert pos == list(range(32))


@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (128, 4096), (517, 2048)])
def test_pack_matches_table_and_unpack_inverts(N, K):
    g = torch.Generator().manual_seed(N * 7 + K)
    codes = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=g)
    dev = codes.cuda()
    packed = q.qerl_nvfp4_pack_codes(dev)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), pack_reference(codes.numpy()))
    back = q.qerl_nvfp4_unpack_codes(packed)
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), codes)
    inplace = dev.clone()
    q.qerl_nvfp4_pack_codes(inplace, out=inplace)
    torch.cuda.synchronize()
    assert torch.equal(inplace, packed)


def test_pack_rejects_overlap_and_bad_k():
    base = torch.zeros(512, dtype=torch.uint8, device="cuda")
    a, b = base[0:256].view(4, 64), base[16:272].view(4, 64)
    with pytest.raises(q.QerlError):
        q.qerl_nvfp4_pack_codes(a, out=b)
    assert q.lib().qerl_nvfp4_pack_codes(base.data_ptr(), 4, 24, base.data_ptr(), None) == 2  # QERL_ERR_SHAPE


def _case(M, K, N, r, idx):
    c = LinearCase(M, K, N, r, config=9, idx=idx).quantize_gpu()
    c.packed = q.qerl_nvfp4_pack_codes(c.codes)
    return c


@pytest.mark.parametrize("algo", [q.ALGO_AUTO, q.ALGO_SIMT], ids=["auto", "simt"])
@pytest.mark.parametrize("M,K,N,r", [(1, 256, 1, 1), (17, 512, 200, 8), (64, 1024, 384, 32), (130, 512, 136, 16),
                                     (3, 48, 33, 5), (257, 2048, 520, 64), (9, 4096, 128, 256)])
def test_forward_packed_matches_oracle_and_standard(algo, M, K, N, r):
    q.set_linear_algo(algo)
    try:
        c = _case(M, K, N, r, M + N)
        t = torch.empty(M, r, dtype=torch.float32, device="cuda")
        t2 = torch.empty(M, r, dtype=torch.float32, device="cuda")
        yp = q.qerl_nvfp4_lora_linear_fwd_packed(c.x, c.packed, c.scales, c.ts, c.A, c.B, c.s, t_out=t)
        ys = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s, t_out=t2)
        # without t (decode tiles take the fused down-projection)
        yp0 = q.qerl_nvfp4_lora_linear_fwd_packed(c.x, c.packed, c.scales, c.ts, c.A, c.B, c.s)
        ys0 = q.qerl_nvfp4_lora_linear_fwd(c.x, c.codes, c.scales, c.ts, c.A, c.B, c.s)
        torch.cuda.synchronize()
        assert q.get_error() == 0
    finally:
        q.set_linear_algo(q.ALGO_AUTO)
    # same arithmetic, only the code layout differs
    assert torch.equal(yp, ys)
    assert torch.equal(yp0, ys0)
    assert torch.equal(t, t2)
    oc, osc, ost = c.oracle_quant()
    ref, tref = oracle.lora_linear_fwd(synth.bits(c.x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s,
                                       want_t=True)
    assert_rel_rms(f64(yp), ref, LIN_TOL, "y")
    assert_rel_rms(f64(yp0), ref, LIN_TOL, "y without t")
    assert_rel_rms(f64(t), tref, 1e-5, "t")


QWEN7B = synth.WORKLOADS[1]


@pytest.mark.parametrize("lin", range(7), ids=[l[0] for l in QWEN7B.linears])
def test_forward_packed_qwen7b_decode_full_size(lin):
    name, N, K = QWEN7B.linears[lin]
    c = LinearCase(64, K, N, QWEN7B.r, config=1, idx=lin).quantize_gpu()
    packed = q.qerl_nvfp4_pack_codes(c.codes)
    y = q.qerl_nvfp4_lora_linear_fwd_packed(c.x, packed, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rows = np.sort(np.random.default_rng(lin).choice(64, 4, replace=False))
    oc, osc, ost = c.oracle_quant()
    ref = oracle.lora_linear_fwd(synth.bits(c.x), oc, osc, ost, synth.bits(c.A), synth.bits(c.B), c.s, rows=rows)
    assert_rel_rms(f64(y)[rows], ref, LIN_TOL, "y")


@pytest.mark.parametrize("M,K,N,r", [(20, 192, 100, 4), (70, 512, 257, 12), (130, 512, 256, 16), (300, 768, 192, 72)])
def test_backward_packed_matches_oracle(M, K, N, r):
    c = _case(M, K, N, r, 5)
    dx, dA, dB = q.qerl_nvfp4_lora_linear_bwd_packed(c.dy, c.x, c.packed, c.scales, c.ts, c.A, c.B, c.s)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    oc, osc, ost = c.oracle_quant()
    rdx, rdA, rdB = oracle.lora_linear_bwd(synth.bits(c.dy), synth.bits(c.x), oc, osc, ost, synth.bits(c.A),
                                           synth.bits(c.B), c.s)
    assert_rel_rms(f64(dx), rdx, LIN_TOL, "dx")
    assert_rel_rms(f64(dA), rdA, LIN_TOL, "dA")
    assert_rel_rms(f64(dB), rdB, LIN_TOL, "dB")
