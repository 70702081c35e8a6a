"""GPU parity of the NVFP4 quantizer and dequantizer against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LinearCase

pytestmark = pytest.mark.gpu


def _check(W, scale_round=0, ldw_pad=0):
    N, K = W.shape
    Wd = W.cuda()
    if ldw_pad:
        big = torch.zeros(N, K + ldw_pad, dtype=torch.bfloat16, device="cuda")
        big[:, :K] = Wd
        Wd = big[:, :K]
    codes, scales, ts = q.qerl_nvfp4_quantize(Wd, scale_round=scale_round)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    rc, oc, osc, ost = oracle.nvfp4_quantize(synth.bits(W), scale_mode=scale_round)
    assert rc == 0
    np.testing.assert_array_equal(scales.cpu().numpy(), osc)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    assert ts.cpu().numpy()[0] == ost  # bit-exact FP32 (no NaN here)
    return codes, scales, ts, oc, osc, ost


def test_config0_q_proj_bit_exact():
    _check(synth.weight(2048, 2048, synth.seed_of(0, 0, synth.T_W)))


@pytest.mark.parametrize("shape", [(1, 16), (33, 48), (7, 4096 + 16), (300, 160)])
@pytest.mark.parametrize("mode", [0, 1])
def test_ragged_shapes_and_modes(shape, mode):
    _check(synth.weight(*shape, seed=shape[0] * 31 + shape[1]), scale_round=mode)


def test_strided_rows():
    _check(synth.weight(64, 96, seed=5), ldw_pad=8)


def test_every_code_and_scale_round_trips():
    rows = []
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
    for sb in range(1, 127):
        rows.append([oracle.e2m1_value(c) * float(e4[sb]) * 2.0 ** -10 for c in range(16) if c != 8] +
                    [6 * float(e4[sb]) * 2.0 ** -10])
    W = torch.tensor(rows, dtype=torch.float64).to(torch.bfloat16)
    _check(W)
    _check(W, scale_round=1)


def test_zero_and_tiny_weights():
    _check(torch.zeros(4, 64, dtype=torch.bfloat16))
    tiny = torch.full((2, 32), 1e-39, dtype=torch.float32).to(torch.bfloat16)  # bf16 subnormal
    tiny[1, 3] = -3e-40
    _check(tiny)
    _check(synth.weight(16, 64, 3) * 1e-30)


def test_nonfinite_weight_latches_error():
    W = synth.weight(8, 64, 9).cuda()
    W[3, 17] = float("inf")
    codes, scales, ts = q.qerl_nvfp4_quantize(W)
    assert q.get_error() == 4
    assert torch.isnan(ts).all()
    assert q.get_error() == 0  # cleared on read


def test_full_size_gate_proj_bit_exact():
    """Qwen2.5-7B gate_proj 18944 x 3584 at full size, every byte."""
    c = LinearCase(1, 3584, 18944, 32, config=1, idx=4)
    codes, scales, ts = q.qerl_nvfp4_quantize(c.W)
    oc, osc, ost = c.oracle_quant()
    np.testing.assert_array_equal(scales.cpu().numpy(), osc)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    assert ts.cpu().numpy()[0] == ost


def test_dequantize_exact_and_scaled():
    W = synth.weight(40, 96, 21)
    codes, scales, ts, oc, osc, ost = _check(W)
    exact = q.qerl_nvfp4_dequantize(codes, scales, ts, 40, 96, apply_tensor_scale=False)
    ref = oracle.nvfp4_dequantize(oc, osc, 1.0, 40, 96)
    np.testing.assert_array_equal(exact.double().cpu().numpy(), ref)  # e2m1*e4m3 is exact in bf16
    scaled = q.qerl_nvfp4_dequantize(codes, scales, ts, 40, 96, apply_tensor_scale=True)
    ref_s = oracle.nvfp4_dequantize(oc, osc, ost, 40, 96)
    np.testing.assert_array_equal(scaled.float().cpu().numpy(),
                                  torch.from_numpy(ref_s).float().to(torch.bfloat16).float().numpy())
