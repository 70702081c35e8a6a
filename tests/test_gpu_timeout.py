"""The tensor-core forward's bounded waits: with the withheld-arrival hook set, one
dequantizing warp of CTA 0 never signals its first stage, the MMA warp's wait runs
out (50 ms), and the call must report QERL_ERR_TIMEOUT through qerl_get_error while
the CUDA context stays usable.  Runs in a child process because the hook is read
once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
torch.cuda.set_device(0)
M, K, N, r = 8, 512, 256, 8
W = synth.weight(N, K, 1, "cuda")
codes, scales, ts = q.qerl_nvfp4_quantize(W)
assert q.get_error() == 0
x = synth.activations(M, K, 2, "cuda")
A = synth.lora_A(r, K, 3, "cuda")
B = synth.lora_B(N, r, 4, "cuda")
q.set_linear_algo(q.ALGO_TCGEN05)
q.qerl_nvfp4_lora_linear_fwd(x, codes, scales, ts, A, B, 2.0)
torch.cuda.synchronize()
print("first", q.get_error())
print("after", q.get_error())
q.set_linear_algo(q.ALGO_SIMT)
y = q.qerl_nvfp4_lora_linear_fwd(x, codes, scales, ts, A, B, 2.0)
torch.cuda.synchronize()
print("simt", q.get_error(), bool(torch.isfinite(y.float()).all()))
"""


def test_withheld_arrival_times_out_and_context_survives():
    env = dict(os.environ, QERL_TEST_WITHHOLD_ARRIVAL="1", PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = dict(l.split(" ", 1) for l in out.stdout.strip().splitlines())
    assert lines["first"] == "6"  # QERL_ERR_TIMEOUT
    assert lines["after"] == "0"  # qerl_get_error clears the latched status
    assert lines["simt"] == "0 True"
