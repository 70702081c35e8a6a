"""The forward with its token tiles shared across clusters of 1, 2 and 4 CTAs
(multicast) gives bit-identical results: only which CTA loads a tile changes,
not the arithmetic.  Each cluster size runs in its own process because the
override is read once per process."""
import hashlib
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import hashlib, torch
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
torch.cuda.set_device(0)
for (M, K, N, r) in [(8, 512, 1024, 8), (64, 3584, 3584, 32), (64, 18944, 512, 32), (200, 1024, 768, 16),
                     (1, 256, 384, 4), (300, 2048, 520, 64)]:
    W = synth.weight(N, K, 1, "cuda")
    codes, scales, ts = q.qerl_nvfp4_quantize(W)
    packed = q.qerl_nvfp4_pack_codes(codes)
    x = synth.activations(M, K, 2, "cuda")
    A = synth.lora_A(r, K, 3, "cuda")
    B = synth.lora_B(N, r, 4, "cuda")
    t = torch.zeros(M, r, device="cuda")
    y = q.qerl_nvfp4_lora_linear_fwd_packed(x, packed, scales, ts, A, B, 2.0, t_out=t)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    h = hashlib.sha256(y.view(torch.uint8).cpu().numpy().tobytes() + t.cpu().numpy().tobytes()).hexdigest()
    print(M, K, N, r, h)
"""


def _run(cluster):
    env = dict(os.environ, PYTHONPATH=ROOT)
    if cluster:
        env["QERL_TC_CLUSTER"] = str(cluster)
    out = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return out.stdout.strip().splitlines()


def test_cluster_sizes_agree_bit_for_bit():
    ref = _run(1)
    assert len(ref) == 6
    assert _run(2) == ref
    assert _run(4) == ref
    assert _run(0) == ref  # automatic choice
