"""Seeded synthetic inputs shaped like Qwen2.5 decoder-layer linears.

This module only draws random tensors; it holds none of the method's arithmetic
(no quantization, no matmul, no normalisation).  The same tensors feed the CUDA
library and the CPU oracle, so both sides see identical bytes.

Distributions (the pages run RL on Qwen2.5 3B-32B checkpoints; these stand in
for those weights and for the prompts, which are not used):
  W  ~ N(0, 0.02) with exactly round(0.001*N*K) positions, drawn without
       replacement, multiplied by 10 ("0.1 % outliers"), then rounded to bf16;
  x  ~ N(0, 1) bf16;   dy ~ N(0, 0.01) bf16 (std 1e-2);
  A  ~ U(-1/sqrt(K), 1/sqrt(K)) bf16 [r, K];   B ~ N(0, 0.01) bf16 [N, r];
  gamma = 1 + 0.1*N(0, 1) bf16.
Seeds: seed(config, layer, tensor) = config*1_000_003 + layer*1009 + tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

T_W, T_X, T_A, T_B, T_GAMMA, T_DY = range(6)


def seed_of(config: int, layer: int, tensor: int) -> int:
    return config * 1_000_003 + layer * 1009 + tensor


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weight(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    W = torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02
    n_out = round(0.001 * N * K)
    if n_out:
        idx = torch.randperm(N * K, generator=g, device=device)[:n_out]
        W.view(-1)[idx] *= 10.0
    return W.to(torch.bfloat16)


def activations(M: int, K: int, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(M, K, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def lora_A(r: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    u = torch.rand(r, K, generator=g, device=device, dtype=torch.float32)
    return ((u * 2.0 - 1.0) / math.sqrt(K)).to(torch.bfloat16)


def lora_B(N: int, r: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(N, r, generator=g, device=device, dtype=torch.float32) * 0.01).to(torch.bfloat16)


def norm_gamma(H: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (1.0 + 0.1 * torch.randn(H, generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@dataclass
class Workload:
    """One named workload: linears as (name, N_out, K_in), token count(s), rank."""
    name: str
    linears: list
    M: list
    r: int
    hidden: int
    lora_scale: float = 2.0
    layers: int = 1
    sigma: tuple = (1e-2, 5e-4)
    extra: dict = field(default_factory=dict)


def _layer(hidden: int, q: int, kv: int, inter: int):
    return [("q_proj", q, hidden), ("k_proj", kv, hidden), ("v_proj", kv, hidden),
            ("o_proj", hidden, q), ("gate_proj", inter, hidden), ("up_proj", inter, hidden),
            ("down_proj", hidden, inter)]


WORKLOADS = {
    # 0: one Qwen2.5-3B q_proj, 16 tokens, r = 16, seed 0.
    0: Workload("qwen2.5-3b q_proj 2048x2048, M=16, r=16", [("q_proj", 2048, 2048)], [16], 16, 2048),
    # 1: Qwen2.5-7B decoder layer in rollout decode.
    1: Workload("qwen2.5-7b decoder layer decode, M in {1,8,64}, r=32",
                _layer(3584, 3584, 512, 18944), [1, 8, 64], 32, 3584),
    # 2: Qwen2.5-14B prefill, 8 prompts x 512 tokens.
    2: Workload("qwen2.5-14b prefill, M=4096, r=32", _layer(5120, 5120, 1024, 13824), [4096], 32, 5120),
    # 3: Qwen2.5-32B 64-layer decode stack, 64 tokens, r = 64.
    3: Workload("qwen2.5-32b 64-layer decode stack, M=64, r=64", _layer(5120, 5120, 1024, 27648),
                [64], 64, 5120, layers=64),
    # 4: Qwen2.5-7B training backward, 8192 tokens.
    4: Workload("qwen2.5-7b backward, M=8192, r=32", _layer(3584, 3584, 512, 18944), [8192], 32, 3584),
}
