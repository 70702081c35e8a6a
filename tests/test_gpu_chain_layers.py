"""GPU parity of the persistent decoder-layer chain (qerl_decoder_chain_*).

The chain per layer is N1(h0) -> q, k, v;  h1 = h0 + o(attn);  N2(h1) -> gate,
up;  m = silu(g) * u;  h2 = h1 + down(m), each linear an NVFP4 + LoRA forward
and N_i the AQN-RMSNorm, every activation carried in bf16.  Two oracle chains,
both built from the oracle's quantizer, linear forward, AQN noise and norm plus
plain fp64 glue (residual add, SwiGLU):

- unfused: a = bf16(N1(h0)) feeds the linear: the norm's textbook output
  rounded to bf16.  The norm's direct consumers q, k, v of the GPU chain match
  it within the linear tolerance: the GPU rounds the norm's output at another
  point (below), a rounding-level difference.  (Past gate/up, SwiGLU and down
  that difference has gone through three products, so the rest of the layer
  is checked against the fused reading.)
- fused (the reading the GPU implements): the norm's output enters the linear
  as xn = bf16(h * (gamma + sigma z)) and the linear's result is scaled per
  token by rs = 1 / sqrt(mean(h^2) + eps); each linear output is rounded to
  bf16, residual sums are rounded to bf16.  Deep chains are checked against
  this one: the two sides round at the same points, so their difference stays
  at the level of one linear's accumulation error instead of compounding a
  different rounding of every norm through the residual stream.

Compared outputs are the oracle's unrounded fp64 values; the rows each side
feeds forward are rounded to bf16.  Every token row is independent in the
chain, so the oracle runs on sampled rows at full sizes.

Tolerances: q, k, v are linear outputs: |got - ref| <= 1e-2 (|ref| + rms).  A
residual output h = bf16(h_prev + bf16(y)) adds, to that, one unit in the last
place of the summand y and one of h: both sides round y before the add, and two
y that agree within the linear tolerance may round to neighbouring bf16 values.

Deep chains: a one-ulp rounding difference in the residual stream of one layer
is carried by every later layer, so layer l of a long chain is checked with the
oracle's own input of that layer (the oracle chain run from the seeded input,
its rows written into the GPU's input), and the whole chain in one plan is
checked to equal, bit for bit, the same layers run one plan at a time."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_quantize_gb300 as q
from nvfp4_weight_only_quantize_gb300 import synth
from helpers import LIN_TOL, assert_rel_rms, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6
NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def bf16_round(a):
    """fp64 -> the nearest bf16 value (ties to even), as fp64."""
    a = np.asarray(a, np.float64)
    m, e = np.frexp(a)
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)


def to_bits(a):
    return (np.asarray(bf16_round(a), np.float32).view(np.uint32) >> 16).astype(np.uint16)


def from_bits(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


class Chain:
    """Seeded weights of L layers: packed NVFP4 on the GPU (quantized there) and,
    for the oracle, the same bf16 weights quantized by the oracle itself."""

    def __init__(self, L, M, H, NQ, NKV, I, r, cfg=11, device="cuda", keep_w=True):
        self.L, self.M, self.H, self.NQ, self.NKV, self.I, self.r = L, M, H, NQ, NKV, I, r
        shapes = {"q": (NQ, H), "k": (NKV, H), "v": (NKV, H), "o": (H, NQ), "gate": (I, H), "up": (I, H),
                  "down": (H, I)}
        self.layers, self.wbits, self._oq = [], [], {}
        for l in range(L):
            Ly, wb = {}, {}
            for i, nm in enumerate(NAMES):
                N, K = shapes[nm]
                base = synth.seed_of(cfg, l, 16 * i)
                W = synth.weight(N, K, base + synth.T_W, device)
                codes, scales, ts = q.qerl_nvfp4_quantize(W)
                q.qerl_nvfp4_pack_codes(codes, out=codes)
                A = synth.lora_A(r, K, base + synth.T_A, device)
                B = synth.lora_B(N, r, base + synth.T_B, device)
                Ly[nm] = (codes, scales, ts, A, B)
                wb[nm] = synth.bits(W) if keep_w else None
                del W
            Ly["gamma_attn"] = synth.norm_gamma(H, synth.seed_of(cfg, l, 200), device)
            Ly["gamma_mlp"] = synth.norm_gamma(H, synth.seed_of(cfg, l, 201), device)
            Ly["attn"] = synth.activations(M, NQ, synth.seed_of(cfg, l, 300), device)
            Ly["q_out"] = torch.empty(M, NQ, dtype=torch.bfloat16, device=device)
            Ly["k_out"] = torch.empty(M, NKV, dtype=torch.bfloat16, device=device)
            Ly["v_out"] = torch.empty(M, NKV, dtype=torch.bfloat16, device=device)
            self.layers.append(Ly)
            self.wbits.append(wb)
        self.x = synth.activations(M, H, synth.seed_of(cfg, 0, 400), device)

    def plan(self, first, last, x_in, x_out, s=2.0):
        return q.DecoderChain(self.layers[first:last], self.M, self.H, self.NQ, self.NKV, self.I, self.r, s, EPS,
                              x_in, x_out)

    def oracle_quant(self, l, nm):
        key = (l, nm)
        if key not in self._oq:
            rc, codes, scales, st = oracle.nvfp4_quantize(self.wbits[l][nm])
            assert rc == 0
            self._oq[key] = (codes, scales, st)
        return self._oq[key]

    def oracle_layer(self, l, h0_bits, rows, sigma, seed, step, s=2.0, fused=True):
        """Layer l (noise keys 2l, 2l + 1) on the token rows `rows`; h0_bits are
        those rows of the layer's input.  Returns fp64 q, k, v (unrounded) and
        h (rounded to bf16, as fed to the next layer)."""
        Ly = self.layers[l]
        H = self.H

        def lin(nm, xb):
            codes, scales, st = self.oracle_quant(l, nm)
            _, _, _, A, B = Ly[nm]
            return oracle.lora_linear_fwd(xb, codes, scales, st, synth.bits(A), synth.bits(B), s)

        def norm_then(h_bits, gamma, key, names):
            """The linears `names` on the norm of h (fused or unfused reading)."""
            if not fused:
                a = to_bits(oracle.aqn_rmsnorm(h_bits, synth.bits(gamma), EPS, sigma, seed, step, key))
                return [lin(nm, a) for nm in names]
            h = from_bits(h_bits)
            ns = from_bits(synth.bits(gamma)) + sigma * oracle.aqn_noise(H, seed, step, key)
            xn = to_bits(h * ns[None, :])
            rs = 1.0 / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + EPS)
            return [rs * lin(nm, xn) for nm in names]

        h0 = from_bits(h0_bits)
        out = dict(zip(("q", "k", "v"), norm_then(h0_bits, Ly["gamma_attn"], 2 * l, ("q", "k", "v"))))
        h1 = bf16_round(h0 + bf16_round(lin("o", synth.bits(Ly["attn"])[rows])))
        g, u = (bf16_round(t) for t in norm_then(to_bits(h1), Ly["gamma_mlp"], 2 * l + 1, ("gate", "up")))
        m = bf16_round(g / (1.0 + np.exp(-g)) * u)
        out["d"] = lin("down", to_bits(m))
        out["h"] = bf16_round(h1 + bf16_round(out["d"]))
        return out

    def oracle_chain(self, rows, sigma, seed, step, fused=True):
        """Every layer from the seeded input on the sampled rows; per-layer outputs."""
        h = synth.bits(self.x)[rows]
        outs = []
        for l in range(self.L):
            o = self.oracle_layer(l, h, rows, sigma, seed, step, fused=fused)
            outs.append(o)
            h = to_bits(o["h"])
        return outs


def ulp_bf16(v):
    """One unit in the last place of bf16 at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 7)


def assert_resid(got, ref, summand, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    bound = LIN_TOL * (np.abs(ref) + rms) + ulp_bf16(summand) + ulp_bf16(ref)
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside; worst at {i}: got {got[i]}, ref {ref[i]}, "
                             f"summand {np.asarray(summand)[i]}, rms {rms}")


def check_layer(ch, l, h_in_bits, rows, sigma, seed, step, fused, what, resid=True):
    """GPU layer l alone (a one-layer plan, noise keys of layer l) on an input
    whose sampled rows are the oracle's h_in_bits, against the oracle's layer l."""
    x = ch.x.clone()
    x[torch.as_tensor(rows)] = torch.from_numpy(h_in_bits.astype(np.int16)).view(torch.bfloat16).to(x.device)
    out = torch.empty_like(x)
    pl = ch.plan(l, l + 1, x, out)
    pl.run(sigma, seed, step, first_layer=l)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    ref = ch.oracle_layer(l, h_in_bits, rows, sigma, seed, step, fused=fused)
    for nm in ("q", "k", "v"):
        assert_rel_rms(f64(ch.layers[l][nm + "_out"])[rows], ref[nm], LIN_TOL, f"{what} layer {l} {nm}")
    if resid:
        assert_resid(f64(out)[rows], ref["h"], ref["d"], f"{what} layer {l} h")
    pl.close()
    return ref


def check_chain(ch, rows, sigma, seed, step, check_layers, what, fused=True, compose=True):
    """The whole chain in one plan; each layer in check_layers against the oracle
    (fed the oracle chain's input of that layer); the one-plan result equal to
    the layer-by-layer plans bit for bit."""
    out = torch.empty(ch.M, ch.H, dtype=torch.bfloat16, device="cuda")
    pl = ch.plan(0, ch.L, ch.x, out)
    pl.run(sigma, seed, step)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    qkv_whole = [[ch.layers[l][nm + "_out"].clone() for nm in ("q", "k", "v")] for l in range(ch.L)]
    full = out.clone()
    # a second run of the same plan (its counters are left clean) gives the same bits
    out.zero_()
    pl.run(sigma, seed, step)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    assert torch.equal(out, full)
    pl.close()
    if compose:
        h = ch.x
        for l in range(ch.L):
            o = torch.empty_like(h)
            p1 = ch.plan(l, l + 1, h, o)
            p1.run(sigma, seed, step, first_layer=l)
            torch.cuda.synchronize()
            assert q.get_error() == 0
            p1.close()
            for i, nm in enumerate(("q", "k", "v")):
                assert torch.equal(ch.layers[l][nm + "_out"], qkv_whole[l][i]), f"{what}: layer {l} {nm} differs"
            h = o
        assert torch.equal(h, full), f"{what}: one plan differs from the layer-by-layer plans"
    # oracle chain from the seeded input; each checked layer fed its oracle input
    hb = synth.bits(ch.x)[rows]
    for l in range(ch.L):
        if l in check_layers:
            ref = check_layer(ch, l, hb, rows, sigma, seed, step, fused, what, resid=fused)
        else:
            ref = ch.oracle_layer(l, hb, rows, sigma, seed, step, fused=fused)
        hb = to_bits(ref["h"])
    return full


@pytest.mark.parametrize("L,M,H,NQ,NKV,I,r", [(3, 5, 512, 512, 128, 768, 16), (2, 64, 256, 256, 128, 512, 64),
                                              (2, 33, 768, 768, 256, 1280, 32), (1, 1, 256, 256, 128, 256, 8)])
def test_chain_small_every_layer(L, M, H, NQ, NKV, I, r):
    """Every layer of small chains, every token."""
    ch = Chain(L, M, H, NQ, NKV, I, r)
    check_chain(ch, np.arange(M), 1e-2, 7, 3, range(L), "small")


def test_chain_64_layers():
    """A 64-layer chain (the depth of the Qwen2.5-32B stack) at reduced width,
    M = 64, r = 64: layers 0 and 63 against the oracle on sampled rows, the whole
    chain against 64 one-layer plans bit for bit."""
    ch = Chain(64, 64, 512, 512, 128, 1024, 64, cfg=13)
    check_chain(ch, np.array([0, 40, 63]), 1e-2, 5, 2, (0, 63), "64 layers")


def test_chain_qwen32b_two_layers():
    """Two Qwen2.5-32B decoder layers (hidden 5120, kv 1024, intermediate 27648),
    M = 64, r = 64, on sampled rows."""
    ch = Chain(2, 64, 5120, 5120, 1024, 27648, 64, cfg=3)
    check_chain(ch, np.array([0, 63]), 1e-2, 3, 1, (0, 1), "qwen2.5-32b")


@pytest.mark.parametrize("fused", [True, False], ids=["fused_reading", "unfused_norm"])
def test_chain_qwen7b_layer(fused):
    """One Qwen2.5-7B decoder layer at M = 64, r = 32 (the bench's decode step),
    against both oracle chains."""
    ch = Chain(1, 64, 3584, 3584, 512, 18944, 32, cfg=1)
    check_chain(ch, np.array([0, 37, 63]), 1e-2, 1, 0, (0,), "qwen2.5-7b", fused=fused, compose=False)


@pytest.mark.parametrize("M,r", [(5, 16), (64, 64)])
def test_chain_one_layer_matches_unfused_norm(M, r):
    """One small layer, every token, against the textbook norm -> bf16 -> linear."""
    ch = Chain(1, M, 512, 512, 128, 768, r, cfg=14)
    check_chain(ch, np.arange(M), 1e-2, 7, 3, (0,), "unfused", fused=False, compose=False)
