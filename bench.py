"""Benchmark of the NVFP4 weight-only LoRA decode layer (Qwen2.5-7B shapes).

One step = one decoder layer of rollout decode through the library:
  AQN-RMSNorm(h) -> q_proj, k_proj, v_proj -> o_proj(attention stand-in)
  -> AQN-RMSNorm -> gate_proj, up_proj -> down_proj(up output),
M = 64 tokens, LoRA r = 32 on every linear.  Attention and SwiGLU are not part of
the path; o_proj takes a random bf16 stand-in for the attention output and
down_proj takes up_proj's output.  Weights rotate over several layer copies
whose NVFP4 bytes exceed L2, so every step streams its weights from HBM.

Metric: HBM GB/s of algorithmic bytes, N*K*0.5625 + 4 + 2*r*(N+K) per linear
(NVFP4 weight + tensor scale + bf16 LoRA), activations excluded.
Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


# DRAM bytes (read + write) per launch of the forward kernel, from one ncu capture
# of the decode step (the tc_fwd capture summarised under profiles/) of
# csrc/linear_tc.cu with this sha256 prefix; reported as roofline.traffic only
# while the source still matches.
NCU_KERNEL_SHA = "d2196cbf4bdd07bb"
NCU_DRAM_BYTES = {"gate_proj": 39.934208e6, "up_proj": 39.936512e6, "down_proj": 42.134272e6}


def ncu_traffic(name):
    import hashlib
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "nvfp4_weight_only_quantize_gb300", "csrc",
                       "linear_tc.cu")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return NCU_DRAM_BYTES.get(name) if sha == NCU_KERNEL_SHA else None


def linear_bytes(N, K, r):
    return N * K * 0.5625 + 4 + 2 * r * (N + K)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ ranks
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def combine_ranks(local_seconds: float, local_units: float):
    """(max time over ranks, total units over ranks); replicas run independently."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_seconds, local_units
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([s.strip() for s in line.split(",")])

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sms = [float(r[0]) for r in self.rows if len(r) >= 7 and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) >= 7 and r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) >= 7:
                for n, v in zip(names, r[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------------------ our arm
class DecodeLayer:
    """NVFP4 weights + LoRA adapters + norm scales of n_copies Qwen2.5-7B layers."""

    def __init__(self, wl, n_copies, device, packed=True):
        import nvfp4_weight_only_quantize_gb300 as q
        from nvfp4_weight_only_quantize_gb300 import synth
        self.q, self.wl, self.copies = q, wl, []
        self.packed = packed
        self.fwd = q.qerl_nvfp4_lora_linear_fwd_packed if packed else q.qerl_nvfp4_lora_linear_fwd
        for c in range(n_copies):
            lins = []
            for i, (name, N, K) in enumerate(wl.linears):
                base = synth.seed_of(1, c, 16 * i)
                W = synth.weight(N, K, base + synth.T_W, device)
                codes, scales, ts = q.qerl_nvfp4_quantize(W)
                del W
                if packed:  # once, when the frozen weight is loaded
                    q.qerl_nvfp4_pack_codes(codes, out=codes)
                A = synth.lora_A(wl.r, K, base + synth.T_A, device)
                B = synth.lora_B(N, wl.r, base + synth.T_B, device)
                lins.append((name, N, K, codes, scales, ts, A, B))
            gammas = [synth.norm_gamma(wl.hidden, synth.seed_of(1, c, 200 + j), device) for j in range(2)]
            self.copies.append((lins, gammas))
        torch.cuda.synchronize()
        self.bytes_per_step = sum(linear_bytes(N, K, wl.r) for _, N, K in wl.linears)

    def buffers(self, M, device):
        wl = self.wl
        outs = {name: torch.empty(M, N, dtype=torch.bfloat16, device=device) for name, N, K in wl.linears}
        ws_lin = max(self.q.workspace_bytes(self.q.OP_LINEAR_FWD, M, N, K, wl.r) for _, N, K in wl.linears)
        Nof = {n: N for n, N, K in wl.linears}
        for names in (("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj")):
            ws_lin = max(ws_lin, self.q.grouped_ws_bytes(M, wl.hidden, wl.r, [Nof[n] for n in names]))
        return dict(outs=outs, h1=torch.empty(M, wl.hidden, dtype=torch.bfloat16, device=device),
                    h2=torch.empty(M, wl.hidden, dtype=torch.bfloat16, device=device),
                    ws=torch.empty(max(ws_lin, 1), dtype=torch.uint8, device=device),
                    ws_side=torch.empty(max(ws_lin, 1), dtype=torch.uint8, device=device),
                    side=torch.cuda.Stream(device=device),
                    ws_norm=self.q.workspace(self.q.OP_AQN_RMSNORM, M, 0, wl.hidden, 0, device))

    def step(self, copy, x, attn, buf, sigma, step_idx):
        """One decoder layer: norm -> q|k|v (one grouped call) -> o -> norm ->
        gate and up (both read the norm's output: up runs on a second stream
        with its own workspace, joined before down) -> down.  Attention and
        SwiGLU are not part of this step (synthetic attention output; down
        reads up's output)."""
        q = self.q
        lins, gammas = self.copies[copy]
        by = {l[0]: l for l in lins}
        o = buf["outs"]
        s = self.wl.lora_scale

        def group(names, xin):
            gs = [by[n][3:8] for n in names]
            q.qerl_nvfp4_lora_linear_fwd_grouped(xin, gs, s, packed=self.packed, ys=[o[n] for n in names],
                                                 ws=buf["ws"])

        def single(name, xin, ws="ws"):
            _, N, K, codes, scales, ts, A, B = by[name]
            self.fwd(xin, codes, scales, ts, A, B, s, y=o[name], ws=buf[ws])

        q.qerl_aqn_rmsnorm(x, gammas[0], 1e-6, sigma, 1, step_idx, 2 * copy, y=buf["h1"], ws=buf["ws_norm"])
        group(("q_proj", "k_proj", "v_proj"), buf["h1"])
        single("o_proj", attn)
        q.qerl_aqn_rmsnorm(o["o_proj"], gammas[1], 1e-6, sigma, 1, step_idx, 2 * copy + 1, y=buf["h2"],
                           ws=buf["ws_norm"])
        # gate and up stay separate calls (grouped they need two waves of
        # one-tile CTAs over the SMs, which measured slower); up runs on a
        # second stream, so its CTAs take each SM as gate's leave it instead of
        # waiting for the whole of gate
        cur, side = torch.cuda.current_stream(), buf["side"]
        side.wait_stream(cur)
        single("gate_proj", buf["h2"])
        with torch.cuda.stream(side):
            single("up_proj", buf["h2"], ws="ws_side")
        cur.wait_stream(side)
        single("down_proj", o["up_proj"])
        return o["down_proj"]


def _graph(fn):
    """Capture fn() into a CUDA graph (on a side stream, as torch requires)."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside capture (sets function attributes, builds nothing new)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def _time_graph(g, reps):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def run_ours(args, rank, world, local_rank):
    import nvfp4_weight_only_quantize_gb300 as q
    from nvfp4_weight_only_quantize_gb300 import synth
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = synth.WORKLOADS[1]
    M = args.M
    per_copy = sum(N * K * 0.5625 for _, N, K in wl.linears)
    n_copies = max(2, int(3 * L2_BYTES // per_copy) + 1)
    layer = DecodeLayer(wl, n_copies, dev, packed=args.codes == "packed")
    buf = layer.buffers(M, dev)
    x = synth.activations(M, wl.hidden, synth.seed_of(1, 0, synth.T_X), dev)
    attn = synth.activations(M, wl.hidden, synth.seed_of(1, 1, synth.T_X), dev)
    sigma = q.qerl_aqn_sigma(0, 1000, wl.sigma[0], wl.sigma[1], 10)

    # One graph per weight copy: a whole decoder-layer step each.
    n0 = q.launch_count()
    layer.step(0, x, attn, buf, sigma, 0)
    torch.cuda.synchronize()
    kernels_per_step = q.launch_count() - n0
    graphs = [_graph(lambda c=c: layer.step(c, x, attn, buf, sigma, c)) for c in range(n_copies)]

    clocks = ClockSampler(torch.cuda.current_device()).start()
    t_start = time.perf_counter()
    i = 0
    while i < args.warmup or time.perf_counter() - t_start < 1.5:  # >= W steps and >= 1.5 s under load
        graphs[i % n_copies].replay()
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert q.get_error() == 0

    # --- device-resident timed region: exactly K steps
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.profile_region:  # lets `ncu --profile-from-start off` see only the timed steps
        torch.cuda.cudart().cudaProfilerStart()
    t0.record()
    for i in range(args.steps):
        graphs[i % n_copies].replay()
    t1.record()
    torch.cuda.synchronize()
    if args.profile_region:
        torch.cuda.cudart().cudaProfilerStop()
    barrier()
    clk = clocks.stop()
    assert q.get_error() == 0
    secs = t0.elapsed_time(t1) / 1e3
    max_secs, total_units = combine_ranks(secs, layer.bytes_per_step * args.steps)
    value = total_units / max_secs / 1e9

    # --- each linear alone: a graph of that linear over all weight copies
    per_linear = {}
    for li, (name, N, K) in enumerate(wl.linears):
        xin = torch.empty(M, K, dtype=torch.bfloat16, device=dev).normal_()
        yout = torch.empty(M, N, dtype=torch.bfloat16, device=dev)

        def run_lin(li=li, xin=xin, yout=yout):
            for c in range(n_copies):
                _, _, _, codes, scales, ts, A, B = layer.copies[c][0][li]
                layer.fwd(xin, codes, scales, ts, A, B, wl.lora_scale, y=yout, ws=buf["ws"])
        g = _graph(run_lin)
        _time_graph(g, 3)
        reps = 20
        us = _time_graph(g, reps) / (reps * n_copies) * 1e6
        per_linear[name] = {"us": round(us, 2), "GBps": round(linear_bytes(N, K, wl.r) / us / 1e3, 1)}

    # --- end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and reads its output back.  Two buffer
    # sets alternate, so that step i + 1's inputs are copied in (one copy
    # stream) and step i - 1's output is read back (another) while step i
    # computes; a set is reused only after the step that last used it finished.
    xh = x.cpu().pin_memory()
    ah = attn.cpu().pin_memory()
    sets = []
    for p_ in range(2):
        bset = buf if p_ == 0 else layer.buffers(M, dev)
        xs = x if p_ == 0 else torch.empty_like(x)
        ats = attn if p_ == 0 else torch.empty_like(attn)
        gs = graphs if p_ == 0 else [_graph(lambda c=c, b_=bset, x_=xs, a_=ats: layer.step(c, x_, a_, b_, sigma, c))
                                     for c in range(n_copies)]
        sets.append(dict(x=xs, attn=ats, graphs=gs, out=bset["outs"]["down_proj"],
                         yh=torch.empty(M, wl.hidden, dtype=torch.bfloat16).pin_memory(),
                         loaded=torch.cuda.Event(), done=torch.cuda.Event(), read=torch.cuda.Event()))
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d.wait_stream(comp)
    d2h.wait_stream(comp)
    for i in range(args.steps):
        st_ = sets[i % 2]
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(st_["done"])  # the set's previous step has finished
            st_["x"].copy_(xh, non_blocking=True)
            st_["attn"].copy_(ah, non_blocking=True)
            st_["loaded"].record(h2d)
        comp.wait_event(st_["loaded"])
        if i >= 2:
            comp.wait_event(st_["read"])  # the set's previous output has been read back
        st_["graphs"][i % n_copies].replay()
        st_["done"].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(st_["done"])
            st_["yh"].copy_(st_["out"], non_blocking=True)
            st_["read"].record(d2h)
    comp.wait_stream(d2h)
    comp.wait_stream(h2d)
    e1.record(comp)
    torch.cuda.synchronize()
    assert q.get_error() == 0
    e2e_secs, e2e_units = combine_ranks(e0.elapsed_time(e1) / 1e3, layer.bytes_per_step * args.steps)

    hbm, bf16, bf16_sus, peak_kind = peaks()
    dom = max(per_linear, key=lambda n: per_linear[n]["us"])
    dN, dK = [(N, K) for n, N, K in wl.linears if n == dom][0]
    ach = linear_bytes(dN, dK, wl.r) / (per_linear[dom]["us"] / 1e6) / 1e9
    ms_step = max_secs / args.steps * 1e3
    line = {
        "metric": "NVFP4+LoRA linear decode HBM GB/s (Qwen2.5-7B decoder layer)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 activations x nvfp4 weights, fp32 accumulate", "data": "synthetic",
        "config": {"workload": wl.name + f"; step at M={M}", "tokens_per_step": M, "lora_rank": wl.r,
                   "layer_copies_rotated": n_copies,
                   "l2": f"inputs larger than L2: {n_copies} rotating layer copies, "
                         f"{n_copies * per_copy / 2**20:.0f} MiB NVFP4 > 129 MiB L2",
                   "launch": "one CUDA graph per step (per weight copy); q|k|v as one grouped call; up_proj on a "
                             "second stream beside gate_proj",
                   "codes": args.codes + " layout (packed once when the weights are loaded)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": round(M * args.steps * world / max_secs, 1),
        "pct_of_hbm_peak": round(100 * value / world / hbm, 2),
        "per_linear": per_linear,
        "roofline": {"bound": "hbm", "kernel": f"linear fwd {dom} {dN}x{dK} (M={M}, r={wl.r})",
                     "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)", "traffic": ncu_traffic(dom),
                     "algorithmic_bytes": linear_bytes(dN, dK, wl.r)},
        "e2e": {"value": round(e2e_units / e2e_secs / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": 2 * M * wl.hidden * 2, "d2h_bytes_per_step": M * wl.hidden * 2},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clk,
    }
    if not args.no_rows:
        del graphs, layer, buf
        torch.cuda.empty_cache()
        line["rows"] = other_rows(dev)
        line["rows"].update(decode_rows(dev))
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, M, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the other rows
def _time_fn(fn, reps, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


SWEEP_RANKS = (8, 16, 32, 64, 128)


def rank_sweep(dev):
    """LoRA-rank sweep of the forward, and the same linear with 16-bit weights.
    Decode: Qwen2.5-7B gate_proj 18944 x 3584 at M = 64, four weight copies
    rotated in one CUDA graph (152 MB NVFP4, 543 MB bf16: both above L2).
    Prefill: Qwen2.5-14B q_proj 5120 x 5120 at M = 4096.  The 16-bit arm is
    y = x W^T + s (x A^T) B^T in torch (cuBLAS) with W the dequantized weight of
    the same codes rounded to bf16, so both arms compute the same product."""
    import nvfp4_weight_only_quantize_gb300 as q
    from nvfp4_weight_only_quantize_gb300 import synth
    out = {}
    for tag, (N, K, M, n_copies) in (("decode", (18944, 3584, 64, 4)), ("prefill", (5120, 5120, 4096, 1))):
        x = synth.activations(M, K, 70, dev)
        qw, w16 = [], []
        for c in range(n_copies):
            W = synth.weight(N, K, 71 + c, dev)
            codes, sc, ts = q.qerl_nvfp4_quantize(W)
            w16.append(q.qerl_nvfp4_dequantize(codes, sc, ts, N, K))  # bf16, tensor scale applied
            del W
            q.qerl_nvfp4_pack_codes(codes, out=codes)
            qw.append((codes, sc, ts))
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        res = {}
        for r in SWEEP_RANKS:
            lora = [(synth.lora_A(r, K, 80 + c, dev), synth.lora_B(N, r, 90 + c, dev)) for c in range(n_copies)]
            ws = q.workspace(q.OP_LINEAR_FWD, M, N, K, r, dev)

            def ours():
                for (codes, sc, ts), (A, B) in zip(qw, lora):
                    q.qerl_nvfp4_lora_linear_fwd_packed(x, codes, sc, ts, A, B, 2.0, y=y, ws=ws)

            def bf16():
                for W16, (A, B) in zip(w16, lora):
                    torch.mm(x, W16.t(), out=y)
                    y.add_(torch.mm(torch.mm(x, A.t()), B.t()), alpha=2.0)

            reps = 20 if tag == "decode" else 5
            us = {}
            for arm, fn in (("nvfp4", ours), ("bf16", bf16)):
                g = _graph(fn)
                _time_graph(g, 3)
                us[arm] = _time_graph(g, reps) / (reps * n_copies) * 1e6
                del g
            fl = 2.0 * M * N * K + 2.0 * M * r * (N + K)
            if tag == "decode":
                res[r] = {"us": round(us["nvfp4"], 2), "GBps": round(linear_bytes(N, K, r) / us["nvfp4"] / 1e3, 1),
                          "bf16_us": round(us["bf16"], 2),
                          "bf16_GBps": round((2.0 * N * K + 2 * r * (N + K)) / us["bf16"] / 1e3, 1),
                          "speedup_vs_bf16": round(us["bf16"] / us["nvfp4"], 3)}
            else:
                res[r] = {"us": round(us["nvfp4"], 1), "TFLOPs": round(fl / us["nvfp4"] / 1e6, 1),
                          "bf16_us": round(us["bf16"], 1), "bf16_TFLOPs": round(fl / us["bf16"] / 1e6, 1),
                          "speedup_vs_bf16": round(us["bf16"] / us["nvfp4"], 3)}
        out[tag] = {"workload": (f"qwen2.5-7b gate_proj {N}x{K}, M={M}, {n_copies} rotated weight copies"
                                 if tag == "decode" else f"qwen2.5-14b q_proj {N}x{K}, M={M}"),
                    "by_rank": res}
        del qw, w16, x, y
        torch.cuda.synchronize()
    return out


def _chain_layers(q, synth, L, M, H, NQ, NKV, I, r, cfg, dev):
    """L distinct decoder layers (packed NVFP4 + LoRA) for the chain kernel."""
    shapes = {"q": (NQ, H), "k": (NKV, H), "v": (NKV, H), "o": (H, NQ), "gate": (I, H), "up": (I, H), "down": (H, I)}
    layers = []
    for l in range(L):
        Ly = {}
        for i, nm in enumerate(("q", "k", "v", "o", "gate", "up", "down")):
            N, K = shapes[nm]
            base = synth.seed_of(cfg, l, 16 * i)
            W = synth.weight(N, K, base + synth.T_W, dev)
            codes, scales, ts = q.qerl_nvfp4_quantize(W)
            del W
            q.qerl_nvfp4_pack_codes(codes, out=codes)
            Ly[nm] = (codes, scales, ts, synth.lora_A(r, K, base + synth.T_A, dev),
                      synth.lora_B(N, r, base + synth.T_B, dev))
        Ly["gamma_attn"] = synth.norm_gamma(H, synth.seed_of(cfg, l, 200), dev)
        Ly["gamma_mlp"] = synth.norm_gamma(H, synth.seed_of(cfg, l, 201), dev)
        Ly["attn"] = synth.activations(M, NQ, synth.seed_of(cfg, l, 300), dev)
        layers.append(Ly)
    torch.cuda.synchronize()
    return layers


def _time_stack_per_linear(q, lay, x, H, NKV, I, wl, sigma):
    """Seconds per step of the decoder stack `lay` (M = 64) run as the library's
    per-linear calls and glue in one CUDA graph."""
    M, r, s, dev = x.shape[0], wl.r, wl.lora_scale, x.device
    bf = dict(dtype=torch.bfloat16, device=dev)
    h, n = torch.empty(M, H, **bf), torch.empty(M, H, **bf)
    qo, ko, vo = torch.empty(M, H, **bf), torch.empty(M, NKV, **bf), torch.empty(M, NKV, **bf)
    o, d = torch.empty(M, H, **bf), torch.empty(M, H, **bf)
    g, u, m = torch.empty(M, I, **bf), torch.empty(M, I, **bf), torch.empty(M, I, **bf)
    wsb = max(q.grouped_ws_bytes(M, H, r, [H, NKV, NKV]),
              *[q.workspace_bytes(q.OP_LINEAR_FWD, M, N, K, r) for N, K in ((H, H), (I, H), (H, I))])
    ws, ws_side = torch.empty(wsb, dtype=torch.uint8, device=dev), torch.empty(wsb, dtype=torch.uint8, device=dev)
    ws_norm = q.workspace(q.OP_AQN_RMSNORM, M, 0, H, 0, dev)
    side = torch.cuda.Stream(device=dev)

    def step():
        h.copy_(x)
        for l, Ly in enumerate(lay):
            q.qerl_aqn_rmsnorm(h, Ly["gamma_attn"], 1e-6, sigma, 1, 0, 2 * l, y=n, ws=ws_norm)
            q.qerl_nvfp4_lora_linear_fwd_grouped(n, [Ly[nm] for nm in ("q", "k", "v")], s, packed=True,
                                                 ys=[qo, ko, vo], ws=ws)
            q.qerl_nvfp4_lora_linear_fwd_packed(Ly["attn"], *Ly["o"], s, y=o, ws=ws)
            q.qerl_residual_add(h, o, out=h)
            q.qerl_aqn_rmsnorm(h, Ly["gamma_mlp"], 1e-6, sigma, 1, 0, 2 * l + 1, y=n, ws=ws_norm)
            cur = torch.cuda.current_stream()
            side.wait_stream(cur)
            q.qerl_nvfp4_lora_linear_fwd_packed(n, *Ly["gate"], s, y=g, ws=ws)
            with torch.cuda.stream(side):
                q.qerl_nvfp4_lora_linear_fwd_packed(n, *Ly["up"], s, y=u, ws=ws_side)
            cur.wait_stream(side)
            q.qerl_swiglu(g, u, out=m)
            q.qerl_nvfp4_lora_linear_fwd_packed(m, *Ly["down"], s, y=d, ws=ws)
            q.qerl_residual_add(h, d, out=h)
    gr = _graph(step)
    _time_graph(gr, 2)
    sec = _time_graph(gr, 5) / 5
    assert q.get_error() == 0
    del gr
    return sec


def layer_bytes(wl):
    return sum(linear_bytes(N, K, wl.r) for _, N, K in wl.linears)


def decode_rows(dev):
    """Configs 0, 1 (M = 1, 8, 64, the CUDA-core / tensor-core crossover, the
    decoder-chain kernel on one layer) and 3 (the 64-layer 32B stack)."""
    import nvfp4_weight_only_quantize_gb300 as q
    from nvfp4_weight_only_quantize_gb300 import synth
    hbm = peaks()[0]
    out = {}
    # config 0: Qwen2.5-3B q_proj, M = 16, r = 16; 64 rotating weight copies (151 MB > L2)
    wl0 = synth.WORKLOADS[0]
    _, N, K = wl0.linears[0]
    copies = [q.qerl_nvfp4_quantize(synth.weight(N, K, synth.seed_of(0, c, synth.T_W), dev)) for c in range(64)]
    for c in copies:
        q.qerl_nvfp4_pack_codes(c[0], out=c[0])
    A = synth.lora_A(16, K, synth.seed_of(0, 0, synth.T_A), dev)
    B = synth.lora_B(N, 16, synth.seed_of(0, 0, synth.T_B), dev)
    x = synth.activations(16, K, synth.seed_of(0, 0, synth.T_X), dev)
    y = torch.empty(16, N, dtype=torch.bfloat16, device=dev)
    ws = q.workspace(q.OP_LINEAR_FWD, 16, N, K, 16, dev)

    def run0():
        for codes, sc, ts in copies:
            q.qerl_nvfp4_lora_linear_fwd_packed(x, codes, sc, ts, A, B, 2.0, y=y, ws=ws)
    g = _graph(run0)
    _time_graph(g, 3)
    us = _time_graph(g, 10) / (10 * len(copies)) * 1e6
    b0 = linear_bytes(N, K, 16)
    out["c0_small"] = {"workload": wl0.name, "us": round(us, 2), "GBps": round(b0 / us / 1e3, 1),
                       "frac_of_hbm": round(b0 / us / 1e3 / hbm, 4),
                       "note": "2.4 MB per call: launch- and latency-bound, not bandwidth-bound (64 rotating "
                               "copies, 151 MB > L2, one CUDA graph)"}
    del g, copies
    # config 1 at M = 1, 8, 64: the decode step, and the crossover of the two forward paths
    wl = synth.WORKLOADS[1]
    per_copy = sum(N * K * 0.5625 for _, N, K in wl.linears)
    n_copies = max(2, int(3 * L2_BYTES // per_copy) + 1)
    layer = DecodeLayer(wl, n_copies, dev)
    sigma = q.qerl_aqn_sigma(0, 1000, wl.sigma[0], wl.sigma[1], 10)
    by_m = {}
    for M in (1, 8, 64):
        buf = layer.buffers(M, dev)
        x = synth.activations(M, wl.hidden, synth.seed_of(1, 0, synth.T_X), dev)
        attn = synth.activations(M, wl.hidden, synth.seed_of(1, 1, synth.T_X), dev)
        graphs = [_graph(lambda c=c: layer.step(c, x, attn, buf, sigma, c)) for c in range(n_copies)]
        for i in range(3 * n_copies):
            graphs[i % n_copies].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10 * n_copies
        e0.record()
        for i in range(reps):
            graphs[i % n_copies].replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        by_m[M] = {"us_per_layer": round(us, 1), "GBps": round(layer.bytes_per_step / us / 1e3, 1),
                   "tokens_per_s": round(M / us * 1e6, 1)}
        del graphs, buf
    out["c1_decode_by_M"] = {"workload": wl.name + " (per-linear kernels, one graph per step)", "by_M": by_m}
    # crossover: gate_proj at M = 1..8: the CUDA-core GEMM, the CUDA-core GEMV
    # (M <= 2) and the tcgen05 path
    cross = {}
    name, N, K = [l for l in wl.linears if l[0] == "gate_proj"][0]
    li = [l[0] for l in wl.linears].index(name)
    for M in (1, 2, 4, 8):
        xin = synth.activations(M, K, 77, dev)
        yout = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        wsl = q.workspace(q.OP_LINEAR_FWD, M, N, K, wl.r, dev)
        row = {}
        algos = [("simt", q.ALGO_SIMT), ("tcgen05", q.ALGO_TCGEN05)] + ([("gemv", q.ALGO_GEMV)] if M <= 2 else [])
        for tag, algo in algos:
            q.set_linear_algo(algo)

            def run_lin(xin=xin, yout=yout, wsl=wsl):
                for c in range(n_copies):
                    _, _, _, codes, scales, ts, A, B = layer.copies[c][0][li]
                    layer.fwd(xin, codes, scales, ts, A, B, wl.lora_scale, y=yout, ws=wsl)
            g = _graph(run_lin)
            _time_graph(g, 3)
            row[tag + "_us"] = round(_time_graph(g, 10) / (10 * n_copies) * 1e6, 2)
            del g
        q.set_linear_algo(q.ALGO_AUTO)
        row["fastest"] = min([t for t, _ in algos], key=lambda t: row[t + "_us"])
        row["GBps_fastest"] = round(linear_bytes(N, K, wl.r) / (row[row["fastest"] + "_us"] * 1e3), 1)
        cross[M] = row
    out["c1_crossover_gate_proj"] = {"workload": f"qwen2.5-7b gate_proj {N}x{K}, {n_copies} rotating copies",
                                     "by_M": cross,
                                     "auto": "AUTO takes the GEMV for single-token calls on weights up to 24M values (not this "
                                             "one) and the tensor-core path otherwise"}
    del layer
    torch.cuda.empty_cache()
    # the decoder-chain kernel on one 7B layer (norms, residuals and SwiGLU fused), 4 rotating layers
    M = 64
    H, I = wl.hidden, 18944
    lay = _chain_layers(q, synth, 4, M, H, H, 512, I, wl.r, 1, dev)
    xc = synth.activations(M, H, 5, dev)
    yc = torch.empty_like(xc)
    plans = [q.DecoderChain([lay[c]], M, H, H, 512, I, wl.r, wl.lora_scale, 1e-6, xc, yc) for c in range(4)]
    g = _graph(lambda: [p.run(sigma, 1, 0, first_layer=0) for p in plans])
    _time_graph(g, 3)
    us = _time_graph(g, 10) / 40 * 1e6
    lb = layer_bytes(wl)
    p4 = q.DecoderChain(lay, M, H, H, 512, I, wl.r, wl.lora_scale, 1e-6, xc, yc)
    us4 = _time_fn(lambda: p4.run(sigma, 1, 0), 10) / 4 * 1e6
    out["c1_chain_layer"] = {"workload": "qwen2.5-7b decoder layer through the decoder-chain kernel (norm -> q|k|v, "
                                         "o + residual, norm -> gate|up, SwiGLU, down + residual), M=64, r=32",
                             "us_per_layer_one_layer_launches": round(us, 1), "GBps": round(lb / us / 1e3, 1),
                             "us_per_layer_four_layers_one_launch": round(us4, 1),
                             "GBps_four_layers": round(lb / us4 / 1e3, 1)}
    del plans, p4, g, lay
    torch.cuda.empty_cache()
    # config 3: the Qwen2.5-32B 64-layer decode stack, one launch per step
    wl3 = synth.WORKLOADS[3]
    H3, NKV3, I3 = 5120, 1024, 27648
    lay = _chain_layers(q, synth, wl3.layers, 64, H3, H3, NKV3, I3, wl3.r, 3, dev)
    x3 = synth.activations(64, H3, synth.seed_of(3, 0, 400), dev)
    y3 = torch.empty_like(x3)
    p64 = q.DecoderChain(lay, 64, H3, H3, NKV3, I3, wl3.r, wl3.lora_scale, 1e-6, x3, y3)
    sec_chain = _time_fn(lambda: p64.run(sigma, 1, 0), 5)
    assert q.get_error() == 0
    del p64
    # the same stack through the per-linear calls (norm, grouped q|k|v, o, residual add,
    # norm, gate and up on two streams, SwiGLU, down, residual add), one CUDA graph per step
    sec_lin = _time_stack_per_linear(q, lay, x3, H3, NKV3, I3, wl3, sigma)
    b3 = layer_bytes(wl3) * wl3.layers
    best, path = (sec_lin, "per-linear calls, one CUDA graph per step") if sec_lin < sec_chain else \
        (sec_chain, "one decoder-chain launch per step")
    out["c3_decode_stack"] = {"workload": wl3.name + ", attention output random bf16",
                              "path": path,
                              "ms_per_step": round(best * 1e3, 3), "GBps": round(b3 / best / 1e9, 1),
                              "frac_of_hbm": round(b3 / best / 1e9 / hbm, 4),
                              "tokens_per_s": round(64 / best, 1), "weight_GB": round(b3 / 1e9, 2),
                              "decoder_chain_ms": round(sec_chain * 1e3, 3),
                              "per_linear_graph_ms": round(sec_lin * 1e3, 3)}
    del lay
    torch.cuda.empty_cache()
    return out



def other_rows(dev, only=None, profile=False):
    """Each remaining hot-path row on its own workload (CUDA events, after warm-up):
    the quantizer on a Qwen2.5-7B gate_proj weight, AQN-RMSNorm at decode and
    prefill sizes, the Qwen2.5-14B prefill linears (M = 4096) and one Qwen2.5-7B
    backward (M = 8192)."""
    import nvfp4_weight_only_quantize_gb300 as q
    from nvfp4_weight_only_quantize_gb300 import synth
    rows = {}
    want = (lambda row: only is None or only == row)

    def timed(fn, reps, warm=3):
        # with --profile-row, ncu (--profile-from-start off) sees only the timed launches
        if profile:
            fn()
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaProfilerStart()
        sec = _time_fn(fn, reps, warm=0 if profile else warm)
        if profile:
            torch.cuda.cudart().cudaProfilerStop()
        return sec
    # a1: 18944 x 3584 bf16 (136 MB, above L2); algorithmic bytes = read W once + write codes/scales
    N, K = 18944, 3584
    W = synth.weight(N, K, 11, dev) if want("a1") else None
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(N, K // 16, dtype=torch.uint8, device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    wsq = q.workspace(q.OP_QUANTIZE, 0, N, K, 0, dev)
    sec = timed(lambda: q.qerl_nvfp4_quantize(W, out=(codes, scales, ts), ws=wsq), 20) if want("a1") else 0.0
    if want("a1"):
        rows["a1_quantize"] = {"workload": f"qwen2.5-7b gate_proj weight {N}x{K} bf16", "us": round(sec * 1e6, 1),
                               "GBps": round(N * K * 2.5625 / sec / 1e9, 1),
                               "bytes": "2 B read + 0.5625 B written per weight (W is read twice; the second, "
                                        "backward pass finds its first part in L2)"}
        # f3: MXFP4 quantization of the same weight (one pass: blocks of 32, power-of-two scales)
        mcodes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
        mscales = torch.empty(N, K // 32, dtype=torch.uint8, device=dev)
        sec = timed(lambda: q.qerl_mxfp4_quantize(W, out=(mcodes, mscales)), 20)
        rows["f3_mxfp4_quantize"] = {"workload": f"qwen2.5-7b gate_proj weight {N}x{K} bf16",
                                     "us": round(sec * 1e6, 1),
                                     "GBps": round(N * K * (2 + 0.5 + 1 / 32) / sec / 1e9, 1),
                                     "bytes": "2 B read + 0.53125 B written per weight"}
        del mcodes, mscales
        # an L2-sized weight (q_proj 3584 x 3584, 25.7 MB), 8 rotating copies so each call starts cold
        N2, K2, nc = 3584, 3584, 8
        Ws = [synth.weight(N2, K2, 30 + c, dev) for c in range(nc)]
        outs = [(torch.empty(N2, K2 // 2, dtype=torch.uint8, device=dev),
                 torch.empty(N2, K2 // 16, dtype=torch.uint8, device=dev),
                 torch.empty(1, dtype=torch.float32, device=dev)) for _ in range(nc)]
        wsq2 = q.workspace(q.OP_QUANTIZE, 0, N2, K2, 0, dev)
        sec = timed(lambda: [q.qerl_nvfp4_quantize(Ws[c], out=outs[c], ws=wsq2) for c in range(nc)], 10) / nc
        rows["a1_quantize_l2_sized"] = {"workload": f"qwen2.5-7b q_proj weight {N2}x{K2} bf16, {nc} rotating copies",
                                        "us": round(sec * 1e6, 1), "GBps": round(N2 * K2 * 2.5625 / sec / 1e9, 1),
                                        "bytes": "2 B read + 0.5625 B written per weight"}
        del Ws, outs
    del W
    # the decoder chain on one Qwen2.5-7B layer, M = 64, r = 32 (a profiling row:
    # its numbers are also in the decode rows)
    if only == "chain":
        wl = synth.WORKLOADS[1]
        M, H, I = 64, wl.hidden, 18944
        lay = _chain_layers(q, synth, 2, M, H, H, 512, I, wl.r, 1, dev)
        xc = synth.activations(M, H, 5, dev)
        yc = torch.empty_like(xc)
        plans = [q.DecoderChain([lay[c]], M, H, H, 512, I, wl.r, wl.lora_scale, 1e-6, xc, yc) for c in range(2)]
        sigma = q.qerl_aqn_sigma(0, 1000, wl.sigma[0], wl.sigma[1], 10)
        sec = timed(lambda: [p_.run(sigma, 1, 0) for p_ in plans], 5) / 2
        rows["chain_layer"] = {"workload": "qwen2.5-7b decoder layer through the decoder-chain kernel, M=64, r=32",
                               "us": round(sec * 1e6, 1), "GBps": round(layer_bytes(wl) / sec / 1e9, 1)}
        del plans, lay
    # the CUDA-core GEMV on one token: Qwen2.5-7B o_proj 3584 x 3584, 8 rotating
    # copies (a profiling row: its numbers are also in the decode rows)
    if only == "gemv":
        N, K, r, nc = 3584, 3584, 32, 8
        wts = []
        for c in range(nc):
            W = synth.weight(N, K, 40 + c, dev)
            cs = q.qerl_nvfp4_quantize(W)
            del W
            q.qerl_nvfp4_pack_codes(cs[0], out=cs[0])
            wts.append((*cs, synth.lora_A(r, K, 50 + c, dev), synth.lora_B(N, r, 60 + c, dev)))
        x1 = synth.activations(1, K, 70, dev)
        y1 = torch.empty(1, N, dtype=torch.bfloat16, device=dev)
        ws1 = q.workspace(q.OP_LINEAR_FWD, 1, N, K, r, dev)
        q.set_linear_algo(q.ALGO_GEMV)
        try:
            sec = timed(lambda: [q.qerl_nvfp4_lora_linear_fwd_packed(x1, *w_, 2.0, y=y1, ws=ws1) for w_ in wts], 5) / nc
        finally:
            q.set_linear_algo(q.ALGO_AUTO)
        rows["gemv_one_token"] = {"workload": f"qwen2.5-7b o_proj {N}x{K}, M=1, r={r}", "us": round(sec * 1e6, 2),
                                  "GBps": round(linear_bytes(N, K, r) / sec / 1e9, 1)}
        del wts
    # f3: the forwards with an MXFP4 weight and with FP32 LoRA adapters beside the
    # NVFP4 forward, on qwen2.5-7b gate_proj at M = 8, r = 32: four weight copies
    # rotated (above L2), on tcgen05 (the default selection) and, for context, on
    # the CUDA-core GEMM
    if want("f3"):
        N, K, M, r, NC = 18944, 3584, 8, 32, 4
        nv, mx = [], []
        for c in range(NC):
            W = synth.weight(N, K, 11 + 100 * c, dev)
            nv.append(q.qerl_nvfp4_quantize(W))
            mx.append(q.qerl_mxfp4_quantize(W))
            del W
        x = synth.activations(M, K, 14, dev)
        A, B = synth.lora_A(r, K, 15, dev), synth.lora_B(N, r, 16, dev)
        Af, Bf = A.float(), B.float()
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        wsl = q.workspace(q.OP_LINEAR_FWD, M, N, K, r, dev)
        wsf = q.workspace(q.OP_LINEAR_FWD_F32AB, M, N, K, r, dev)
        wsm = q.workspace(q.OP_MXFP4_FWD, M, N, K, r, dev)
        arms = {
            "nvfp4_bf16_adapters": lambda: [q.qerl_nvfp4_lora_linear_fwd(x, *w_, A, B, 2.0, y=y, ws=wsl) for w_ in nv],
            "nvfp4_fp32_adapters": lambda: [q.qerl_nvfp4_lora_linear_fwd_f32ab(x, *w_, Af, Bf, 2.0, y=y, ws=wsf)
                                            for w_ in nv],
            "mxfp4_bf16_adapters": lambda: [q.qerl_mxfp4_lora_linear_fwd(x, *w_, A, B, 2.0, y=y, ws=wsm) for w_ in mx]}
        res = {}
        for name, fn in arms.items():
            sec = timed(fn, 10) / NC
            wbytes = N * K * (0.5 + (1 / 32 if name.startswith("mx") else 1 / 16))
            res[name] = {"us": round(sec * 1e6, 1), "weight_GBps": round(wbytes / sec / 1e9, 1)}
            if name != "nvfp4_bf16_adapters":
                q.set_linear_algo(q.ALGO_SIMT)
                res[name]["cuda_core_gemm_us"] = round(timed(fn, 2, warm=1) / NC * 1e6, 1)
                q.set_linear_algo(q.ALGO_AUTO)
        rows["f3_format_variants_fwd"] = {
            "workload": f"qwen2.5-7b gate_proj {N}x{K}, M={M}, r={r}, {NC} weight copies rotated (above L2)",
            "by_format": res,
            "path": "tcgen05 for all three (MXFP4: scales written at one byte per 16 values each call, E8M0 factor "
                    "in the dequantizer; FP32 adapters: LoRA term as three bf16 hi/lo products); "
                    "cuda_core_gemm_us: the same call on the CUDA-core GEMM"}
        del nv, mx
    # a2: decode and prefill norms
    for M, H, tag in ([(64, 3584, "decode M=64 H=3584"), (4096, 5120, "prefill M=4096 H=5120")] if want("a2") else []):
        x = synth.activations(M, H, 12, dev)
        g = synth.norm_gamma(H, 13, dev)
        y = torch.empty_like(x)
        wsn = q.workspace(q.OP_AQN_RMSNORM, M, 0, H, 0, dev)
        sec = timed(lambda: q.qerl_aqn_rmsnorm(x, g, 1e-6, 1e-2, 1, 5, 0, y=y, ws=wsn), 50)
        row = {"workload": tag, "us": round(sec * 1e6, 2), "GBps": round((4 * M * H + 6 * H) / sec / 1e9, 1)}
        if M == 64:
            # the same call 20 times in one CUDA graph (chained launches): the device time per call,
            # without the host's per-call dispatch that paces the eager loop at this size
            gr = _graph(lambda: [q.qerl_aqn_rmsnorm(x, g, 1e-6, 1e-2, 1, 5 + i, 0, y=y, ws=wsn) for i in range(20)])
            _time_graph(gr, 3)
            row["us_in_graph"] = round(_time_graph(gr, 10) / 200 * 1e6, 2)
            del gr
        rows[f"a2_aqn_rmsnorm_{'decode' if M == 64 else 'prefill'}"] = row
    # a4: Qwen2.5-14B prefill linears, M = 4096, r = 32
    wl = synth.WORKLOADS[2]
    M, tot_f, tot_s, per = 4096, 0.0, 0.0, {}
    per_lin_args, per_lin_N, per_flops, w16_gu = {}, {}, {}, {}
    _, bf16, _, kind = peaks()
    if not want("a4"):
        wl = synth.Workload(wl.name, [], wl.M, wl.r, wl.hidden)
    x = synth.activations(M, max(K for _, _, K in wl.linears), 14, dev) if wl.linears else None
    for i, (name, N, K) in enumerate(wl.linears):
        W = synth.weight(N, K, 20 + i, dev)
        c, sc, t = q.qerl_nvfp4_quantize(W)
        del W
        if name in ("gate_proj", "up_proj") and want("a4"):  # the 16-bit arm of the grouped gate|up below
            w16_gu[name] = q.qerl_nvfp4_dequantize(c, sc, t, N, K)
        q.qerl_nvfp4_pack_codes(c, out=c)
        A = synth.lora_A(wl.r, K, 40 + i, dev)
        B = synth.lora_B(N, wl.r, 60 + i, dev)
        xi = x[:, :K].contiguous()
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = q.workspace(q.OP_LINEAR_FWD, M, N, K, wl.r, dev)
        sec = timed(lambda: q.qerl_nvfp4_lora_linear_fwd_packed(xi, c, sc, t, A, B, 2.0, y=y, ws=ws), 10)
        fl = 2.0 * M * N * K + 2.0 * M * wl.r * (N + K)
        per[name] = {"us": round(sec * 1e6, 1), "TFLOPs": round(fl / sec / 1e12, 1)}
        tot_f, tot_s = tot_f + fl, tot_s + sec
        per_lin_args[name], per_lin_N[name], per_flops[name] = (c, sc, t, A, B), N, fl
        if name == "q_proj":
            per_lin_N["K_qkv"] = K
    if want("a4"):
        # q|k|v as one grouped call (they read the same x)
        gq = [per_lin_args[n] for n in ("q_proj", "k_proj", "v_proj")]
        yq = [torch.empty(M, Nq, dtype=torch.bfloat16, device=dev) for Nq in (per_lin_N[n] for n in ("q_proj", "k_proj", "v_proj"))]
        wsg = torch.empty(q.grouped_ws_bytes(M, per_lin_N["K_qkv"], wl.r,
                                             [per_lin_N[n] for n in ("q_proj", "k_proj", "v_proj")]),
                          dtype=torch.uint8, device=dev)
        xq = x[:, :per_lin_N["K_qkv"]].contiguous()
        sec_g = timed(lambda: q.qerl_nvfp4_lora_linear_fwd_grouped(xq, gq, 2.0, packed=True, ys=yq, ws=wsg), 10)
        fl_g = sum(per_flops[n] for n in ("q_proj", "k_proj", "v_proj"))
        per["qkv_grouped"] = {"us": round(sec_g * 1e6, 1), "TFLOPs": round(fl_g / sec_g / 1e12, 1)}
        lay_s = sec_g + sum(per[n]["us"] for n in ("o_proj", "gate_proj", "up_proj", "down_proj")) / 1e6
        # gate|up as one grouped call too (one pass over x for both down-projections,
        # one launch of twice the tiles)
        gu = [per_lin_args[n] for n in ("gate_proj", "up_proj")]
        yu = [torch.empty(M, per_lin_N[n], dtype=torch.bfloat16, device=dev) for n in ("gate_proj", "up_proj")]
        wsu = torch.empty(q.grouped_ws_bytes(M, per_lin_N["K_qkv"], wl.r, [per_lin_N[n] for n in ("gate_proj", "up_proj")]),
                          dtype=torch.uint8, device=dev)
        sec_u = timed(lambda: q.qerl_nvfp4_lora_linear_fwd_grouped(xq, gu, 2.0, packed=True, ys=yu, ws=wsu), 10)
        fl_u = sum(per_flops[n] for n in ("gate_proj", "up_proj"))
        # the same product in torch (cuBLAS bf16) on the dequantized weights of the same codes, concatenated:
        # y_gate | y_up = x [W_gate; W_up]^T, plus each LoRA branch (x [A_gate; A_up]^T, then one small
        # product per linear)
        Ng, Nu = per_lin_N["gate_proj"], per_lin_N["up_proj"]
        Wcat = torch.cat([w16_gu["gate_proj"], w16_gu["up_proj"]])
        Acat = torch.cat([per_lin_args["gate_proj"][3], per_lin_args["up_proj"][3]])
        Bg, Bu = per_lin_args["gate_proj"][4], per_lin_args["up_proj"][4]
        ycat = torch.empty(M, Ng + Nu, dtype=torch.bfloat16, device=dev)
        del w16_gu

        def gate_up_bf16():
            torch.mm(xq, Wcat.t(), out=ycat)
            tcat = torch.mm(xq, Acat.t())
            ycat[:, :Ng].add_(torch.mm(tcat[:, :wl.r], Bg.t()), alpha=2.0)
            ycat[:, Ng:].add_(torch.mm(tcat[:, wl.r:], Bu.t()), alpha=2.0)
        sec_b = timed(gate_up_bf16, 10)
        per["gate_up_grouped"] = {"us": round(sec_u * 1e6, 1), "TFLOPs": round(fl_u / sec_u / 1e12, 1),
                                  "bf16_cublas_us": round(sec_b * 1e6, 1),
                                  "bf16_cublas_TFLOPs": round(fl_u / sec_b / 1e12, 1),
                                  "speedup_vs_bf16": round(sec_b / sec_u, 3)}
        del Wcat, ycat
        lay_gg = sec_g + sec_u + sum(per[n]["us"] for n in ("o_proj", "down_proj")) / 1e6
        # the layer's two AQN-RMSNorms at M = 4096, H = 5120
        xn = synth.activations(M, wl.hidden, 15, dev)
        gn = synth.norm_gamma(wl.hidden, 16, dev)
        yn = torch.empty_like(xn)
        wsn = q.workspace(q.OP_AQN_RMSNORM, M, 0, wl.hidden, 0, dev)
        sec_n = timed(lambda: q.qerl_aqn_rmsnorm(xn, gn, 1e-6, 1e-2, 1, 5, 0, y=yn, ws=wsn), 20)
        lay_n = lay_gg + 2 * sec_n
        rows["a4_prefill"] = {"workload": wl.name, "TFLOPs": round(tot_f / tot_s / 1e12, 1),
                              "frac_of_bf16_peak": round(tot_f / tot_s / 1e12 / bf16, 3),
                              "layer_with_grouped_qkv_TFLOPs": round(tot_f / lay_s / 1e12, 1),
                              "layer_with_grouped_qkv_frac": round(tot_f / lay_s / 1e12 / bf16, 3),
                              "layer_with_grouped_qkv_and_gate_up_TFLOPs": round(tot_f / lay_gg / 1e12, 1),
                              "layer_with_grouped_qkv_and_gate_up_frac": round(tot_f / lay_gg / 1e12 / bf16, 3),
                              "layer_with_norms_us": round(lay_n * 1e6, 1),
                              "layer_with_norms_is": "q|k|v and gate|up as grouped calls, o and down, two norms",
                              "layer_with_norms_TFLOPs": round(tot_f / lay_n / 1e12, 1),
                              "layer_with_norms_frac": round(tot_f / lay_n / 1e12 / bf16, 3),
                              "norm_us": round(sec_n * 1e6, 1),
                              "peak": f"{kind} bf16_tflops {bf16}", "per_linear": per}
    if want("f2"):
        rows["f2_lora_rank_sweep"] = rank_sweep(dev)
    if not want("a5"):
        torch.cuda.synchronize()
        return rows
    # a5: the seven Qwen2.5-7B linears' backward, M = 8192, r = 32 (dx, dA, dB)
    wl = synth.WORKLOADS[4]
    M = 8192
    per5, tot_f5, tot_s5 = {}, 0.0, 0.0
    for i, (name, N, K) in enumerate(wl.linears):
        W = synth.weight(N, K, 30 + i, dev)
        c, sc, t = q.qerl_nvfp4_quantize(W)
        del W
        A = synth.lora_A(wl.r, K, 31, dev)
        B = synth.lora_B(N, wl.r, 32, dev)
        x = synth.activations(M, K, 33, dev)
        dy = synth.activations(M, N, 34, dev, std=1e-2)
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dA = torch.empty(wl.r, K, dtype=torch.float32, device=dev)
        dB = torch.empty(N, wl.r, dtype=torch.float32, device=dev)
        ws = q.workspace(q.OP_LINEAR_BWD, M, N, K, wl.r, dev)
        sec = timed(lambda: q.qerl_nvfp4_lora_linear_bwd(dy, x, c, sc, t, A, B, 2.0, dx=dx, dA=dA, dB=dB, ws=ws), 3,
                    warm=1)
        fl = 2.0 * M * N * K + 2.0 * M * wl.r * (3 * N + 2 * K)
        per5[name] = {"us": round(sec * 1e6, 1), "TFLOPs": round(fl / sec / 1e12, 1)}
        tot_f5, tot_s5 = tot_f5 + fl, tot_s5 + sec
        del c, sc, t, A, B, x, dy, dx, dA, dB, ws
        torch.cuda.empty_cache()
    rows["a5_backward"] = {"workload": f"qwen2.5-7b layer, all 7 linears, M={M}, r={wl.r}",
                           "us": round(tot_s5 * 1e6, 1), "TFLOPs": round(tot_f5 / tot_s5 / 1e12, 2),
                           "frac_of_bf16_peak": round(tot_f5 / tot_s5 / 1e12 / bf16, 3), "per_linear": per5,
                           "path": "every product on tensor cores (tcgen05): dx with transposed dequant; v = dy B, "
                                   "t = x A^T, dA = s v^T x, dB = s dy^T t as split-K rank products"}
    torch.cuda.synchronize()
    return rows


# ------------------------------------------------------------------ oracle arm
_ORACLE_INPUTS = {}


def _oracle_layer_inputs(wl, stride):
    """The decode layer's inputs for the oracle, prepared once (untimed): per
    linear a weight of N / stride output features drawn like the full one
    (the same distribution, so the same work per output feature), quantized by
    the oracle, LoRA A and B, and 64 token rows of x."""
    import oracle
    from nvfp4_weight_only_quantize_gb300 import synth
    key = (wl.name, stride)
    if key not in _ORACLE_INPUTS:
        lins = []
        for i, (name, N, K) in enumerate(wl.linears):
            base = synth.seed_of(1, 0, 16 * i)
            W = synth.bits(synth.weight(N // stride, K, base + synth.T_W))
            rc, codes, scales, st = oracle.nvfp4_quantize(W)
            assert rc == 0
            B = synth.bits(synth.lora_B(N // stride, wl.r, base + synth.T_B))
            lins.append((name, W.shape[0], K, codes, scales, st, synth.bits(synth.lora_A(wl.r, K, base + synth.T_A)),
                         B, synth.bits(synth.activations(64, K, base + synth.T_X))))
        _ORACLE_INPUTS[key] = lins
    return _ORACLE_INPUTS[key]


def _oracle_step(wl, M, stride, threads):
    """One sampled decode step on the CPU oracle: every linear of the layer at
    M tokens with N / stride output features.  Returns (seconds, NVFP4 + LoRA
    bytes of those weights)."""
    import numpy as np
    import oracle
    lins = _oracle_layer_inputs(wl, stride)
    oracle.set_threads(threads)
    secs = byts = 0.0
    try:
        for name, Ns, K, codes, scales, st, A, B, x in lins:
            t = time.perf_counter()
            oracle.lora_linear_fwd(x[:M], codes, scales, st, A, B, wl.lora_scale, rows=np.arange(M))
            secs += time.perf_counter() - t
            byts += linear_bytes(Ns, K, wl.r)
    finally:
        oracle.set_threads(1)
    return secs, byts


ORACLE_STRIDE = 64  # the sampled steps run 1/64 of every linear's output features


def cpu_baseline(wl, M, budget_s=20.0):
    """The oracle on a bounded sample of the decode step (every linear at M
    tokens with 1/64 of its output features), measured single-threaded and on
    all host cores; value = sampled weight bytes / measured time (all cores)."""
    ncpu = os.cpu_count() or 1
    _oracle_layer_inputs(wl, ORACLE_STRIDE)  # untimed preparation
    res = {}
    for tag, th in (("single", 1), ("all", ncpu)):
        secs = byts = 0.0
        n = 0
        while n < 1 or (secs < budget_s / 2 and n < 8):
            s_, b_ = _oracle_step(wl, M, ORACLE_STRIDE, th)
            secs, byts, n = secs + s_, byts + b_, n + 1
        res[tag] = (byts / secs / 1e9, secs / n, n)
    return {"value": round(res["all"][0], 4), "unit": "GB/s", "cores": ncpu, "kind": "oracle",
            "single_thread_GBps": round(res["single"][0], 4),
            "ms_per_sampled_step": {"single": round(res["single"][1] * 1e3, 1), "all": round(res["all"][1] * 1e3, 1)},
            "sample": f"the decode step's 7 linears at M={M}, each with 1/{ORACLE_STRIDE} of its output features "
                      f"(same distribution), fp64 C oracle; {res['all'][2]} sampled steps on "
                      f"{ncpu} cores (OpenMP over output features), {res['single'][2]} single-threaded; measured, "
                      "not extrapolated"}


def run_reference(args, rank, world):
    from nvfp4_weight_only_quantize_gb300 import synth
    if rank != 0:
        return
    wl = synth.WORKLOADS[1]
    M = args.M
    ncpu = os.cpu_count() or 1
    _oracle_layer_inputs(wl, ORACLE_STRIDE)
    for i in range(args.warmup):
        _oracle_step(wl, M, ORACLE_STRIDE, ncpu)
    secs = byts = 0.0
    for i in range(args.steps):
        s_, b_ = _oracle_step(wl, M, ORACLE_STRIDE, ncpu)
        secs, byts = secs + s_, byts + b_
    value = byts / secs / 1e9
    sample = (f"each step: the decode step's 7 linears at M={M}, each with 1/{ORACLE_STRIDE} of its output features "
              f"(same distribution), fp64 C oracle on {ncpu} cores; measured time per step")
    line = {"impl": "reference", "metric": "NVFP4+LoRA linear decode HBM GB/s (Qwen2.5-7B decoder layer)",
            "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": wl.name + f"; step at M={M}", "tokens_per_step": M, "lora_rank": wl.r,
                       "sample": f"1/{ORACLE_STRIDE} of every linear's output features"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": ncpu, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--M", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the quantize/norm/prefill/backward lines")
    ap.add_argument("--profile-row", choices=["a1", "a2", "a4", "a5", "f2", "f3", "chain", "gemv"],
                    help="run only that row's measurement, its timed launches bracketed by "
                         "cudaProfilerStart/Stop (for ncu --profile-from-start off), and print it")
    ap.add_argument("--codes", default="packed", choices=["packed", "standard"],
                    help="code layout of the frozen weights (packed once at load time, or as quantized)")
    ap.add_argument("--profile-region", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_init()
    if args.gpus != world:
        raise SystemExit(f"bench.py --gpus {args.gpus} needs {args.gpus} ranks (torchrun --nproc-per-node "
                         f"{args.gpus}); this launch has WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.profile_row:
        torch.cuda.set_device(local_rank)
        print(json.dumps(other_rows(torch.device("cuda", local_rank), only=args.profile_row, profile=True)),
              flush=True)
    else:
        import nvfp4_weight_only_quantize_gb300 as q
        q.lib()  # the CUDA library must be built; no fallback
        run_ours(args, rank, world, local_rank)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
