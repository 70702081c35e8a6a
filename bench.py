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
# (profiles/tc_fwd_decode_qwen7b_m64.md) of csrc/linear_tc.cu with this sha256
# prefix; reported as roofline.traffic only while the source still matches.
NCU_KERNEL_SHA = "883e2b82deff5143"
NCU_DRAM_BYTES = {"gate_proj": 39.939072e6, "up_proj": 39.938304e6, "down_proj": 42.14656e6}


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
                    ws_norm=self.q.workspace(self.q.OP_AQN_RMSNORM, M, 0, wl.hidden, 0, device))

    def step(self, copy, x, attn, buf, sigma, step_idx):
        """One decoder layer: norm -> q|k|v (one grouped call) -> o -> norm ->
        gate -> up -> down.  Attention and SwiGLU are not part
        of this step (synthetic attention output; down reads up's output)."""
        q = self.q
        lins, gammas = self.copies[copy]
        by = {l[0]: l for l in lins}
        o = buf["outs"]
        s = self.wl.lora_scale

        def group(names, xin):
            gs = [by[n][3:8] for n in names]
            q.qerl_nvfp4_lora_linear_fwd_grouped(xin, gs, s, packed=self.packed, ys=[o[n] for n in names],
                                                 ws=buf["ws"])

        def single(name, xin):
            _, N, K, codes, scales, ts, A, B = by[name]
            self.fwd(xin, codes, scales, ts, A, B, s, y=o[name], ws=buf["ws"])

        q.qerl_aqn_rmsnorm(x, gammas[0], 1e-6, sigma, 1, step_idx, 2 * copy, y=buf["h1"], ws=buf["ws_norm"])
        group(("q_proj", "k_proj", "v_proj"), buf["h1"])
        single("o_proj", attn)
        q.qerl_aqn_rmsnorm(o["o_proj"], gammas[1], 1e-6, sigma, 1, step_idx, 2 * copy + 1, y=buf["h2"],
                           ws=buf["ws_norm"])
        # gate and up stay separate calls: grouped they need two waves of
        # one-tile CTAs over the SMs, which measured slower than two launches
        single("gate_proj", buf["h2"])
        single("up_proj", buf["h2"])
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

    # --- end to end through the public API with host buffers
    xh = x.cpu().pin_memory()
    ah = attn.cpu().pin_memory()
    yh = torch.empty(M, wl.hidden, dtype=torch.bfloat16).pin_memory()
    out = buf["outs"]["down_proj"]
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        x.copy_(xh, non_blocking=True)
        attn.copy_(ah, non_blocking=True)
        graphs[i % n_copies].replay()
        yh.copy_(out, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
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
                   "launch": "one CUDA graph per step (per weight copy); q|k|v as one grouped call",
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
                               "bytes": "2 B read + 0.5625 B written per weight (the kernel reads W twice)"}
    del W
    # a2: decode and prefill norms
    for M, H, tag in ([(64, 3584, "decode M=64 H=3584"), (4096, 5120, "prefill M=4096 H=5120")] if want("a2") else []):
        x = synth.activations(M, H, 12, dev)
        g = synth.norm_gamma(H, 13, dev)
        y = torch.empty_like(x)
        wsn = q.workspace(q.OP_AQN_RMSNORM, M, 0, H, 0, dev)
        sec = timed(lambda: q.qerl_aqn_rmsnorm(x, g, 1e-6, 1e-2, 1, 5, 0, y=y, ws=wsn), 50)
        rows[f"a2_aqn_rmsnorm_{'decode' if M == 64 else 'prefill'}"] = {
            "workload": tag, "us": round(sec * 1e6, 2), "GBps": round((4 * M * H + 6 * H) / sec / 1e9, 1)}
    # a4: Qwen2.5-14B prefill linears, M = 4096, r = 32
    wl = synth.WORKLOADS[2]
    M, tot_f, tot_s, per = 4096, 0.0, 0.0, {}
    per_lin_args, per_lin_N, per_flops = {}, {}, {}
    _, bf16, _, kind = peaks()
    if not want("a4"):
        wl = synth.Workload(wl.name, [], wl.M, wl.r, wl.hidden)
    x = synth.activations(M, max(K for _, _, K in wl.linears), 14, dev) if wl.linears else None
    for i, (name, N, K) in enumerate(wl.linears):
        W = synth.weight(N, K, 20 + i, dev)
        c, sc, t = q.qerl_nvfp4_quantize(W)
        del W
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
        rows["a4_prefill"] = {"workload": wl.name, "TFLOPs": round(tot_f / tot_s / 1e12, 1),
                              "frac_of_bf16_peak": round(tot_f / tot_s / 1e12 / bf16, 3),
                              "layer_with_grouped_qkv_TFLOPs": round(tot_f / lay_s / 1e12, 1),
                              "layer_with_grouped_qkv_frac": round(tot_f / lay_s / 1e12 / bf16, 3),
                              "peak": f"{kind} bf16_tflops {bf16}", "per_linear": per}
    if want("f2"):
        rows["f2_lora_rank_sweep"] = rank_sweep(dev)
    if not want("a5"):
        torch.cuda.synchronize()
        return rows
    # a5: Qwen2.5-7B q_proj backward, M = 8192, r = 32 (dx, dA, dB)
    wl = synth.WORKLOADS[4]
    name, N, K = wl.linears[0]
    M = 8192
    W = synth.weight(N, K, 30, dev)
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
    rows["a5_backward"] = {"workload": f"qwen2.5-7b {name} {N}x{K}, M={M}, r={wl.r}", "us": round(sec * 1e6, 1),
                           "TFLOPs": round(fl / sec / 1e12, 2),
                           "frac_of_bf16_peak": round(fl / sec / 1e12 / bf16, 3),
                           "path": "every product on tensor cores (tcgen05): dx with transposed dequant; v = dy B, "
                                   "t = x A^T, dA = s v^T x, dB = s dy^T t as split-K rank products"}
    torch.cuda.synchronize()
    return rows


# ------------------------------------------------------------------ oracle arm
_ORACLE_INPUTS = {}


def _oracle_linear_sample(wl, lin_idx, rows=1):
    """Quantize one linear and run `rows` token rows of the forward with the oracle;
    returns (seconds, NVFP4+LoRA bytes of that linear)."""
    import numpy as np
    import oracle
    from nvfp4_weight_only_quantize_gb300 import synth
    name, N, K = wl.linears[lin_idx]
    key = (lin_idx, rows)
    if key not in _ORACLE_INPUTS:  # inputs and the quantized weight are prepared once, untimed
        base = synth.seed_of(1, 0, 16 * lin_idx)
        rc, codes, scales, st = oracle.nvfp4_quantize(synth.bits(synth.weight(N, K, base + synth.T_W)))
        _ORACLE_INPUTS[key] = (synth.bits(synth.activations(rows, K, base + synth.T_X)), codes, scales, st,
                               synth.bits(synth.lora_A(wl.r, K, base + synth.T_A)),
                               synth.bits(synth.lora_B(N, wl.r, base + synth.T_B)))
    xb, codes, scales, st, Ab, Bb = _ORACLE_INPUTS[key]
    t = time.perf_counter()
    oracle.lora_linear_fwd(xb, codes, scales, st, Ab, Bb, wl.lora_scale, rows=np.arange(rows))
    return time.perf_counter() - t, linear_bytes(N, K, wl.r)


def cpu_baseline(wl, M, budget_s=20.0):
    """The oracle forward on a bounded sample of the decode layer: one token row
    through the linears (cycling q..down) until ~budget_s of CPU work; the
    throughput is scaled to the M-token step (time x M)."""
    secs = byts = 0.0
    n = 0
    while secs < budget_s and n < 7 * 4:
        s, b = _oracle_linear_sample(wl, n % 7)
        secs, byts, n = secs + s, byts + b, n + 1
    return {"value": round(byts / (secs * M) / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} linear forwards of 1 token row (cycling q..down of the 7B layer), "
                      f"{secs:.1f} s of single-thread fp64 oracle; time scaled x{M} to the M={M} step"}


def run_reference(args, rank, world):
    from nvfp4_weight_only_quantize_gb300 import synth
    if rank != 0:
        return
    wl = synth.WORKLOADS[1]
    M = args.M
    for i in range(args.warmup):
        _oracle_linear_sample(wl, i % 7)
    secs = byts = 0.0
    for i in range(args.steps):
        s, b = _oracle_linear_sample(wl, i % 7)
        secs, byts = secs + s, byts + b
    value = byts / (secs * M) / 1e9
    line = {"impl": "reference", "metric": "NVFP4+LoRA linear decode HBM GB/s (Qwen2.5-7B decoder layer)",
            "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * M * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": wl.name + f"; step at M={M}", "tokens_per_step": M, "lora_rank": wl.r},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "each step: the CPU oracle forward of 1 token row through one linear of "
                                       f"the 7B layer (cycling q..down), time scaled x{M} to the M={M} step"},
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
    ap.add_argument("--profile-row", choices=["a1", "a2", "a4", "a5", "f2"],
                    help="run only that row's measurement, its timed launches bracketed by "
                         "cudaProfilerStart/Stop (for ncu --profile-from-start off), and print it")
    ap.add_argument("--codes", default="packed", choices=["packed", "standard"],
                    help="code layout of the frozen weights (packed once at load time, or as quantized)")
    ap.add_argument("--profile-region", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_init()
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
