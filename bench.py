#!/usr/bin/env python
"""Benchmark of the NVFP4 mixture-of-experts FFN forward on GB300.

One step = one full forward of the MoE layer (routing, slot sort, gather +
NVFP4 quantization, L1 grouped GEMM with fused SwiGLU + requantization, L2
grouped GEMM with fused weighted combine, bf16 finalize) over one batch of
the prefill workload: T=8192 tokens, H=4096, I=2048, E=48 local experts,
top_k=6, Zipf(1.1) expert popularity, 2% outlier channels x20 (synthetic,
seeded).  Weights are random N(0, 0.02), quantized to NVFP4 by the library;
activation global scales are calibrated on the device before timing.

Prints ONE JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM; `e2e` times the library's host pipeline (api.HostPipeline):
every step copies its pinned host inputs in and its output back inside the
timed region, the copies of neighbouring steps overlapping the forward.  `roofline` is the L1
grouped GEMM (the dominant kernel) against the dense FP4 tensor peak.
`--impl reference` times the CPU oracle on a bounded sample of the same
workload (there is no other implementation of this method to run).

Multi-GPU (torchrun): every rank runs its own batch of T tokens with the full
local expert set (data parallel over tokens, no collective on the data path);
scaling is weak and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "moe_layer_tokens_per_s"
UNIT = "tokens/s"
SHAPES = {
    "prefill": dict(T=8192, H=4096, I=2048, E=48, top_k=6),
    "decode": dict(T=128, H=4096, I=2048, E=32, top_k=6),
}
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / BF16 tensor throughput ratio
NOMINAL_FP4_TFLOPS = 13500.0  # GB300 dense FP4 tensor peak (nominal)
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e bandwidth (nominal)
GATE_LIMIT = UP_LIMIT = 10.0


def workload_name(shape_key):
    s = SHAPES[shape_key]
    extra = "Zipf(1.1) expert prior, 2% outlier channels x20" if shape_key == "prefill" else \
        "per-expert logit bias N(0,0.5)"
    return (f"{shape_key} NVFP4 MoE layer forward T={s['T']} H={s['H']} I={s['I']} E={s['E']} "
            f"top_k={s['top_k']}, {extra}")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(SHAPES), default="prefill")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true", help="skip the decode-size side measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--swap-l2", type=int, choices=[0, 1], default=0,
                    help="1: small batches run the L2 GEMM with swapped operands (nvfp4_moe_set_swap_l2)")
    return ap.parse_args()


def fp4_peak_burst(peaks):
    """Dense FP4 denominator: the measured bf16 burst rate x the nominal FP4/BF16 ratio."""
    return peaks["bf16_tflops"] * FP4_OVER_BF16


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def stored_traffic(kernel):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, or None when
    the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "nvfp4_mixture_experts_expert_gb300", "csrc", "gemm.cu")
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != ent.get("gemm_cu_sha256_16"):
            return None
    return ent.get("bytes_per_launch")


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        import threading
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.reader = threading.Thread(target=lambda: self.lines.extend(self.proc.stdout), daemon=True)
        self.reader.start()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)
        rows = []
        for line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- distributed

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """Slowest rank's value (every rank gets it)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_rank, world, ms_per_step):
    """Units processed by all ranks per second, timed by the slowest rank."""
    return units_per_rank * world / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------- our implementation

def build_layer(shape_key, seed, rank):
    import numpy as np
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    s = SHAPES[shape_key]
    T, H, I, E, k = s["T"], s["H"], s["I"], s["E"], s["top_k"]
    wl = (W.prefill_moe if shape_key == "prefill" else W.decode_moe)(seed=seed + rank, with_weights=False)
    hidden = torch.from_numpy(wl.hidden.view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.from_numpy(wl.logits).cuda()
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + seed)
    w13 = (torch.randn((E, 2 * I, H), generator=g, device="cuda", dtype=torch.float32) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn((E, H, I), generator=g, device="cuda", dtype=torch.float32) * 0.02).to(torch.bfloat16)
    weights = api.quantize_moe_weights(w13, w2)
    del w13, w2
    fwd = api.MoEForward(T, H, I, E, k)
    a1, a2 = fwd.calibrate(hidden, logits, weights, GATE_LIMIT, UP_LIMIT)
    torch.cuda.synchronize()
    return dict(T=T, H=H, I=I, E=E, k=k, hidden=hidden, logits=logits, w=weights, fwd=fwd, a1=a1, a2=a2,
                wl=wl)


def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    B.nvfp4_moe_set_swap_l2(args.swap_l2)
    L = build_layer(args.workload, args.seed, rank)
    T, H, I, E, k = L["T"], L["H"], L["I"], L["E"], L["k"]
    fwd, w = L["fwd"], L["w"]
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        fwd(L["hidden"], L["logits"], w, L["a1"], L["a2"], GATE_LIMIT, UP_LIMIT, out=out)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()

    # ---- device-resident timed region (no per-stage events: an event record
    # between two kernels would stop the next one from starting early)
    clocks = ClockSampler(local)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(ms, world)

    # ---- the same forward replayed from a CUDA graph (captured after the eager
    # warm-up; launch overhead leaves the host entirely)
    g_stream = torch.cuda.Stream()
    g_stream.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=g_stream):
        fwd(L["hidden"], L["logits"], w, L["a1"], L["a2"], GATE_LIMIT, UP_LIMIT, out=out, stream=g_stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world)
    del graph

    # ---- the forward with no L2 activation scales given: L1 keeps bf16 h and
    # its per-expert amax, a quantize pass derives the scales from this batch
    def step_batch_scale():
        fwd(L["hidden"], L["logits"], w, L["a1"], None, GATE_LIMIT, UP_LIMIT, out=out)

    for _ in range(3):
        step_batch_scale()
    n_bs = max(1, min(args.steps, 100))
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(n_bs):
        step_batch_scale()
    b1.record(stream)
    torch.cuda.synchronize()
    batch_scale_ms = max_over_ranks(b0.elapsed_time(b1) / n_bs, world)

    # the same with the L1 output kept as FP8 blocks instead of bf16
    def step_batch_scale_fp8():
        fwd(L["hidden"], L["logits"], w, L["a1"], None, GATE_LIMIT, UP_LIMIT, out=out, l1_output="fp8")

    for _ in range(3):
        step_batch_scale_fp8()
    b0.record(stream)
    for _ in range(n_bs):
        step_batch_scale_fp8()
    b1.record(stream)
    torch.cuda.synchronize()
    batch_scale_fp8_ms = max_over_ranks(b0.elapsed_time(b1) / n_bs, world)

    # ---- per-stage breakdown in a separate pass, events recorded by the library
    # on the launching stream before each stage
    n_stage = max(1, min(args.steps, 20))
    stage_events = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n_stage)]
    for evs in stage_events:  # torch creates the CUDA event on its first record
        for ev in evs:
            ev.record(stream)
    torch.cuda.synchronize()
    for i in range(n_stage):
        B.nvfp4_moe_set_stage_events(stage_events[i])
        step()
    torch.cuda.synchronize()
    B.nvfp4_moe_set_stage_events(None)
    names = ["route", "slot_scan", "slot_scatter", "gather_quantize", "l1_gemm_swiglu_quant", "l2_gemm_weighted",
             "token_combine"]
    stages = {n: statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in stage_events) for i, n in enumerate(names)}
    staged_ms = statistics.mean(ev[0].elapsed_time(ev[7]) for ev in stage_events)

    # ---- end to end through the C ABI with pinned host buffers
    h_hidden = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    h_hidden.copy_(L["hidden"].cpu())
    h_logits = torch.empty((T, E), dtype=torch.float32, pin_memory=True)
    h_logits.copy_(L["logits"].cpu())
    h_out = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    # the library's host pipeline: every step uploads its inputs, runs the
    # forward and downloads its output; the upload of step i+1 and the
    # download of step i-1 overlap the forward of step i (three streams)
    from nvfp4_mixture_experts_expert_gb300 import api
    pipe = api.HostPipeline(fwd, w, L["a1"], L["a2"], GATE_LIMIT, UP_LIMIT)
    for _ in range(3):
        pipe.submit(h_hidden, h_logits, h_out)
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_in)  # before the first upload
    for _ in range(args.steps):
        pipe.submit(h_hidden, h_logits, h_out)
    e1.record(pipe.s_out)  # after the last download
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    status = max(B.nvfp4_device_status(), fwd.status(), pipe.fwd.status(stream=pipe.s_comp))
    P = int(fwd.view("meta", torch.int32, 1).cpu()[0])

    # ---- roofline of the dominant kernel (L1 grouped GEMM).  Its duration comes
    # from the short stage pass (n_stage forwards, ~16 ms at full clocks), so
    # the burst peak applies: measured bf16 burst x the nominal FP4/BF16 ratio.
    peaks = measured_peaks()
    fp4_peak = fp4_peak_burst(peaks)
    A = T * k
    l1_flops = 2.0 * A * H * (2 * I)
    l2_flops = 2.0 * A * I * H
    l1_tflops = l1_flops / (stages["l1_gemm_swiglu_quant"] * 1e-3) / 1e12
    l2_tflops = l2_flops / (stages["l2_gemm_weighted"] * 1e-3) / 1e12
    traffic = stored_traffic("l1_gemm_swiglu_quant_" + args.workload)
    roofline = {"kernel": "l1_gemm_swiglu_quant", "bound": "tensor", "achieved": round(l1_tflops, 1),
                "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(l1_tflops / fp4_peak, 4),
                "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} TFLOP/s x "
                               f"{FP4_OVER_BF16:g} (nominal dense FP4/BF16 ratio)",
                "peak_choice": f"burst: the kernel is timed in a {n_stage}-forward pass of "
                               f"{n_stage * staged_ms:.0f} ms at full clocks",
                "frac_nominal": round(l1_tflops / NOMINAL_FP4_TFLOPS, 4),
                "flops_per_launch": l1_flops, "flops_rule": "2*T*top_k*H*2I (real rows only)"}
    res = {
        "metric": METRIC, "value": round(whole_job_throughput(T, world, ms), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1 block-scaled, fp32 accumulate)", "data": "synthetic",
        "config": {"workload": workload_name(args.workload), "tokens_per_gpu": T, "hidden": H,
                   "intermediate": I, "experts": E, "top_k": k, "padded_rows": P,
                   "parallelism": f"dp{world} over tokens (replicated local experts)",
                   "swapped_l2": bool(args.swap_l2),
                   "l2_flush": "not needed: weights (0.76 GB NVFP4) and activations exceed the 129 MB L2"},
        "roofline": roofline,
        "stages_ms": {n: round(v, 4) for n, v in stages.items()},
        "stages_note": f"separate pass of {n_stage} forwards with an event before each stage "
                       f"({staged_ms:.4f} ms per forward there)",
        "l2_gemm": {"achieved": round(l2_tflops, 1), "unit": "TFLOP/s", "frac": round(l2_tflops / fp4_peak, 4),
                    "frac_nominal": round(l2_tflops / NOMINAL_FP4_TFLOPS, 4)},
        "cuda_graph": {"value": round(whole_job_throughput(T, world, graph_ms), 1), "unit": UNIT,
                       "ms_per_step": round(graph_ms, 4),
                       "note": "the same forward captured once into a CUDA graph and replayed"},
        "batch_l2_scale": {"value": round(whole_job_throughput(T, world, batch_scale_ms), 1), "unit": UNIT,
                           "ms_per_step": round(batch_scale_ms, 4),
                           "note": f"{n_bs} forwards with a2_gs NULL: bf16 L1 output + per-expert amax, "
                                   "then a quantize pass with scales from the batch (8 launches + 1 memset)"},
        "batch_l2_scale_fp8": {"value": round(whole_job_throughput(T, world, batch_scale_fp8_ms), 1), "unit": UNIT,
                               "ms_per_step": round(batch_scale_fp8_ms, 4),
                               "note": f"{n_bs} forwards as batch_l2_scale with the L1 output kept as FP8 blocks "
                                       "(E4M3, a power-of-two scale per 16 features) instead of bf16"},
        "e2e": {"value": round(whole_job_throughput(T, world, e2e_ms), 1), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": pipe.h2d_bytes, "d2h_bytes_per_step": pipe.d2h_bytes,
                "mode": "api.HostPipeline: pinned host inputs uploaded and output downloaded every step; "
                        "upload of step i+1 and download of step i-1 overlap the forward of step i"},
        "clocks": clk,
        "gpu_launches": 7 * args.steps,
        "device_status": status,
    }
    return res, L


def linear_side_measurement(seed):
    """The dense NVFP4 linear (M=2048, K=3584, N=6144) and the grouped linear
    (G=8, T=2048, D=2048 -> R=1024, strided (T,G,D) in, (T,G,R) out): amax ->
    global scale -> quantization of the activations, then the block-scaled
    GEMM; weights quantized once beforehand.  L2 flushed before each step
    (these inputs fit in L2)."""
    import numpy as np
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    peaks = measured_peaks()
    fp4_peak = fp4_peak_burst(peaks)  # each GEMM is timed alone, in a few-ms window
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def bf16(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    def timed(fn, gemm_ev):
        for _ in range(3):
            fn()
        tot, gem = [], []
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        for _ in range(20):
            flush.fill_(1)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot.append(a.elapsed_time(b))
            gem.append(gemm_ev[0].elapsed_time(gemm_ev[1]))
        return statistics.median(tot), statistics.median(gem)

    res = {}
    # dense linear
    wl = W.dense_gemm(seed)
    M, N, K = wl.M, wl.N, wl.K
    a = bf16(wl.a)
    fb, sfb, gb = api.quantize(bf16(wl.b))
    fa = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sfa = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
    ga = torch.empty(1, dtype=torch.float32, device="cuda")
    wsb = B.nvfp4_quantize_workspace_size(1)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    offs = torch.tensor([0, M], dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def dense():
        B.nvfp4_quantize(a, M, K, K, 0, 1, None, ga, ws, wsb, fa, sfa, M)
        ev[0].record()
        B.nvfp4_grouped_gemm(fa, sfa, ga, fb, sfb, gb, offs, None, 1, M, N, K, D, N, 0)
        ev[1].record()

    ms, gms = timed(dense, ev)
    flops = 2.0 * M * N * K
    res["dense_linear"] = {"workload": "NVFP4 linear M=2048 K=3584 N=6144 (activation quantized per call)",
                           "ms_per_call": round(ms, 4), "gemm_ms": round(gms, 4),
                           "gemm_tflops": round(flops / (gms * 1e-3) / 1e12, 1),
                           "gemm_frac_fp4": round(flops / (gms * 1e-3) / 1e12 / fp4_peak, 4),
                           "gemm_frac_fp4_nominal": round(flops / (gms * 1e-3) / 1e12 / NOMINAL_FP4_TFLOPS, 4)}
    # grouped linear
    gl = W.grouped_linear(seed)
    T, G, Dd, R = gl.T, gl.G, gl.D, gl.R
    x = bf16(gl.x)
    fw, sfw, gw = api.quantize_expert_weights(bf16(gl.w), gs=torch.from_numpy(gl.w_gs).cuda())
    fx = torch.empty((G * T, Dd // 2), dtype=torch.uint8, device="cuda")
    sfx = torch.empty(G * T * Dd // 16, dtype=torch.uint8, device="cuda")
    gx = torch.empty(G, dtype=torch.float32, device="cuda")
    wsg = B.nvfp4_quantize_workspace_size(G)
    wsx = torch.empty(wsg, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, G, R), dtype=torch.bfloat16, device="cuda")
    goffs = torch.arange(G + 1, dtype=torch.int32, device="cuda") * T
    gcnt = torch.full((G,), T, dtype=torch.int32, device="cuda")

    def grouped():
        B.nvfp4_quantize(x, T, Dd, G * Dd, Dd, G, None, gx, wsx, wsg, fx, sfx, T)
        ev[0].record()
        B.nvfp4_grouped_gemm(fx, sfx, gx, fw, sfw, gw, goffs, gcnt, G, G * T, R, Dd, out, G * R, R)
        ev[1].record()

    ms, gms = timed(grouped, ev)
    flops = 2.0 * G * T * R * Dd
    gbytes = G * T * Dd * (1 / 2 + 1 / 16) + G * R * Dd * (1 / 2 + 1 / 16) + G * T * R * 2
    res["grouped_linear"] = {"workload": "NVFP4 grouped linear G=8 T=2048 D=2048 R=1024, strided (T,G,D) -> (T,G,R)",
                             "ms_per_call": round(ms, 4), "gemm_ms": round(gms, 4),
                             "gemm_tflops": round(flops / (gms * 1e-3) / 1e12, 1),
                             "gemm_frac_fp4": round(flops / (gms * 1e-3) / 1e12 / fp4_peak, 4),
                             "gemm_gbs": round(gbytes / (gms * 1e-3) / 1e9, 1),
                             "gemm_frac_hbm": round(gbytes / (gms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                             "gemm_frac_hbm_nominal": round(gbytes / (gms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4)}
    # shared expert: the same SwiGLU FFN on every token (one group, no routing)
    swl = W.moe_workload(8192, 4096, 2048, 1, 1, seed, with_weights=False)
    rng = np.random.default_rng(seed + 1)
    w13 = torch.from_numpy((rng.standard_normal((1, 4096, 4096), dtype=np.float32) * np.float32(0.02))).cuda()
    w2 = torch.from_numpy((rng.standard_normal((1, 4096, 2048), dtype=np.float32) * np.float32(0.02))).cuda()
    sw = api.quantize_moe_weights(w13.to(torch.bfloat16), w2.to(torch.bfloat16))
    sh = bf16(swl.hidden)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    a1s = torch.full((1,), 2688.0 / float(sh.abs().max()), dtype=torch.float32, device="cuda")
    se = api.SharedExpertForward(8192, 4096, 2048)
    sout = torch.empty((8192, 4096), dtype=torch.bfloat16, device="cuda")
    se_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def shared():
        se_ev[0].record()
        se(sh, sw, a1s, one * 200.0, GATE_LIMIT, UP_LIMIT, out=sout)  # fixed L2 scale: timing only
        se_ev[1].record()

    ms, _ = timed(shared, se_ev)
    flops = 2.0 * 8192 * 4096 * 2048 * 3
    res["shared_expert"] = {"workload": "shared-expert NVFP4 SwiGLU FFN T=8192 H=4096 I=2048 (quantize + L1 + L2)",
                            "ms_per_call": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                            "frac_fp4": round(flops / (ms * 1e-3) / 1e12 / fp4_peak, 4)}
    res["l2"] = "flushed (512 MB write) before each call"
    res["peak"] = f"FP4 {fp4_peak:.1f} TFLOP/s ({peaks['source']} bf16 burst x {FP4_OVER_BF16:g}); " \
                  f"HBM {peaks['hbm_gbs']} GB/s ({peaks['source']} copy)"
    return res


MMA_SHAPES = {0: ("cta_group::1 128x256", 128, 256), 1: ("cta_group::2 256x256", 256, 256),
              2: ("cta_group::2 256x128", 256, 128), 3: ("cta_group::1 128x128", 128, 128)}


MMA_RATE_FLAGS = 128  # nvfp4_debug_mma_rate: the MMA loop on the whole warp with one elected lane issuing


def fp4_ceiling_measurement(local):
    """The bare block-scaled FP4 MMA stream (nvfp4_debug_mma_rate) on every SM,
    per tile shape, on operands made by the library's quantizer: CUDA events
    around 10 launches of ~20 ms each, SM clocks sampled meanwhile."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api, binding as B
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    a = torch.randn((256, 1024), generator=g, device="cuda").to(torch.bfloat16)
    b = (torch.randn((512, 1024), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    fa, sfa, _ = api.quantize(a)
    fb, sfb, _ = api.quantize(b)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    res = {}
    for shape, (name, m, n) in MMA_SHAPES.items():
        units = sms // 2 if m == 256 else sms
        flop_iter = 2.0 * m * n * 256
        iters = 4096
        args = (fa, fa.numel(), sfa, sfa.numel(), fb, fb.numel(), sfb, sfb.numel(), shape, units)
        B.nvfp4_debug_mma_rate(*args, iters, MMA_RATE_FLAGS)  # warm-up
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        B.nvfp4_debug_mma_rate(*args, iters, MMA_RATE_FLAGS)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        iters = max(1, min(1 << 21, int(iters * 20.0 / max(ms, 1e-3))))  # ~20 ms per launch
        clk = ClockSampler(local)
        e0.record()
        for _ in range(10):
            B.nvfp4_debug_mma_rate(*args, iters, MMA_RATE_FLAGS)
        e1.record()
        torch.cuda.synchronize()
        c = clk.stop()
        ms = e0.elapsed_time(e1) / 10
        tflops = units * iters * flop_iter / (ms * 1e-3) / 1e12
        res[name] = {"tflops": round(tflops, 1), "ms_per_launch": round(ms, 3), "units": units, "iters": iters,
                     "sm_mhz": c["sm_mhz"] if c else None, "reasons": c["reasons"] if c else None}
    res["status"] = B.nvfp4_device_status()
    res["note"] = ("bare MMA stream: 4 operand sets staged once per CTA, iters x 4 back-to-back MMAs (K=64) "
                   "into one accumulator, issued as the GEMM issues them (warp-uniform loop, one elected lane), "
                   "no loads, hand-offs or epilogue")
    return res


def tiny_side_measurement(seed):
    """The tiny layer (T=64, H=256, I=128, E=8, top_k=2): latency-bound; eager
    and CUDA-graph forward latency over 200 forwards (everything fits in L2)."""
    import numpy as np
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    wl = W.tiny_moe(seed)
    hidden = torch.from_numpy(wl.hidden.view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.from_numpy(wl.logits).cuda()
    w = api.quantize_moe_weights(torch.from_numpy(wl.w13.view(np.int16)).view(torch.bfloat16).cuda(),
                                 torch.from_numpy(wl.w2.view(np.int16)).view(torch.bfloat16).cuda())
    fwd = api.MoEForward(wl.T, wl.H, wl.I, wl.E, wl.top_k)
    a1, a2 = fwd.calibrate(hidden, logits, w)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    cur = torch.cuda.current_stream()

    def step(stream=None):
        fwd(hidden, logits, w, a1, a2, GATE_LIMIT, UP_LIMIT, out=out, stream=stream)

    for _ in range(10):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(200):
        step()
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 200
    gs = torch.cuda.Stream()
    gs.wait_stream(cur)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        step(stream=gs)
    for _ in range(10):
        graph.replay()
    torch.cuda.synchronize()
    e0.record(cur)
    for _ in range(200):
        graph.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    gms = e0.elapsed_time(e1) / 200
    return {"workload": "tiny NVFP4 MoE layer forward T=64 H=256 I=128 E=8 top_k=2 (5% zero, 5% tiny blocks)",
            "latency_us": round(ms * 1e3, 2), "tokens_per_s": round(wl.T / (ms * 1e-3), 1),
            "cuda_graph": {"latency_us": round(gms * 1e3, 2), "tokens_per_s": round(wl.T / (gms * 1e-3), 1)},
            "note": "back-to-back forwards on one stream; launch-latency bound"}


def decode_side_measurement(seed):
    """Decode-size forward (T=128, E=32): HBM-bound weight streaming."""
    import torch
    L = build_layer("decode", seed, 0)
    fwd, w = L["fwd"], L["w"]
    out = torch.empty((L["T"], L["H"]), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")

    def flush_l2():
        # evict the weights: write 512 MB, then read 256 MB so that the lines
        # left in L2 are clean (no write-back traffic lands in the timed step)
        flush.fill_(1)
        flush_rd.max()

    def step(stream=None):
        fwd(L["hidden"], L["logits"], w, L["a1"], L["a2"], GATE_LIMIT, UP_LIMIT, out=out, stream=stream)

    from nvfp4_mixture_experts_expert_gb300 import binding as B
    for _ in range(5):
        step()
    times, stage_times, graph_times = [], [], []
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    for _ in range(20):
        flush_l2()
        a.record()
        step()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    # the same step replayed from a CUDA graph (no host launch work in the step)
    cur = torch.cuda.current_stream()
    g_stream = torch.cuda.Stream()
    g_stream.wait_stream(cur)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=g_stream):
        step(stream=g_stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for _ in range(20):
        flush_l2()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        graph_times.append(a.elapsed_time(b))
    graph_ms = statistics.median(graph_times)
    del graph
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for ev in evs:  # materialise the CUDA events (torch creates them on first record)
        ev.record()
    torch.cuda.synchronize()
    for _ in range(10):  # separate pass: per-stage events (they serialise the kernels)
        flush_l2()
        B.nvfp4_moe_set_stage_events(evs)
        step()
        B.nvfp4_moe_set_stage_events(None)
        torch.cuda.synchronize()
        stage_times.append([evs[i].elapsed_time(evs[i + 1]) for i in range(7)])
    names = ["route", "slot_scan", "slot_scatter", "gather_quantize", "l1_gemm_swiglu_quant", "l2_gemm_weighted",
             "token_combine"]
    stages = {n: round(statistics.median(st[i] for st in stage_times), 4) for i, n in enumerate(names)}
    counts = fwd.view("counts", torch.int32, L["E"]).cpu()
    active = [e for e in range(L["E"]) if int(counts[e]) > 0]
    H, I = L["H"], L["I"]
    wbytes = len(active) * (2 * I * H // 2 + 2 * I * H // 16 + H * I // 2 + H * I // 16)
    peaks = measured_peaks()
    gbs = wbytes / (ms * 1e-3) / 1e9
    return {"workload": workload_name("decode"), "ms_per_step": round(ms, 4),
            "tokens_per_s": round(L["T"] / (ms * 1e-3), 1), "active_experts": len(active),
            "weight_bytes": wbytes, "weight_stream_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
            "cuda_graph": {"ms_per_step": round(graph_ms, 4),
                           "weight_stream_gbs": round(wbytes / (graph_ms * 1e-3) / 1e9, 1),
                           "hbm_frac": round(wbytes / (graph_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
            "stages_ms": stages,
            "l2": "flushed before each step (512 MB write, then 256 MB read: clean lines left)"}


# --------------------------------------------------------------------------- CPU oracle (baseline / reference arm)

def oracle_prepare(shape_key, seed):
    """Inputs of the oracle's forward over one whole batch of a MoE workload
    (untimed): hidden states and router logits from the seeded generators,
    NVFP4 expert weights drawn directly as random codes (the oracle's cost
    does not depend on their values, and drawing them skips minutes of CPU
    weight quantization), fixed activation global scales."""
    import numpy as np
    from oracle import nvfp4_oracle as O
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    sh = SHAPES[shape_key]
    T, H, I, E, k = sh["T"], sh["H"], sh["I"], sh["E"], sh["top_k"]
    wl = (W.prefill_moe if shape_key == "prefill" else W.decode_moe)(seed=seed, with_weights=False)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    return dict(T=T, H=H, I=I, E=E, k=k, hidden=hidden, logits=wl.logits,
                w13q=W.random_nvfp4_codes(E, 2 * I, H, seed + 11), w2q=W.random_nvfp4_codes(E, H, I, seed + 12),
                a1=np.full(E, O.global_scale(np.abs(hidden).max()), np.float32), a2=np.full(E, 200.0, np.float32))


def oracle_piece(st, experts, first, last):
    """One piece of the oracle's MoE forward on a prepared batch, in the
    oracle's own steps and order: the first piece routes and sorts the slots,
    each piece runs the per-expert steps (quantize, L1, SwiGLU, requantize,
    L2, routing-weighted accumulate) for its experts, the last rounds the sum
    to bf16 and returns it.  Consecutive pieces over all experts are one call
    of the oracle's moe_forward (checked on the CPU by the tests)."""
    import numpy as np
    from oracle import nvfp4_oracle as O
    if first:
        ids, w = O.route(st["logits"], st["k"])
        st["meta"] = O.sort_slots(ids, w, st["E"])
        st["acc"] = np.zeros((st["T"], st["H"]), dtype=np.float64)
    meta, w13q, w2q = st["meta"], st["w13q"], st["w2q"]
    quiet = np.errstate(over="ignore")  # random weight codes: exp(-g) may overflow to inf (SiLU -> 0)
    quiet.__enter__()
    for e in experts:
        lo, n = int(meta["offsets"][e]), int(meta["counts"][e])
        if n == 0:
            continue
        toks = meta["sorted_token_ids"][lo:lo + n]
        h = O.expert_l1(st["hidden"][toks], st["a1"][e], w13q[0][e], w13q[1][e], w13q[2][e], GATE_LIMIT, UP_LIMIT)
        Y = O.expert_l2(h, st["a2"][e], w2q[0][e], w2q[1][e], w2q[2][e])
        np.add.at(st["acc"], toks, meta["row_weight"][lo:lo + n, None] * Y)
    quiet.__exit__(None, None, None)
    if last:
        return O.bf16_round(st["acc"].astype(np.float32))
    return None


def expert_pieces(E, n_pieces):
    """Experts 0..E-1 in n_pieces consecutive groups of nearly equal size
    (some groups are empty when n_pieces > E)."""
    return [list(range(E * i // n_pieces, E * (i + 1) // n_pieces)) for i in range(n_pieces)]


def _cpu_seconds():
    t = os.times()
    return t.user + t.system


def oracle_timed_pieces(st, n_pieces, warmup=0):
    """Time one whole batch of the oracle's forward as n_pieces consecutive
    pieces (see oracle_piece).  Warm-up runs the routing and slot sort only.
    Returns (seconds per piece, process CPU seconds, output)."""
    for _ in range(warmup):
        oracle_piece(st, [], True, False)
    groups = expert_pieces(st["E"], n_pieces)
    times, out = [], None
    c0 = _cpu_seconds()
    for i, g in enumerate(groups):
        t0 = time.perf_counter()
        r = oracle_piece(st, g, i == 0, i == len(groups) - 1)
        times.append(time.perf_counter() - t0)
        out = r if r is not None else out
    return times, _cpu_seconds() - c0, out


def cpu_threads_available():
    n = os.environ.get("OMP_NUM_THREADS") or os.environ.get("OPENBLAS_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)


def _cores_used(cpu_s, wall_s):
    """Threads the run actually kept busy on average: process CPU time / wall time."""
    return round(cpu_s / wall_s, 1) if wall_s > 0 else None


def cpu_baseline(shape_key, seed):
    """The oracle's forward over the whole batch, timed in one piece."""
    st = oracle_prepare(shape_key, seed)
    times, cpu_s, _ = oracle_timed_pieces(st, 1)
    wall = sum(times)
    T = SHAPES[shape_key]["T"]
    return {"value": round(T / wall, 2), "unit": UNIT, "cores": _cores_used(cpu_s, wall),
            "threads_available": cpu_threads_available(), "kind": "oracle", "seconds": round(wall, 2),
            "sample": f"the whole batch: one oracle forward over all {T} tokens and {SHAPES[shape_key]['E']} "
                      "experts (routing, slot sort, per-expert quantize/L1/SwiGLU/requantize/L2, combine), "
                      "no extrapolation; weights are random NVFP4 codes"}


def oracle_side_baselines(seed):
    """The oracle timed on the other workloads, each once on the whole
    workload: decode layer, tiny layer, dense linear, grouped linear, shared
    expert (the per-call work: activation quantization with its amax-derived
    global scale and the GEMM; weights given as NVFP4 codes)."""
    import numpy as np
    from oracle import nvfp4_oracle as O
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    res = {}

    def timed(fn):
        c0, t0 = _cpu_seconds(), time.perf_counter()
        fn()
        wall = time.perf_counter() - t0
        return wall, _cores_used(_cpu_seconds() - c0, wall)

    st = oracle_prepare("decode", seed)
    wall, cores = timed(lambda: oracle_timed_pieces(st, 1))
    res["decode"] = {"value": round(st["T"] / wall, 2), "unit": UNIT, "seconds": round(wall, 3), "cores": cores}
    del st
    tw = W.tiny_moe(seed)
    w13q = O.quantize_expert_weights(W.bf16_bits_to_f32(tw.w13))
    w2q = O.quantize_expert_weights(W.bf16_bits_to_f32(tw.w2))
    th = W.bf16_bits_to_f32(tw.hidden)
    a = np.full(tw.E, O.global_scale(np.abs(th).max()), np.float32)
    wall, cores = timed(lambda: O.moe_forward(th, tw.logits, tw.top_k, w13q, w2q, a, a * 0 + 200.0))
    res["tiny"] = {"value": round(tw.T / wall, 2), "unit": UNIT, "latency_us": round(wall * 1e6, 1),
                   "seconds": round(wall, 4), "cores": cores}
    dg = W.dense_gemm(seed)
    a32 = W.bf16_bits_to_f32(dg.a)
    bq = W.random_nvfp4_codes(1, dg.N, dg.K, seed + 21)

    def dense():
        gs = O.global_scale(np.abs(a32).max())
        an, asc = O.quantize_blocks(a32, gs)
        O.nvfp4_gemm(an, asc, gs, bq[0][0], bq[1][0], bq[2][0])

    wall, cores = timed(dense)
    res["dense_linear"] = {"ms_per_call": round(wall * 1e3, 1),
                           "tflops": round(2.0 * dg.M * dg.N * dg.K / wall / 1e12, 4), "seconds": round(wall, 3),
                           "cores": cores}
    gw = W.grouped_linear(seed)
    gx = W.bf16_bits_to_f32(gw.x)
    wq = W.random_nvfp4_codes(gw.G, gw.R, gw.D, seed + 22)

    def grouped():
        for g in range(gw.G):
            xg = gx[:, g, :]
            gs = O.global_scale(np.abs(xg).max())
            an, asc = O.quantize_blocks(xg, gs)
            O.nvfp4_gemm(an, asc, gs, wq[0][g], wq[1][g], wq[2][g])

    wall, cores = timed(grouped)
    res["grouped_linear"] = {"ms_per_call": round(wall * 1e3, 1),
                             "tflops": round(2.0 * gw.G * gw.T * gw.R * gw.D / wall / 1e12, 4),
                             "seconds": round(wall, 3), "cores": cores}
    sh = W.bf16_bits_to_f32(W.moe_workload(8192, 4096, 2048, 1, 1, seed, with_weights=False).hidden)
    s13 = W.random_nvfp4_codes(1, 4096, 4096, seed + 23)
    s2 = W.random_nvfp4_codes(1, 4096, 2048, seed + 24)
    wall, cores = timed(lambda: O.shared_expert_forward(sh, s13, s2, O.global_scale(np.abs(sh).max()),
                                                         np.float32(200.0), GATE_LIMIT, UP_LIMIT))
    res["shared_expert"] = {"ms_per_call": round(wall * 1e3, 1), "value": round(8192 / wall, 2), "unit": UNIT,
                            "seconds": round(wall, 3), "cores": cores}
    res["kind"] = "oracle"
    res["threads_available"] = cpu_threads_available()
    return res


def run_reference(args):
    """The reference arm: the CPU oracle (the only other implementation of
    this method), timed over exactly one whole batch split into `steps`
    consecutive pieces (warm-up: the routing and slot sort, untimed)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    st = oracle_prepare(args.workload, args.seed)
    times, cpu_s, _ = oracle_timed_pieces(st, max(args.steps, 1), warmup=args.warmup)
    wall = sum(times)
    T = SHAPES[args.workload]["T"]
    value = T / wall
    sample = (f"one whole batch ({T} tokens, all {st['E']} experts) as {len(times)} consecutive pieces, one per "
              f"step; warm-up: routing + slot sort; no extrapolation; weights are random NVFP4 codes")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / len(times) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle; fp32 quantizer)",
            "data": "synthetic", "config": {"workload": workload_name(args.workload)},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": _cores_used(cpu_s, wall),
                             "threads_available": cpu_threads_available(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    args = parse()
    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    world, rank, local = dist_setup()
    res, _ = run_ours(args, world, rank, local)
    if rank == 0:
        if not args.no_extras and world == 1:
            res["extra"] = {"decode": decode_side_measurement(args.seed), "linear": linear_side_measurement(args.seed),
                            "tiny": tiny_side_measurement(args.seed), "fp4_mma_ceiling": fp4_ceiling_measurement(local)}
            ceil = res["extra"]["fp4_mma_ceiling"].get(MMA_SHAPES[0][0], {}).get("tflops")
            if ceil:
                res["roofline"]["measured_fp4_mma_ceiling"] = ceil
                res["roofline"]["frac_of_measured_ceiling"] = round(res["roofline"]["achieved"] / ceil, 4)
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload, args.seed)
            if not args.no_extras and world == 1:
                res["extra"]["cpu_baseline"] = oracle_side_baselines(args.seed)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
