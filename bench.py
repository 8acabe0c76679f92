"""Benchmark of the FP8 W8A8 linear on one GB300 (or N independent replicas).

Headline workload (one "step"): the four Llama-3-8B decoder linears (qkv 4096->6144,
o_proj 4096->4096, gate_up 4096->28672, down 14336->4096) at M = 16384 tokens with
per-output-channel weight scales and a dynamic per-tensor activation scale, i.e. per
layer: amax(A) -> e4m3 cast -> tcgen05 FP8 GEMM -> channelwise rescale epilogue -> bf16 Y.
value = sum(2*M*N*K) / step time in TFLOP/s, inputs resident in HBM.

Also reported on the same line:
  decode    weight GB/s of the split-K GEMV on the Mistral-7B layers at M in {1,2,4,8,15}
            (per-tensor scales), rotating through weight copies so L2 never holds them;
  roofline  the GEMM kernel's achieved TFLOP/s (fp8_scaled_mm launches timed with CUDA
            events) against the FP8 dense peak;
  e2e       the same step through the C-ABI call with host buffers: pinned host->device
            copy of A, fp8_linear_channelwise, device->host copy of Y, per layer;
  cpu_baseline  the CPU oracle on a bounded sample of the workload.

  sweep     the TinyLlama-1.1B decoder-stack sweep (22 layers x 4 linears, both weight
            modes, M from 1 to 16384): per-M time, TFLOP/s, weight-GB/s, roofline fraction;
  crossover GEMV against GEMM at M around 16 on the Mistral-7B and TinyLlama linears;
  unaligned weight-GB/s of the four shapes whose dimensions are not multiples of 16;
  tiny      latency of the 16 x 256 x 256 linear.

`--impl reference` times the CPU oracle alone on that bounded sample (rank 0 only).
One GPU only: the library's pair GEMM uses cluster-scoped operations meant for a single
device, and the path is not sharded, so a launch with more than one process (torchrun,
WORLD_SIZE > 1) or --gpus > 1 prints an "unavailable" line and does no GPU work.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 W8A8 linear TFLOP/s (prefill) and weight GB/s (decode M<16) vs roofline"
NOMINAL_FP8_OVER_BF16 = 2.0  # 4.5 PF fp8 / 2.25 PF bf16 dense (nominal)
NOMINAL_HBM_GBS = 8000.0     # the HBM3e rate GB300 is specified at (context beside the measured copy rate)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# clocks: nvidia-smi sampled during the timed regions
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def selected_layers(names):
    from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
    return [(i, L) for i, L in enumerate(I.LLAMA8B_LAYERS) if names is None or L.name in names]


def prefill_inputs(M: int, names=None):
    from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
    return [(L, I.prefill_activations(i, M=M), I.prefill_weight(i)) for i, L in selected_layers(names)]


def source_digest(path: str) -> str:
    """sha256 of a CUDA source with comments and whitespace removed: a recorded counter capture
    stays valid across comment-only edits and lapses with any change to the code itself."""
    import hashlib
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return hashlib.sha256(re.sub(r"\s+", "", text).encode()).hexdigest()


def gemm_traffic(layers):
    """Mean DRAM bytes per GEMM launch from the committed ncu summary, if that summary was taken
    on the current GEMM code (else None: the counters no longer describe this kernel)."""
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_tcgen05_dram_llama8b_m16384.json")) as f:
            rec = json.load(f)
        src = os.path.join(ROOT, "fp8_w8a8_quantized_dynamic_gb300", "csrc", "gemm_tcgen05.cu")
        if source_digest(src) != rec["gemm_code_digest"]:
            return None, None
        per = {L.name: rec["per_launch_bytes"][L.name] for L in layers}
        return sum(per.values()) / len(per), per
    except (OSError, KeyError, ValueError):
        return None, None


def flops(M, layers):
    return sum(2.0 * M * L.N * L.K for L in layers)


def time_loop(torch, fn, steps: int, warmup: int):
    """Median-free timing: W warm-up calls, then K calls between two events (both synced)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps  # ms per call


def graph_of(torch, fn):
    """Capture fn (already warmed up) into a CUDA graph; decode steps are launch-bound."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def measure_variants(torch, F, I, args, dev, layers, names, host, A, Y, ws, M):
    """Prefill TFLOP/s and decode weight GB/s of the wider calls on the headline workloads:
    float8_e5m2 for both operands (dynamic scale), e4m3 with a static activation scale (the
    calibrated value is the dynamic scale of the same activations), and the weight-only path
    (bf16 activations, e4m3 weights up-converted to bf16)."""
    out = {}
    steps = max(3, args.steps // 4)
    W5 = [F.fp8_quantize_weight_ex(w.to(dev), "e5m2", per_channel=True) for _, _, w in host]
    W4 = [F.fp8_quantize_weight(w.to(dev), per_channel=True) for _, _, w in host]
    S = [F.fp8_quantize_act(a)[1] for a in A]
    torch.cuda.synchronize()
    total = flops(M, layers)

    def pre_e5m2():
        for i in range(len(layers)):
            F.fp8_linear_ex(A[i], W5[i][0], W5[i][1], per_channel=True, out=Y[i], ws=ws, fmt_a="e5m2",
                            fmt_w="e5m2")

    def pre_static():
        for i in range(len(layers)):
            F.fp8_linear_static(A[i], S[i], W4[i][0], W4[i][1], per_channel=True, out=Y[i], ws=ws)

    ws_wo = torch.empty(max(F.fp8_weight_only_workspace_bytes(M, L.K, L.N) for L in layers), dtype=torch.uint8,
                        device=dev)

    def pre_weight_only():
        for i in range(len(layers)):
            F.fp8_linear_weight_only(A[i], W4[i][0], W4[i][1], per_channel=True, out=Y[i], ws=ws_wo)

    for name, fn in (("e5m2_dynamic", pre_e5m2), ("e4m3_static", pre_static), ("weight_only_e4m3", pre_weight_only)):
        t = time_loop(torch, fn, steps, 2)
        out[name] = {"prefill_tflops": round(total / (t * 1e-3) / 1e12, 1), "prefill_ms_per_step": round(t, 4)}
    out["weight_only_e4m3"]["note"] = ("bf16 A x up-converted bf16 W on tcgen05 kind::f16 (the up-conversion pass "
                                       "is inside the step); compare with the bf16 peak, not the FP8 one")
    del W5, W4, ws_wo
    if not args.no_decode:
        li = [i for i, _ in selected_layers(names)]
        copies = args.decode_copies
        wbytes = copies * sum(L.N * L.K for L in layers)
        d5 = [[F.fp8_quantize_weight_ex(I.decode_weight(i, c).to(dev), "e5m2") for i in li] for c in range(copies)]
        d4 = [[F.fp8_quantize_weight(I.decode_weight(i, c).to(dev)) for i in li] for c in range(copies)]
        yd = [torch.empty((16, L.N), dtype=torch.bfloat16, device=dev) for L in layers]
        for Md in (1, 15):
            ad = [I.decode_activations(Md, i).to(dev) for i in li]
            sd = [F.fp8_quantize_act(a)[1] for a in ad]

            def d_e5m2(ad=ad, Md=Md):
                for c in range(copies):
                    for i in range(len(layers)):
                        F.fp8_linear_ex(ad[i], d5[c][i][0], d5[c][i][1], out=yd[i][:Md], fmt_a="e5m2", fmt_w="e5m2")

            def d_static(ad=ad, sd=sd, Md=Md):
                for c in range(copies):
                    for i in range(len(layers)):
                        F.fp8_linear_static(ad[i], sd[i], d4[c][i][0], d4[c][i][1], out=yd[i][:Md])

            def d_weight_only(ad=ad, Md=Md):
                for c in range(copies):
                    for i in range(len(layers)):
                        F.fp8_linear_weight_only(ad[i], d4[c][i][0], d4[c][i][1], out=yd[i][:Md])

            for name, fn in (("e5m2_dynamic", d_e5m2), ("e4m3_static", d_static), ("weight_only_e4m3", d_weight_only)):
                t = time_loop(torch, graph_of(torch, fn).replay, max(5, args.steps), 3)
                out[name][f"decode_M{Md}_weight_gbs"] = round(wbytes / (t * 1e-3) / 1e9, 1)
        del d5, d4
    torch.cuda.synchronize()
    return out


def roofline_time_s(M, K, N, per_channel, fp8_tflops, hbm_gbs):
    """Roofline time of one linear: the slower of its FP8 flops at the compute peak and its
    algorithmic bytes (A read, qW, scales, Y write) at the HBM rate."""
    flop = 2.0 * M * N * K
    byts = 2.0 * M * K + float(N) * K + (4.0 * N if per_channel else 4.0) + 2.0 * M * N
    return max(flop / (fp8_tflops * 1e12), byts / (hbm_gbs * 1e9))


def measure_sweep(torch, F, I, dev, args, fp8_tflops, hbm_gbs):
    """TinyLlama-1.1B decoder stack: 22 layers x (qkv, o_proj, gate_up, down), 22 distinct
    weight sets (969 MB of FP8 per mode, far above L2), both weight-scale modes, every M of the
    workload; activations quantized per layer. One step = all 88 linears, CUDA graph replay."""
    layers, depth = I.TINYLLAMA_LAYERS, I.TINYLLAMA_DEPTH
    Ms = [m for m in I.TINYLLAMA_MS if m <= args.sweep_max_m]
    W = {}
    for mode in (False, True):
        W[mode] = []
        for d in range(depth):
            row = []
            for j in range(len(layers)):
                w = I.tinyllama_weight_device(d, j, dev)
                row.append(F.fp8_quantize_weight(w, per_channel=mode))
                del w
            W[mode].append(row)
    copies = 2  # consecutive layers read different activation buffers
    Mmax = max(Ms)
    A = [[I.tinyllama_activations_device(Mmax, c, j, dev) for j in range(len(layers))] for c in range(copies)]
    Y = [torch.empty((Mmax, L.N), dtype=torch.bfloat16, device=dev) for L in layers]
    ws = torch.empty(max(1, max(F.fp8_workspace_bytes(Mmax, L.K, L.N) for L in layers)), dtype=torch.uint8,
                     device=dev)
    torch.cuda.synchronize()
    wbytes = depth * sum(L.N * L.K for L in layers)
    out = {}
    for mode in (False, True):
        fn = F.fp8_linear_channelwise if mode else F.fp8_linear
        rows = []
        for M in Ms:
            def step(M=M):
                for d in range(depth):
                    for j in range(len(layers)):
                        fn(A[d % copies][j][:M], W[mode][d][j][0], W[mode][d][j][1], out=Y[j][:M], ws=ws)

            t = time_loop(torch, graph_of(torch, step).replay, max(3, min(args.steps, 10)), 2)
            fl = depth * sum(2.0 * M * L.N * L.K for L in layers)
            t_roof = depth * sum(roofline_time_s(M, L.K, L.N, mode, fp8_tflops, hbm_gbs) for L in layers)
            rows.append({"M": M, "ms_per_stack": round(t, 4), "tflops": round(fl / (t * 1e-3) / 1e12, 1),
                         "weight_gbs": round(wbytes / (t * 1e-3) / 1e9, 1),
                         "roofline_frac": round(t_roof / (t * 1e-3), 4),
                         "path": "gemv" if F.fp8_uses_gemv(M, layers[0].K, layers[0].N) else "gemm"})
        out["channelwise" if mode else "per_tensor"] = rows
    del W, A, Y, ws
    torch.cuda.synchronize()
    return {"workload": "TinyLlama-1.1B linears (qkv 2048->2560, o_proj 2048->2048, gate_up 2048->11264, "
                        "down 5632->2048) x 22 distinct layers per step, activations ~N(0,1) quantized per layer "
                        "(dynamic e4m3), weights ~N(0,0.02) drawn on the device (timing only)",
            "timing": "CUDA graph replay of the 88 linears; roofline_frac = sum of per-linear roofline times "
                      "(max of 2MNK / FP8 peak and algorithmic bytes / HBM) over the measured time",
            "weight_mb_per_mode": round(wbytes / 1e6, 1), "by_mode": out}


def measure_crossover(torch, F, I, dev, args):
    """Decode GEMV against the GEMM path for the same calls at M around the crossover, on the
    Mistral-7B decode linears (three weight copies rotated past L2) and the TinyLlama linears
    (22 layers): the GEMV (up to 32 tokens), the GEMM with the library's K split, and the GEMM
    with K unsplit (FP8W8A8_GEMM_SPLITK=1)."""
    res = {}
    prev = F.fp8_set_gemv_max_m(-1)
    fams = {"mistral7b": (I.LLAMA8B_LAYERS, [[F.fp8_quantize_weight(I.decode_weight(i, c).to(dev))
                                               for i in range(4)] for c in range(3)]),
            "tinyllama": (I.TINYLLAMA_LAYERS, [[F.fp8_quantize_weight(I.tinyllama_weight_device(d, j, dev))
                                                for j in range(4)] for d in range(I.TINYLLAMA_DEPTH)])}
    Ms = (8, 16, 17, 24, 32, 64, 128, 256, 512)
    try:
        for fam, (layers, Wq) in fams.items():
            A = [I.normal_device(max(Ms), L.K, (1005, j), 1.0, dev) for j, L in enumerate(layers)]
            Y = [torch.empty((max(Ms), L.N), dtype=torch.bfloat16, device=dev) for L in layers]
            ws = torch.empty(max(F.fp8_workspace_bytes(m, L.K, L.N) for m in Ms for L in layers) + 256,
                             dtype=torch.uint8, device=dev)
            rows = []
            for M in Ms:
                row = {"M": M}
                for path, thr, split_env in (("gemv", 32, None), ("gemm", 0, None), ("gemm_unsplit", 0, "1")):
                    if path == "gemv" and M > 32:
                        continue
                    F.fp8_set_gemv_max_m(thr)
                    if split_env is None:
                        os.environ.pop("FP8W8A8_GEMM_SPLITK", None)
                    else:
                        os.environ["FP8W8A8_GEMM_SPLITK"] = split_env

                    def step(M=M):
                        for Wc in Wq:
                            for j in range(len(layers)):
                                F.fp8_linear(A[j][:M], Wc[j][0], Wc[j][1], out=Y[j][:M], ws=ws)

                    t = time_loop(torch, graph_of(torch, step).replay, 10, 3)
                    row[path + "_us_per_linear"] = round(t * 1e3 / (len(Wq) * len(layers)), 2)
                os.environ.pop("FP8W8A8_GEMM_SPLITK", None)
                rows.append(row)
            both = [r for r in rows if "gemv_us_per_linear" in r]
            wins = [r["M"] for r in both if r["gemv_us_per_linear"] <= r["gemm_us_per_linear"]]
            res[fam] = {"rows": rows, "gemv_faster_at": wins}
            del A, Y, ws
    finally:
        F.fp8_set_gemv_max_m(prev)
        os.environ.pop("FP8W8A8_GEMM_SPLITK", None)
    del fams
    torch.cuda.synchronize()
    return res


def measure_unaligned(torch, F, I, dev, hbm_gbs):
    """The four shapes whose dimensions are not multiples of 16 (per-tensor, outlier channels),
    decode GEMV path; enough weight copies per shape to exceed twice the L2."""
    out = []
    for c in I.unaligned_cases():
        M, K, N = c.M, c.K, c.N
        copies = max(3, -(-256_000_000 // (N * K)))
        w = c.w.to(dev)
        Wq = [F.fp8_quantize_weight(w) for _ in range(copies)]
        a = c.a.to(dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def step():
            for qw, s_w in Wq:
                F.fp8_linear(a, qw, s_w, out=y)

        t = time_loop(torch, graph_of(torch, step).replay, 10, 3)
        per = t * 1e-3 / copies
        gbs = N * K / per / 1e9
        out.append({"M": M, "K": K, "N": N, "us_per_call": round(per * 1e6, 2), "weight_gbs": round(gbs, 1),
                    "hbm_frac": round(gbs / hbm_gbs, 4), "weight_copies": copies,
                    "path": "gemv" if F.fp8_uses_gemv(M, K, N) else "gemm"})
        del Wq
    torch.cuda.synchronize()
    return out


def measure_tiny(torch, F, I, dev):
    """Latency of the 16 x 256 x 256 per-tensor linear (one call, decode GEMV)."""
    c = I.tiny_case()
    a, (qw, s_w) = c.a.to(dev), F.fp8_quantize_weight(c.w.to(dev))
    y = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    reps = 100

    def step():
        for _ in range(reps):
            F.fp8_linear(a, qw, s_w, out=y)

    t_graph = time_loop(torch, graph_of(torch, step).replay, 5, 2) / reps
    t_eager = time_loop(torch, lambda: F.fp8_linear(a, qw, s_w, out=y), 200, 20)
    return {"M": c.M, "K": c.K, "N": c.N, "us_per_call_graph": round(t_graph * 1e3, 2),
            "us_per_call_eager": round(t_eager * 1e3, 2)}


def run_ours(args):
    import torch
    import fp8_w8a8_quantized_dynamic_gb300 as F
    from fp8_w8a8_quantized_dynamic_gb300 import _build
    from fp8_w8a8_quantized_dynamic_gb300 import inputs as I

    _build.build()
    F.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * NOMINAL_FP8_OVER_BF16
    hbm = peaks["hbm_gbs"]
    M = args.m
    names = args.layers.split(",") if args.layers else None
    layers = [L for _, L in selected_layers(names)]

    clocks = ClockSampler(dev.index)
    clocks.start()
    host, value, ms, launches, roofline, quant_ms, gemm_ms = [], None, None, 0, None, [], []
    total_flops = flops(M, layers)
    if not args.no_prefill:
        # ---- inputs: bf16 A per layer, FP8 weights quantized once on the device (load time)
        host = prefill_inputs(M, names)
        A = [a.to(dev) for _, a, _ in host]
        Wq = []
        for _, _, w in host:
            qw, s_w = F.fp8_quantize_weight(w.to(dev), per_channel=True)
            Wq.append((qw, s_w))
        Y = [torch.empty((M, L.N), dtype=torch.bfloat16, device=dev) for L in layers]
        ws = torch.empty(max(F.fp8_workspace_bytes(M, L.K, L.N) for L in layers), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

        def step():
            for i in range(len(layers)):
                F.fp8_linear_channelwise(A[i], Wq[i][0], Wq[i][1], out=Y[i], ws=ws)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            step()
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / args.steps
        value = total_flops / (ms * 1e-3) / 1e12
        launches = args.steps * len(layers) * 3  # amax, cast, gemm per layer

        # ---- GEMM kernel alone (fp8_scaled_mm on the quantized activations), per layer
        Q = [F.fp8_quantize_act(a) for a in A]
        torch.cuda.synchronize()
        plans = {}
        for i, L in enumerate(layers):
            qa, s_a = Q[i]
            f = lambda i=i, qa=qa, s_a=s_a, L=L: F.fp8_scaled_mm(qa, L.K, s_a, Wq[i][0], Wq[i][1], True, out=Y[i])
            gemm_ms.append(time_loop(torch, f, max(10, args.steps), 5))
            plans[L.name] = F.fp8_gemm_config(qa, Wq[i][0])

        def gemm_step():  # the step's four GEMMs back to back, as the prefill step runs them
            for i, L in enumerate(layers):
                F.fp8_scaled_mm(Q[i][0], L.K, Q[i][1], Wq[i][0], Wq[i][1], True, out=Y[i])

        gemm_step_ms = time_loop(torch, gemm_step, max(10, args.steps), 5)
        for i, L in enumerate(layers):
            f = lambda i=i: F.fp8_quantize_act(A[i], ws=ws)
            quant_ms.append(time_loop(torch, f, max(3, args.steps // 2), 2))
        del Q
        gemm_flops = [2.0 * M * L.N * L.K for L in layers]
        gemm_tflops = sum(gemm_flops) / (gemm_step_ms * 1e-3) / 1e12
        sustained = peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"]) * NOMINAL_FP8_OVER_BF16
        traffic, traffic_per = gemm_traffic(layers)
        two = all(p["two_sm"] for p in plans.values())
        roofline = {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                    "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                    "frac_of_sustained": round(gemm_tflops / sustained, 4),
                    "achieved_note": "the four layers' GEMMs (fp8_scaled_mm) back to back, CUDA events over "
                                     f"{max(10, args.steps)} such steps after 5 warm-up steps; peak: burst",
                    "traffic": None if traffic is None else int(traffic),
                    "traffic_note": "mean dram__bytes_read.sum + dram__bytes_write.sum per GEMM launch "
                                    "(ncu, profiles/gemm_tcgen05_dram_llama8b_m16384.json); null when that "
                                    "capture predates the current GEMM source",
                    "traffic_per_launch": traffic_per,
                    "kernel": "gemm_kernel (tcgen05 kind::f8f6f4, " +
                              ("CTA pairs on the two-SM MMA, cta_group::2)" if two else "one CTA per tile)"),
                    "launch_plans": plans,
                    "peak_source": f"{peak_src} bf16 burst x {NOMINAL_FP8_OVER_BF16} nominal fp8/bf16 ratio",
                    "per_layer_ms": {L.name: round(t, 4) for L, t in zip(layers, gemm_ms)},
                    "per_layer_frac": {L.name: round(f / (t * 1e-3) / 1e12 / fp8_peak, 4)
                                       for L, f, t in zip(layers, gemm_flops, gemm_ms)}}

    # ---- wider rows on the same workloads: e5m2 operands, static activation scale
    variants = None
    if not args.no_variants and not args.no_prefill:
        variants = measure_variants(torch, F, I, args, dev, layers, names, host, A, Y, ws, M)

    # ---- decode GEMV: Mistral-7B layers, per-tensor scales, weight copies rotated past L2
    decode = None
    if not args.no_decode:
        copies = args.decode_copies
        li = [i for i, _ in selected_layers(names)]
        dq = [[F.fp8_quantize_weight(I.decode_weight(i, c).to(dev)) for i in li] for c in range(copies)]
        wbytes_step = copies * sum(L.N * L.K for L in layers)
        yd = [torch.empty((16, L.N), dtype=torch.bfloat16, device=dev) for L in layers]
        per_m, per_layer = {}, {}
        decode_ms = args.decode_ms or list(I.DECODE_MS)
        for Md in decode_ms:
            ad = [I.decode_activations(Md, i).to(dev) for i in li]
            ydm = [y[:Md] for y in yd]

            def dstep(ad=ad, Md=Md):
                for c in range(copies):
                    for i in range(len(layers)):
                        F.fp8_linear(ad[i], dq[c][i][0], dq[c][i][1], out=ydm[i])

            t_eager = time_loop(torch, dstep, max(5, args.steps), 3)
            t = time_loop(torch, graph_of(torch, dstep).replay, max(5, args.steps), 3)
            per_m[str(Md)] = {"weight_gbs": round(wbytes_step / (t * 1e-3) / 1e9, 1),
                              "us_per_layer": round(t * 1e3 / (copies * len(layers)), 2),
                              "eager_us_per_layer": round(t_eager * 1e3 / (copies * len(layers)), 2)}
            if Md in (1, 15):
                rows = {}
                for i, L in enumerate(layers):
                    def lstep(i=i, ad=ad):
                        for c in range(copies):
                            F.fp8_linear(ad[i], dq[c][i][0], dq[c][i][1], out=ydm[i])

                    tl = time_loop(torch, graph_of(torch, lstep).replay, max(10, args.steps), 3) / copies
                    gbs = L.N * L.K / (tl * 1e-3) / 1e9
                    rows[L.name] = {"us": round(tl * 1e3, 2), "weight_gbs": round(gbs, 1),
                                    "hbm_frac": round(gbs / hbm, 4),
                                    "ideal_us": round(L.N * L.K / (hbm * 1e9) * 1e6, 2)}
                per_layer[f"M{Md}"] = rows
        gbs = [v["weight_gbs"] for v in per_m.values()]
        decode = {"metric": "decode weight GB/s (one fused quantize + split-K GEMV kernel per layer, "
                            "CUDA graph replay of the 4 layers x weight copies)", "unit": "GB/s",
                  "value": round(statistics.median(gbs), 1), "per_M": per_m, "per_layer": per_layer,
                  "workload": "Mistral-7B linears qkv/o_proj/gate_up/down, M in "
                              + ",".join(str(m) for m in decode_ms) + ", per-tensor scales",
                  "roofline": {"bound": "hbm", "peak": hbm, "unit": "GB/s",
                               "frac_median": round(statistics.median(gbs) / hbm, 4),
                               "frac_median_of_nominal": round(statistics.median(gbs) / NOMINAL_HBM_GBS, 4),
                               "peak_source": f"{peak_src} copy bandwidth; nominal {NOMINAL_HBM_GBS:.0f} GB/s"},
                  "l2": f"{copies} weight copies of {sum(L.N * L.K for L in layers) / 1e6:.0f} MB rotated",
                  "gpu_launches_per_replay": copies * len(layers)}
        del dq

    sweep = crossover = unaligned = tiny = None
    if not args.no_sweep:
        sweep = measure_sweep(torch, F, I, dev, args, fp8_peak, hbm)
        crossover = measure_crossover(torch, F, I, dev, args)
        unaligned = measure_unaligned(torch, F, I, dev, hbm)
        tiny = measure_tiny(torch, F, I, dev)

    clk = clocks.stop()

    # ---- e2e: host buffers through the C-ABI call, copies inside the timed region
    e2e = None
    if not args.no_e2e and not args.no_prefill:
        A_h = [a.pin_memory() for _, a, _ in host]
        Y_h = [torch.empty((M, L.N), dtype=torch.bfloat16).pin_memory() for L in layers]
        A_d = A
        # A user's pipeline: host->device copies on one stream, the linears on the compute
        # stream, device->host copies on a third, ordered per layer by events, so the two
        # copy directions overlap each other and the compute of neighbouring layers.
        compute = torch.cuda.current_stream(dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        n = len(layers)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for e in ev_done + ev_out:
            e.record(compute)

        def estep(with_linear=True):
            for i in range(n):
                s_in.wait_event(ev_done[i])          # A_d[i] is free once the last step's linear read it
                with torch.cuda.stream(s_in):
                    A_d[i].copy_(A_h[i], non_blocking=True)
                ev_in[i].record(s_in)
            for i in range(n):
                compute.wait_event(ev_in[i])
                compute.wait_event(ev_out[i])        # Y[i] is free once the last step's copy read it
                if with_linear:
                    F.fp8_linear_channelwise(A_d[i], Wq[i][0], Wq[i][1], out=Y[i], ws=ws)
                ev_done[i].record(compute)
                s_out.wait_event(ev_done[i])
                with torch.cuda.stream(s_out):
                    Y_h[i].copy_(Y[i], non_blocking=True)
                ev_out[i].record(s_out)
            for i in range(n):
                compute.wait_event(ev_out[i])        # the step ends when its results are on the host

        def copies_only():
            # the link alone: every input copy on one stream, every output copy on the other
            with torch.cuda.stream(s_in):
                for i in range(n):
                    A_d[i].copy_(A_h[i], non_blocking=True)
            with torch.cuda.stream(s_out):
                for i in range(n):
                    Y_h[i].copy_(Y[i], non_blocking=True)
            compute.wait_stream(s_in)
            compute.wait_stream(s_out)

        # median of three repetitions each: the host link is shared with the rest of the machine
        reps = max(3, args.steps // 4)
        te = statistics.median(time_loop(torch, estep, reps, 2) for _ in range(3))
        t_chain = statistics.median(time_loop(torch, lambda: estep(False), reps, 2) for _ in range(3))
        t_link = statistics.median(time_loop(torch, copies_only, reps, 2) for _ in range(3))
        h2d = int(sum(a.numel() * 2 for a in A_h))
        d2h = int(sum(y.numel() * 2 for y in Y_h))
        e2e = {"value": round(total_flops / (te * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(te, 3),
               "copy_bound_ms": round(t_link, 3), "link_gbs": round((h2d + d2h) / (t_link * 1e-3) / 1e9, 1),
               "frac_of_copy_bound": round(t_link / te, 4),
               "copies_in_step_order_ms": round(t_chain, 3),
               "note": "copy_bound_ms: the same host copies alone, inputs on one stream and outputs on "
                       "another; copies_in_step_order_ms: the step's copy and event chain without the linears"}

    cpu = None
    if not args.no_cpu_baseline and not args.no_prefill:
        cpu = oracle_sample(host, M, args.cpu_rows, args.cpu_cols)

    return {
        "metric": METRIC, "value": None if value is None else round(value, 1), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None if ms is None else round(ms, 4),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> fp32 accumulate, bf16 out", "data": "synthetic",
        "config": {"workload": "prefill: Llama-3-8B linears qkv/o_proj/gate_up/down at M=16384, channelwise "
                               "weight scales, dynamic per-tensor activation scale",
                   "M": M, "layers": [[L.name, L.K, L.N] for L in layers], "global_batch": M,
                   "parallelism": "single GPU",
                   "l2": "inputs larger than L2: each step streams 0.87 GB of bf16 activations and writes "
                         "1.4 GB of outputs across four layers"},
        "roofline": roofline, "kernels_ms": {"quantize_act(amax+cast)": [round(t, 4) for t in quant_ms],
                                             "gemm": [round(t, 4) for t in gemm_ms]},
        "decode": decode, "sweep": sweep, "crossover": crossover, "unaligned": unaligned, "tiny": tiny,
        "variants": variants, "e2e": e2e, "gpu_launches": launches,
        "gpu_launches_note": "timed prefill region: 3 kernels per layer per step (amax, cast, GEMM)",
        "clocks": clk, "cpu_baseline": cpu,
    }


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(host, M: int, rows: int, cols: int, repeats: int = 1):
    """Oracle on `rows` activation rows x `cols` output channels of every layer; the amax
    runs over the full A as the method defines. Returns TFLOP/s of the sampled product."""
    from oracle import fp8_oracle as O
    g = np.random.default_rng(0)
    work = []
    for L, a, w in host:
        r = np.sort(g.choice(a.shape[0], rows, replace=False))
        c = np.sort(g.choice(w.shape[0], cols, replace=False))
        work.append((L, a.float().numpy(), w[c].float().numpy(), r))
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(repeats):
        for L, a32, w32, r in work:
            s_a = np.float32(O.scale_from_amax(O.amax(a32)))
            qa = O.quantize_with_scale(a32[r], s_a)
            qw, s_w = O.quantize_per_row(w32)
            O.scaled_mm(qa, s_a, qw, s_w)
            fl += 2.0 * rows * cols * L.K
    dt = time.perf_counter() - t0
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"{rows} activation rows x {cols} output channels per layer of the M={M} prefill step "
                      f"(full-tensor amax included), numpy float64"}


def run_reference(args):
    from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
    M = args.m
    host = prefill_inputs(M)
    layers = I.LLAMA8B_LAYERS
    for _ in range(args.warmup):
        oracle_sample(host, M, args.cpu_rows, args.cpu_cols)
    res = oracle_sample(host, M, args.cpu_rows, args.cpu_cols, repeats=args.steps)
    step_s = res["seconds"] / args.steps
    value = res["value"]
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (exact product)",
        "data": "synthetic",
        "config": {"workload": f"prefill: Llama-3-8B linears qkv/o_proj/gate_up/down at M={M}, channelwise "
                               "weight scales, dynamic per-tensor activation scale (bounded CPU sample)",
                   "M": M, "layers": [[L.name, L.K, L.N] for L in layers]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": res["cores"], "kind": "oracle",
                         "sample": res["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--m", type=int, default=16384, help="tokens per prefill layer")
    ap.add_argument("--decode-copies", type=int, default=3)
    ap.add_argument("--decode-ms", type=lambda s: [int(x) for x in s.split(",")], default=None,
                    help="token counts of the decode leg, comma-separated (default 1,2,4,8,15)")
    ap.add_argument("--cpu-rows", type=int, default=16)
    ap.add_argument("--cpu-cols", type=int, default=512)
    ap.add_argument("--sweep-max-m", type=int, default=16384, help="largest M of the TinyLlama sweep")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="decode leg only (profiling)")
    ap.add_argument("--layers", default="", help="comma list of qkv,o_proj,gate_up,down (default all)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-variants", action="store_true", help="skip the e5m2 / static-scale legs")
    ap.add_argument("--no-sweep", action="store_true", help="skip the sweep, crossover, unaligned and tiny legs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1 or args.gpus > 1:
        # the path runs on one GPU; no rank touches a device here
        if rank == 0:
            print(json.dumps({"metric": METRIC, "n_gpus": max(world, args.gpus),
                              "unavailable": "single-GPU path only: the linear is not sharded across GPUs and its "
                                             "pair GEMM is built for one device; run with --gpus 1"}))
        return
    print(json.dumps(run_ours(args)))


if __name__ == "__main__":
    main()
