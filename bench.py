#!/usr/bin/env python3
"""Benchmark of the NVFP4 MoE layer forward (libmoe_nvfp4.so, C ABI).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload prefill|mid|tiny|dsv3|w4a16] [--tokens T]
                    [--precision nvfp4|mxfp8] [--four-over-six] [--routing logits|given|gate]
                    [--fused] [--gemm auto|standard|swapped|pairs] [--sweep dsv3|none]

A step is one full layer forward (router, permutation, activation
quantization, FC1 + activation + requantization, FC2, finalize) over one
batch of T synthetic tokens.  Default workload: the prefill-scale
configuration, the largest that runs on one GPU (T=16384, H=7168, I=2048,
E=256, top-8, SwiGLU, W4A4 per-token scales, Zipf-skewed expert
popularity, deterministic finalize).  With --sweep dsv3 (the default at N=1) the
line also carries the DeepSeek-V3-like expert shape (H=7168, I=2048, E=256,
top-8, per-tensor, deterministic finalize) at T in {1, 8, 64, 256, 1024,
4096, 8192}: device-timed tokens/s, TFLOP/s and % of the dense FP4 peak
per token count (cold-L2 median with p10 / p90, the warm-L2 median, and up
to 256 tokens a CUDA-graph replay).

Prints one JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM; L2 is defeated by rotating several copies of the prepared
weights (together larger than the 129 MB L2) across steps.  `e2e` is the same
metric through the C ABI with each step's x and logits copied from pinned
host memory and y copied back inside the timed region.  `roofline` is the
dominant kernel's algorithmic bytes (or FLOPs) per launch over its mean
CUDA-event duration.  `per_forward` times single forwards of the workload
(median, p10, p90) with L2 evicted before each and with L2 warm, and up to
256 tokens as one CUDA-graph replay.  `cpu_baseline` carries the oracle on
all host threads and on one.  Multi-GPU: independent replicas (one per
rank, no collective on the data path), weak scaling.

--impl reference times the CPU oracle (oracle/, plain C++ FP64) on the host
cores on a bounded token sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and NVFP4 TFLOPS (% of GB300 dense FP4 peak) vs tokens"
L2_BYTES = 129 * 1024 * 1024
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense-rate ratios used to scale the measured bf16 peak
FP8_OVER_BF16 = 4.5 / 2.25


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="prefill", choices=["tiny", "mid", "dsv3", "w4a16", "prefill"])
    p.add_argument("--sweep", default="dsv3", choices=["dsv3", "none"],
                   help="dsv3: also time the DSV3-like expert shape over its token counts (N=1 only)")
    p.add_argument("--tokens", type=int, default=None, help="token count (sweeps of dsv3 / w4a16)")
    p.add_argument("--experts", type=int, default=None,
                   help="expert count in place of the workload's (same shapes and distributions otherwise; "
                        "fewer experts = more rows per expert, a compute-bound GEMM at a small footprint)")
    p.add_argument("--stage-steps", type=int, default=200)
    p.add_argument("--precision", default="nvfp4", choices=["nvfp4", "mxfp8"],
                   help="mxfp8: the W4A4 workloads' shapes and routing in MXFP8 W8A8")
    p.add_argument("--four-over-six", action="store_true",
                   help="4-over-6 activation quantization (per-token W4A4 workloads)")
    p.add_argument("--routing", default="logits", choices=["logits", "given", "gate"],
                   help="given: caller-supplied top-K ids and weights (moe_nvfp4_forward_routed); "
                        "gate: logits computed by the layer from the gate projection (moe_nvfp4_forward_gate)")
    p.add_argument("--fused", action="store_true",
                   help="the whole forward as one persistent kernel (MOE_FUSED_LAYER; W4A4, E <= 256)")
    p.add_argument("--gemm", default="auto", choices=["auto", "standard", "swapped", "pairs"],
                   help="W4A4 / W4A16 GEMM variant (default: by routes per expert): single-CTA standard or "
                        "swapped orientation, or CTA pairs")
    p.add_argument("--finalize", default="config", choices=["config", "fused", "deterministic"],
                   help="finalize mode: the workload's own (default), the FC2-epilogue scatter or the fixed-order kernel")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def workload_config(name, tokens, precision="nvfp4", four_over_six=False, fused=False, gemm="auto",
                    finalize="config", experts=None):
    from nvfp4_mixture_experts_router_gb300 import synth
    idx = {"tiny": 0, "mid": 1, "dsv3": 2, "w4a16": 3, "prefill": 4}[name]
    c = synth.config(idx, tokens)
    if experts is not None:
        if not (c.K <= experts <= 1024):
            raise SystemExit(f"--experts must lie in [{c.K}, 1024]")
        c = c.with_(E=experts, name=c.name.replace(f"_E{c.E}_", f"_E{experts}_"))
    if precision == "mxfp8":
        if c.mode == synth.MODE_W4A16:
            raise SystemExit("--precision mxfp8 applies to the W4A4 workloads")
        c = c.with_(mode=synth.MODE_MXFP8)
    if four_over_six:
        if c.mode != synth.MODE_PER_TOKEN:
            raise SystemExit("--four-over-six needs a per-token W4A4 workload (mid, prefill)")
        c = c.with_(four_over_six=True)
    if fused:
        if c.mode not in (synth.MODE_PER_TENSOR, synth.MODE_PER_TOKEN) or c.E > 256:
            raise SystemExit("--fused needs a W4A4 workload with E <= 256")
        c = c.with_(fused=True)
    if gemm == "pairs":
        c = c.with_(gemm_pairs="always", gemm_swap="never")
    elif gemm == "standard":
        c = c.with_(gemm_pairs="never", gemm_swap="never")
    elif gemm == "swapped":
        c = c.with_(gemm_pairs="never", gemm_swap="always")
    if finalize != "config":
        c = c.with_(deterministic=finalize == "deterministic")
    return c


def describe(c):
    from nvfp4_mixture_experts_router_gb300 import synth
    act = "SwiGLU" if c.act == synth.ACT_SWIGLU else "ReLU2"
    mode = {0: "W4A4 per-tensor", 1: "W4A4 per-token", 2: "W4A16", 3: "W8A8 MXFP8"}[c.mode]
    if c.four_over_six:
        mode += " 4-over-6"
    if c.fused:
        mode += ", one persistent kernel"
    place = "router weight on FC2 input" if c.router_on_input else "router weight at output"
    fin = "deterministic finalize" if c.deterministic else "fused finalize"
    return f"{c.name}: T={c.T}, H={c.H}, I={c.I}, E={c.E}, top-{c.K}, {act}, {mode}, {place}, {fin}"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def flops_per_step(c):
    R = c.T * c.K
    return 2.0 * R * (c.N1 * c.H + c.I * c.H)


def stage_bytes(c, active, h_fp32=False):
    """Algorithmic bytes per launch of each stage (minimum HBM traffic).
    h_fp32: per-token mode on its fallback path (FC1 stores the FP32 FC2
    input and a separate kernel quantizes it)."""
    from nvfp4_mixture_experts_router_gb300 import synth
    T, H, I, E, K, N1 = c.T, c.H, c.I, c.E, c.K, c.N1
    R = T * K
    mx = c.mode == synth.MODE_MXFP8
    nv = 1.03125 if mx else 0.5625               # MXFP8: 1 B + 1/32 B; NVFP4: 0.5 B code + 1/16 B scale
    w4a16 = c.mode == synth.MODE_W4A16
    per_token = c.mode == synth.MODE_PER_TOKEN
    a_elem = 2.0 if w4a16 else nv
    h_out = 2.0 if w4a16 else (4.0 if (per_token and h_fp32) else nv)
    fused = not c.deterministic
    return {
        "router_gemm": T * H * 2 + E * H * 2 + T * E * 4,
        "router": T * E * 4 + T * K * 8 + (E * 4 if c.bias != "none" else 0),
        "permute": T * K * 4 * 4,
        "quantize_x": T * H * 2 + R * H * a_elem + (T * H * 4 if fused else 0),
        "fc1": active * N1 * H * nv + R * H * a_elem + R * I * h_out,
        "quantize_h": (R * I * 4 + R * I * nv) if (per_token and h_fp32) else 0,
        "fc2": active * H * I * nv + R * I * (2.0 if w4a16 else nv) + (T * H * 4 if fused else R * H * 2),
        "finalize": (T * H * 4 + T * H * 2) if fused else (R * H * 2 + T * H * 2),
    }


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    e = d.get(f"{workload}:{kernel}")
    if not e:
        return None
    if e.get("source_sha") != source_sha(e.get("source")):
        return None
    return e.get("dram_bytes_per_launch")


def traffic_key(args):
    """Workload key of profiles/traffic.json (precision and quantization
    variants have their own entries)."""
    key = args.workload
    if args.precision != "nvfp4":
        key += "-" + args.precision
    if args.four_over_six:
        key += "-4over6"
    if args.fused:
        key += "-fused"
    if args.finalize != "config":
        key += "-" + args.finalize
    if args.experts is not None:
        key += f"-E{args.experts}"
    if args.tokens is not None:
        key += f"-T{args.tokens}"
    return key


def source_sha(unit=None):
    """Hash of the kernel sources: one translation unit of csrc/ and every
    header it includes (transitively), or all of csrc/ when unit is None."""
    csrc = os.path.join(ROOT, "nvfp4_mixture_experts_router_gb300", "csrc")
    if unit is None:
        files = [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith((".cu", ".cuh", ".h"))]
    else:
        files, todo = [], [os.path.join(csrc, unit)]
        while todo:
            f = os.path.normpath(todo.pop())
            if f in files or not os.path.exists(f):
                continue
            files.append(f)
            for line in open(f, encoding="utf-8", errors="replace"):
                line = line.strip()
                if line.startswith("#include \""):
                    todo.append(os.path.join(os.path.dirname(f), line.split('"')[1]))
        files.sort()
    h = hashlib.sha256()
    for f in files:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        def reader():
            for line in self.proc.stdout:
                self.samples.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        time.sleep(1.0)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.1 <= t <= t1 + 0.1]
        if not rows:
            # nearest samples around a very short region
            rows = [s for t, s in sorted(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[:2]]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        mhz.sort()
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(mhz)}


def init_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """The largest value of x over all ranks (x itself on a single rank);
    the timed region's duration is the slowest replica's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens, steps, ms):
    """Whole-job throughput: the tokens every replica processed in `steps`
    steps over the slowest replica's time `ms` (milliseconds)."""
    return world * tokens * steps / (ms / 1000.0)


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------

class OracleRunner:
    """The oracle on host cores, weights prepared once (untimed)."""

    def __init__(self, c, device):
        import numpy as np
        import torch
        import oracle
        from nvfp4_mixture_experts_router_gb300 import synth
        self.np, self.oracle, self.c = np, oracle, c
        self.layer = oracle.Layer(c.H, c.I, c.E, c.K, act=c.act, mode=c.mode, router_on_input=c.router_on_input,
                                  renorm=c.renorm, four_over_six=c.four_over_six)
        x = synth.gen_x(c, device)
        self.x_np = x.cpu().view(torch.int16).numpy().view(np.uint16)
        self.logits = synth.gen_logits(c, device, x).cpu().numpy()
        b = synth.gen_bias(c, device)
        self.bias = None if b is None else b.cpu().numpy()
        self.dev = device
        self.prepared = {}
        self.G1 = self.G2 = None
        if c.mode == synth.MODE_PER_TENSOR:
            self.G1 = oracle.tensor_global_scale(oracle.bf16_bits_to_f64(self.x_np).astype(np.float32))
            self.G2 = np.float32(self.G1)          # any positive scale: the arithmetic done is the same

    def weights(self, e):
        import torch
        from nvfp4_mixture_experts_router_gb300 import synth
        w1 = synth.gen_w1_expert(self.c, e, self.dev).cpu().view(torch.int16).numpy().view(self.np.uint16)
        w2 = synth.gen_w2_expert(self.c, e, self.dev).cpu().view(torch.int16).numpy().view(self.np.uint16)
        return w1, w2

    def prepare_for(self, tokens):
        ids, _ = self.oracle.router(self.logits, self.bias, self.c.K, self.c.renorm)
        need = sorted(set(int(e) for t in tokens for e in ids[t]))
        for e in need:
            if e not in self.prepared:
                self.prepared[e] = self.oracle.prepare_expert(self.layer, self.weights, e)

    def run(self, tokens):
        return self.oracle.forward(self.layer, self.x_np, self.logits, self.bias, self.weights, G1=self.G1,
                                   G2=self.G2, tokens=tokens, prepared=self.prepared)


def cpu_cores():
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return int(os.environ.get("OMP_NUM_THREADS", n))


def cpu_baseline(c, device, budget_s=15.0):
    from nvfp4_mixture_experts_router_gb300 import synth
    r = OracleRunner(c, device)
    probe = synth.sample_tokens(c, min(4, c.T))
    r.prepare_for(probe)
    t0 = time.perf_counter()
    r.run(probe)
    per_tok = (time.perf_counter() - t0) / len(probe)
    n = max(1, min(c.T, int(budget_s / max(per_tok, 1e-6))))
    toks = synth.sample_tokens(c, n)
    r.prepare_for(toks)
    t0 = time.perf_counter()
    r.run(toks)
    dt = time.perf_counter() - t0
    out = {"value": round(len(toks) / dt, 3), "unit": "tokens/s", "cores": r.oracle.max_threads(), "kind": "oracle",
           "sample": f"{len(toks)} of the workload's {c.T} tokens (seeded subset), all their routes; "
                     f"expert weights prepared by the oracle beforehand (untimed)"}
    # the same oracle on one host thread, over a third of the time budget
    n1 = max(1, min(len(toks), int(budget_s / 3 / max(dt * r.oracle.max_threads() / len(toks), 1e-6))))
    try:
        r.oracle.set_threads(1)
        t0 = time.perf_counter()
        r.run(toks[:n1])
        dt1 = time.perf_counter() - t0
    finally:
        r.oracle.set_threads(0)
    out["single_thread"] = {"value": round(n1 / dt1, 3), "unit": "tokens/s", "cores": 1,
                            "sample": f"the first {n1} tokens of the same sample"}
    return out


def run_reference(args, c, world, rank):
    if rank != 0:
        return
    import torch
    from nvfp4_mixture_experts_router_gb300 import synth
    device = "cuda" if torch.cuda.is_available() else "cpu"
    r = OracleRunner(c, device)
    # per-step sample sized so that warmup + steps fit in about two minutes
    probe = synth.sample_tokens(c, 1)
    r.prepare_for(probe)
    t0 = time.perf_counter()
    r.run(probe)
    per_tok = max(time.perf_counter() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = max(1, min(c.T, int(budget / per_tok)))
    samples = [synth.sample_tokens(c.with_(seed=c.seed), n)]
    toks = samples[0]
    r.prepare_for(toks)
    for _ in range(args.warmup):
        r.run(toks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r.run(toks)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1000 * dt / args.steps, 4), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64 (oracle, NVFP4 emulated)", "data": "synthetic",
           "config": {"workload": describe(c), "tokens_per_step": n},
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": r.oracle.max_threads(),
                            "kind": "oracle",
                            "sample": f"{n} token(s) of the workload per step, weights prepared untimed"},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

SWEEP_T = [1, 8, 64, 256, 1024, 4096, 8192]


def per_tensor_scales(api, c, flags, prepared, x, logits, bias, dev):
    """Calibration of the per-tensor activation scales: G1 = amax(x)/2688,
    G2 = the largest per-row FC2-input scale of a per-token pass of the
    library itself over the same tokens."""
    import torch
    g1 = (x.float().abs().max() / 2688.0).reshape(1).contiguous()
    tok = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, (flags & ~(3 << 2)) | api.MOE_W4A4_PER_TOKEN, dev)
    tok.prepared = prepared
    tok.forward(x, logits, bias)
    cap = tok.layout()["rows_cap"]
    rows = int(tok.view("meta", torch.int32, 4)[0])
    g2 = tok.view("g2", torch.float32, cap)[:rows].max().reshape(1).contiguous()
    del tok
    return g1, g2


def forward_times(fn, n, flush=None, graph=False):
    """CUDA-event times of n forwards, each timed alone: median, p10, p90 (ms).
    flush: a buffer larger than L2, written before every forward outside its
    events (cold L2).  graph: the forward is captured once into a CUDA graph
    and each timed call is one replay (launch overhead of one graph)."""
    import torch
    call = fn
    if graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        call = g.replay
        for _ in range(3):
            call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        if flush is not None:
            flush.fill_(1)
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) for a, b in evs)
    q = lambda f: round(t[min(n - 1, int(round(f * (n - 1))))], 5)
    return {"median_ms": q(0.5), "p10_ms": q(0.1), "p90_ms": q(0.9), "n": n}


def dsv3_sweep(dev, steps, warmup, fp4_peak):
    """The DSV3-like expert shape over its token counts, one prepared weight
    set (6.3 GB) for all of them.  Every timed forward follows a 256 MB write
    that evicts L2 and is timed alone with CUDA events; the median is kept
    (p10 / p90 beside it), with the warm-L2 median (the same forward back to
    back) and, up to 256 tokens, the median of a CUDA-graph replay."""
    import torch
    from nvfp4_mixture_experts_router_gb300 import api, synth
    c0 = synth.config(2)
    flags = c0.flags()
    s0 = api.shape(SWEEP_T[-1], c0.H, c0.I, c0.E, c0.K)
    prep = torch.empty(api.moe_nvfp4_prepared_bytes(s0, flags), dtype=torch.uint8, device=dev)
    w1 = synth.gen_w1(c0, dev)
    w2 = synth.gen_w2(c0, dev)
    api.moe_nvfp4_prepare_weights(s0, flags, w1, w2, prep)
    torch.cuda.synchronize()
    del w1, w2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    points = []
    for T in SWEEP_T:
        c = synth.config(2, T)
        s = api.shape(T, c.H, c.I, c.E, c.K)
        x = synth.gen_x(c, dev)
        logits = synth.gen_logits(c, dev, x)
        g1, g2 = per_tensor_scales(api, c, flags, prep, x, logits, None, dev)
        ws = torch.empty(api.moe_nvfp4_workspace_bytes(s, flags), dtype=torch.uint8, device=dev)
        y = torch.empty(T, c.H, dtype=torch.bfloat16, device=dev)
        for _ in range(max(warmup, 3)):
            api.moe_nvfp4_forward(s, flags, x, logits, None, g1, g2, prep, ws, y)
        torch.cuda.synchronize()
        if api.moe_nvfp4_last_device_status(ws) != api.MOE_OK:
            raise RuntimeError(f"device status not OK in the DSV3 sweep at T={T}")
        n = max(5, min(steps, 50))
        fwd = lambda: api.moe_nvfp4_forward(s, flags, x, logits, None, g1, g2, prep, ws, y)
        cold = forward_times(fwd, n, flush)
        warm = forward_times(fwd, n)
        ms = cold["median_ms"]
        tflops = flops_per_step(c) / (ms / 1000.0) / 1e12
        pt = {"T": T, "ms": ms, "tokens_per_s": round(T / (ms / 1000.0), 1),
              "tflops": round(tflops, 2), "pct_fp4_peak": round(100 * tflops / fp4_peak, 3),
              "timed_steps": n, "p10_ms": cold["p10_ms"], "p90_ms": cold["p90_ms"], "warm_ms": warm["median_ms"]}
        if T <= 256:
            try:
                pt["graph_ms"] = forward_times(fwd, n, flush, graph=True)["median_ms"]
            except Exception as exc:
                pt["graph_ms"] = f"capture failed: {type(exc).__name__}"
        points.append(pt)
        del ws, y, x, logits
    return {"workload": describe(c0).split(":", 1)[1].replace(" T=4096,", "").strip(),
            "l2": "256 MB write before every timed forward (evicts L2); median (p10, p90) of per-forward "
                  "CUDA-event times; warm_ms: the same forward back to back; graph_ms: one CUDA-graph replay",
            "points": points}


def run_ours(args, c, world, rank, local):
    import torch
    import torch.distributed as dist
    from nvfp4_mixture_experts_router_gb300 import api, build, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    api.lib()

    gate = args.routing == "gate"
    flags = c.flags() | (api.MOE_ROUTER_GEMM if gate else 0)
    s = api.shape(c.T, c.H, c.I, c.E, c.K)
    x = synth.gen_x(c, dev)
    logits = synth.gen_logits(c, dev, x)
    wg = synth.gen_wg(c, dev) if gate else None
    if gate:
        # the logits the layer will compute itself (the calibration pass and
        # the stage timings below run on them)
        logits = torch.empty(c.T, c.E, dtype=torch.float32, device=dev)
        api.moe_nvfp4_router_logits(x, wg, logits)
    bias = synth.gen_bias(c, dev)
    g1 = g2 = None

    # prepared weights: enough copies that consecutive steps miss in L2
    pb = api.moe_nvfp4_prepared_bytes(s, flags)
    n_sets = max(1, min(8, math.ceil(3 * L2_BYTES / pb) if pb < 3 * L2_BYTES else 1))
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, flags, device=dev)
    w1 = synth.gen_w1(c, dev)
    w2 = synth.gen_w2(c, dev)
    preps = []
    for i in range(n_sets):
        buf = torch.empty(pb, dtype=torch.uint8, device=dev)
        api.moe_nvfp4_prepare_weights(s, flags, w1, w2, buf)
        preps.append(buf)
    torch.cuda.synchronize()
    del w1, w2
    if c.mode == synth.MODE_PER_TENSOR:
        g1, g2 = per_tensor_scales(api, c, c.flags(), preps[0], x, logits, bias, dev)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=dev)
    ws = layer.workspace
    given = args.routing == "given"
    if given:
        # caller-supplied routing: the ids and weights of one router pass,
        # fed to moe_nvfp4_forward_routed every step
        layer.prepared = preps[0]
        layer.forward(x, logits, bias, g1, g2)
        torch.cuda.synchronize()
        ids = layer.view("topk_ids", torch.int32, c.T * c.K).view(c.T, c.K).clone()
        wts = layer.view("topk_w", torch.float32, c.T * c.K).view(c.T, c.K).clone()

    def step(i, yy=y, xx=x, ll=logits, ii=None, ww=None):
        if given:
            api.moe_nvfp4_forward_routed(s, flags, xx, ids if ii is None else ii, wts if ww is None else ww,
                                         g1, g2, preps[i % n_sets], ws, yy)
        elif gate:
            api.moe_nvfp4_forward_gate(s, flags, xx, wg, bias, g1, g2, preps[i % n_sets], ws, yy)
        else:
            api.moe_nvfp4_forward(s, flags, xx, ll, bias, g1, g2, preps[i % n_sets], ws, yy)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    status = api.moe_nvfp4_last_device_status(ws)
    if status != api.MOE_OK:
        raise RuntimeError(f"device status {api.STATUS_NAMES.get(status)} after warm-up")

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record()
    for i in range(args.steps):
        step(i)
    ev1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    if rank == 0:
        clocks.stop()
    ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / args.steps
    value = job_tokens_per_s(world, c.T, args.steps, ms)

    # per-stage durations (stage events; programmatic dependent launch off)
    nst = min(args.stage_steps, max(args.steps, 1))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(api.NUM_STAGE_EVENTS)] for _ in range(nst)]
    staged_flags = flags & ~api.MOE_ROUTER_GEMM
    for i in range(nst):
        api.moe_nvfp4_forward_staged(s, staged_flags, x, logits, bias, g1, g2, preps[i % n_sets], ws, y, evs[i])
    torch.cuda.synchronize()
    stage_ms = {name: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(nst)) / nst
                for j, name in enumerate(api.STAGES)}
    if gate:
        # the logits kernel, timed on its own in front of the staged forward
        lg = torch.empty_like(logits)
        gevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nst)]
        for a, b in gevs:
            a.record()
            api.moe_nvfp4_router_logits(x, wg, lg)
            b.record()
        torch.cuda.synchronize()
        stage_ms = {"router_gemm": sum(a.elapsed_time(b) for a, b in gevs) / nst, **stage_ms}
    count = layer.view("count", torch.int32, c.E).cpu()
    active = int((count > 0).sum())
    # per-token: the FC2-input quantization is inside FC1 unless the launch
    # count shows the separate kernel
    h_fp32 = (c.mode == synth.MODE_PER_TOKEN and not c.fused and
              api.moe_nvfp4_forward_launches(s, c.flags()) == (6 if c.T <= 32 else 7))
    sbytes = stage_bytes(c, active, h_fp32)
    if not h_fp32:
        stage_ms.pop("quantize_h", None)        # no kernel between the FC1 and FC2 events
    if c.fused:
        # one kernel: its time is the forward's, its algorithmic bytes the
        # layer's irreducible traffic (routing input, x, the active experts'
        # weights, y); the intermediates may stay in L2
        stage_ms = {"fused_layer": sum(stage_ms.values())}
        nv = 0.5625
        sbytes = {"fused_layer": sbytes["router"] + c.T * c.H * 2 + active * (c.N1 * c.H + c.H * c.I) * nv +
                  c.T * c.H * 2}

    # each forward timed alone: cold L2 (a write larger than L2 before
    # every forward), warm L2 (the same inputs and weights back to back),
    # and up to 256 tokens the forward as one CUDA-graph replay
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    nd = max(5, min(args.steps, 50))
    per_forward = {"cold": forward_times(lambda: step(0), nd, flush), "warm": forward_times(lambda: step(0), nd),
                   "l2": "cold: a 256 MB write before every forward, outside its events; warm: the same "
                         "inputs and prepared weights back to back"}
    if c.T <= 256:
        try:
            per_forward["graph_cold"] = forward_times(lambda: step(0), nd, flush, graph=True)
        except Exception as exc:
            per_forward["graph_cold"] = f"capture failed: {type(exc).__name__}"
    del flush
    torch.cuda.synchronize()
    if api.moe_nvfp4_last_device_status(ws) != api.MOE_OK:
        raise RuntimeError("device status not OK after the per-forward timings")

    # end to end through the C ABI: every step copies its inputs (x and the
    # logits, or the given ids and weights) from pinned host memory, runs the
    # forward and copies y back to pinned host memory.  Pipelined as a user
    # of the library would: two device slots, the host-to-device copy of
    # step i+1 and the device-to-host copy of step i-1 on their own streams
    # while step i computes; events keep a slot from being overwritten
    # before the step that uses it is done.
    n_slot = 2
    hx = [x.cpu().pin_memory() for _ in range(n_slot)]
    hl = [logits.cpu().pin_memory() for _ in range(n_slot)]   # (unused by the gate routing: x is the input)
    if given:
        h_ids = [ids.cpu().pin_memory() for _ in range(n_slot)]
        h_wts = [wts.cpu().pin_memory() for _ in range(n_slot)]
        d_ids = [torch.empty_like(ids) for _ in range(n_slot)]
        d_wts = [torch.empty_like(wts) for _ in range(n_slot)]
    hy = [torch.empty(c.T, c.H, dtype=torch.bfloat16).pin_memory() for _ in range(n_slot)]
    dx = [torch.empty_like(x) for _ in range(n_slot)]
    dl = [torch.empty_like(logits) for _ in range(n_slot)]
    dy = [torch.empty_like(y) for _ in range(n_slot)]
    cs, ds = torch.cuda.Stream(), torch.cuda.Stream()
    h2d_done = [torch.cuda.Event() for _ in range(n_slot)]
    fwd_done = [torch.cuda.Event() for _ in range(n_slot)]
    d2h_done = [torch.cuda.Event() for _ in range(n_slot)]

    def e2e_step(i, ms):
        b = i % n_slot
        with torch.cuda.stream(cs):
            if i >= n_slot:
                cs.wait_event(fwd_done[b])         # step i - 2 has read slot b's inputs
            dx[b].copy_(hx[b], non_blocking=True)
            if given:
                d_ids[b].copy_(h_ids[b], non_blocking=True)
                d_wts[b].copy_(h_wts[b], non_blocking=True)
            elif not gate:
                dl[b].copy_(hl[b], non_blocking=True)
            h2d_done[b].record(cs)
        ms.wait_event(h2d_done[b])
        if i >= n_slot:
            ms.wait_event(d2h_done[b])             # step i - 2's y has left slot b
        with torch.cuda.stream(ms):
            if given:
                step(i, dy[b], dx[b], None, d_ids[b], d_wts[b])
            else:
                step(i, dy[b], dx[b], dl[b])
        fwd_done[b].record(ms)
        with torch.cuda.stream(ds):
            ds.wait_event(fwd_done[b])
            hy[b].copy_(dy[b], non_blocking=True)
            d2h_done[b].record(ds)

    def e2e_steps_on(ms, n):
        # fork the copy streams from ms, run n steps, join them back into ms
        fork = torch.cuda.Event()
        fork.record(ms)
        cs.wait_event(fork)
        ds.wait_event(fork)
        for i in range(n):
            e2e_step(i, ms)
        for ev in d2h_done[:min(n, n_slot)]:
            ms.wait_event(ev)
        join = torch.cuda.Event()
        join.record(cs)
        ms.wait_event(join)

    # A group of steps is captured once into a CUDA graph and replayed, so
    # that the host enqueues one graph per group instead of every copy,
    # event and kernel (at small T the host's launch rate would otherwise
    # bound the step); without a graph the same calls are enqueued directly.
    # Consecutive replays do not overlap (the first copy of a group waits
    # for the last step of the previous one), so a group is long: the
    # largest divisor of the step count up to 64, so that exactly `steps`
    # steps are timed.
    group = max(d for d in range(1, min(64, max(args.steps, 1)) + 1) if max(args.steps, 1) % d == 0)
    reps = max(args.steps, 1) // group
    e2e_steps = reps * group
    e2e_graph = None
    main = torch.cuda.current_stream()
    e2e_steps_on(main, group)                        # warm-up, outside any capture
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(main)
        # thread-local capture: CUDA calls of other threads (NCCL's watchdog
        # under torchrun) are not affected by it
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            e2e_steps_on(cap, group)
        torch.cuda.synchronize()
        for _ in range(min(args.warmup, 3)):
            g.replay()
        torch.cuda.synchronize()
        e2e_graph = g
        e2e_mode = f"steps replayed from a CUDA graph of {group} pipelined steps"
    except Exception as exc:                       # capture refused: enqueue the calls directly
        torch.cuda.synchronize()
        e2e_mode = f"pipelined steps enqueued directly (graph capture failed: {type(exc).__name__})"
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _ in range(reps):
        if e2e_graph is not None:
            e2e_graph.replay()
        else:
            e2e_steps_on(main, group)
    e1.record(main)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    # the pipelined steps returned the layer's output (the fused finalize's
    # reduction order may differ from run to run, hence a tolerance)
    y_ref = y.float().cpu()
    y_e2e = hy[(e2e_steps - 1) % n_slot].float()
    tol = 0.02 * float(y_ref.pow(2).mean().sqrt()) + 0.01 * float(y_ref.abs().max())
    if not bool(torch.isfinite(y_e2e).all()) or float((y_e2e - y_ref).abs().max()) > tol:
        raise RuntimeError("end-to-end output differs from the device-timed forward's")
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = job_tokens_per_s(world, c.T, e2e_steps, e2e_ms)
    h2d = c.T * c.H * 2 + (c.T * c.K * 8 if given else (0 if gate else c.T * c.E * 4))
    d2h = c.T * c.H * 2

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm, bf16, bf16s, peak_src = measured_peaks()
    mx = c.mode == synth.MODE_MXFP8
    w4a16 = c.mode == synth.MODE_W4A16
    ratio = FP8_OVER_BF16 if mx else FP4_OVER_BF16
    fp4_peak = bf16 * ratio           # the dense FP4 peak (FP8 for MXFP8): the metric's reference rate
    # the peak of the MMA kind the GEMMs run on: W4A16 widens the weights to
    # BF16 on chip and runs kind::f16, so its GEMMs are bounded by the BF16 peak
    gemm_peak, gemm_ratio = (bf16, 1.0) if w4a16 else (fp4_peak, ratio)
    gemm_kind = "bf16" if w4a16 else ("fp8" if mx else "fp4")
    flops = flops_per_step(c)
    dom = max(stage_ms, key=lambda k: stage_ms[k])
    dom_ms = stage_ms[dom]
    if dom in ("fc1", "fc2"):
        # GEMM: report the bound that limits it at this shape
        gemm_flops = 2.0 * c.T * c.K * c.H * (c.N1 if dom == "fc1" else c.I)
        t_flop = gemm_flops / (gemm_peak * 1e12)
        t_byte = sbytes[dom] / (hbm * 1e9)
        bound = "tensor" if t_flop > t_byte else "hbm"
    else:
        bound = "hbm"
        gemm_flops = 0.0
    if bound == "hbm":
        achieved = sbytes[dom] / (dom_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic_for(dom, traffic_key(args)),
                "kernel": dom, "algorithmic_bytes_per_launch": int(sbytes[dom]),
                "mean_launch_us": round(dom_ms * 1000, 2), "peak_source": f"{peak_src} hbm_gbs"}
    else:
        achieved = gemm_flops / (dom_ms / 1000.0) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(gemm_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / gemm_peak, 4), "traffic": traffic_for(dom, traffic_key(args)),
                "kernel": dom, "algorithmic_flops_per_launch": gemm_flops,
                "mean_launch_us": round(dom_ms * 1000, 2),
                "peak_source": (f"{peak_src} bf16_tflops (kind::f16 MMAs)" if w4a16 else
                                f"{peak_src} bf16_tflops x {gemm_ratio:g} (nominal {gemm_kind}/bf16 ratio)")}

    sweep = None
    if args.sweep == "dsv3" and world == 1:
        sweep = dsv3_sweep(dev, args.steps, args.warmup, bf16 * FP4_OVER_BF16)

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        try:
            cpu = cpu_baseline(c, dev)
        except Exception as ex:   # the baseline must not sink the GPU line
            cpu = {"value": None, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"failed: {type(ex).__name__}: {ex}"}

    tflops = flops / (ms_per_step / 1000.0) / 1e12
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp8 (e4m3 x e8m0/32) -> f32" if mx else "nvfp4 (e2m1 x e4m3/16) -> f32",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": describe(c), "T": c.T, "H": c.H, "I": c.I, "E": c.E, "K": c.K,
                   "l2": f"inputs larger than L2: {n_sets} prepared-weight copies "
                         f"({n_sets * pb / 1e6:.0f} MB) rotated across steps",
                   "parallelism": f"replicas x{world}"},
        "tflops": round(tflops, 2), "pct_fp4_peak": round(100 * tflops / fp4_peak, 3),
        "fp4_peak_tflops": round(fp4_peak, 1),
        "routing": args.routing + ("" if args.routing == "logits" else " (stage times from the logits path)"),
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipeline": "2 device slots; the H2D copy of step i+1 and the D2H copy of step i-1 run on two "
                            "copy streams while step i computes; " + e2e_mode},
        "gpu_launches": (api.moe_nvfp4_forward_launches(s, flags & ~api.MOE_ROUTER_GEMM) + (1 if gate else 0))
                        * args.steps,
        "roofline": roof,
        "per_forward": per_forward,
        "stages_us": {k: round(v * 1000, 2) for k, v in stage_ms.items()},
        "stage_gbs": {k: round(sbytes[k] / (stage_ms[k] / 1000) / 1e9, 1) for k in stage_ms if stage_ms[k] > 0},
        "active_experts": active,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
    }
    if sweep is not None:
        out["sweep"] = sweep
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    world, rank, local = init_dist(args)
    c = workload_config(args.workload, args.tokens, args.precision, args.four_over_six, args.fused, args.gemm,
                        args.finalize, args.experts)
    if args.impl == "reference":
        run_reference(args, c, world, rank)
    else:
        run_ours(args, c, world, rank, local)


if __name__ == "__main__":
    main()
