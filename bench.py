#!/usr/bin/env python3
"""Throughput of the W4A16 routed-expert MoE layer on one GB300 (per rank).

Workload (default, "decode"): 16 independent OLMoE-shaped MoE layers
(H=2048, I=1024, E=64, top-8, all experts resident), each run on its own batch
of T decode tokens.  One step = one forward of each of the 16 layers, i.e. the
whole hot path (router top-k, permutation, gate/up with in-kernel int4
dequantisation, SiLU*up, down, top-k combine) 16 times over 3.27 GB of
distinct packed weights, so every step streams its experts from HBM (the
touched weights of a step exceed the 129 MB L2).  The activations rotate over
8 seeded batches per layer.  Metric: MoE-layer tokens/s = 16 * T * steps /
time.  "prefill" runs the same stack at T = 2048.

Prints ONE JSON line (rank 0).  --impl reference times the float64 CPU oracle
on the same workload instead (bounded sample, host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (OLMoE-shaped W4A16 layer, packed-weight HBM roofline)"
UNIT = "tokens/s"
H, I, E, K_TOP = 2048, 1024, 64, 8
EXPERT_BYTES = 3_194_880
LAYERS = 16
ROTATE = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "prefill"], default="decode")
    ap.add_argument("--tokens", type=int, default=None, help="T per layer forward")
    ap.add_argument("--force", choices=["auto", "gemv", "unfused", "gemm"], default="auto",
                    help="gemv: decode kernels (single launch when it fits); unfused: decode kernels as "
                         "separate launches; gemm: tensor-core grouped GEMM")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=16, help="independent layers per step (16 = headline)")
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-max-steps", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args()


def tokens_of(args) -> int:
    if args.tokens:
        return args.tokens
    return 4 if args.workload == "decode" else 2048


def workload_config(args, T):
    global LAYERS
    LAYERS = args.layers
    return {"workload": f"OLMoE-shaped W4A16 MoE layer ({args.workload}), H={H} I={I} E={E} top-{K_TOP}, "
                        f"T={T} tokens per layer forward, {LAYERS} independent layers per step",
            "tokens_per_layer": T, "layers_per_step": LAYERS, "hidden": H, "inter": I, "experts": E, "top_k": K_TOP,
            "weights": "int4 qpacked, 256-value blocks, FP16 scales; all experts resident",
            "l2": "inputs larger than L2: 3.27 GB of distinct packed weights per step rotation",
            "activation_rotation": ROTATE}


# ------------------------------------------------------------ CPU oracle leg

def cpu_leg(args):
    """Times the float64 oracle (as it stands) on one OLMoE layer at T tokens."""
    import numpy as np  # noqa: F401
    from oracle import moe_oracle
    from w4a16_compact_expert_gb300 import synth
    T = tokens_of(args)
    layer = synth.olmoe_decode_layer()
    xs = [synth.draw_x(synth.SEED_OLMOE_DECODE + r, T, H) for r in range(ROTATE)]
    arrays = layer.experts.arrays()
    done, t0 = 0, time.perf_counter()
    while True:
        moe_oracle.moe_layer(xs[done % ROTATE], layer.router_w, layer.bias, arrays, K_TOP)
        done += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds or (args.cpu_max_steps and done >= args.cpu_max_steps):
            break
    print(json.dumps({"value": T * done / el, "steps": done, "seconds": el, "tokens": T}))


def run_cpu_leg(args, seconds, max_steps=0):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-leg", "--workload", args.workload,
           "--tokens", str(tokens_of(args)), "--cpu-seconds", str(seconds), "--cpu-max-steps", str(max_steps)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=seconds * 4 + 300)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, max_mhz_fallback):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz_fallback, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def src_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "w4a16_compact_expert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(kernel, tokens, sha):
    """dram bytes per launch recorded by an ncu capture (profiles/*.md line
    'bench-traffic: kernel=<k> tokens=<T> src=<sha> dram_bytes_per_launch=<n>')."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    pat = re.compile(r"bench-traffic: kernel=(\S+) tokens=(\d+) src=(\S+) dram_bytes_per_launch=(\d+)")
    for f in sorted(os.listdir(d)):
        if f.endswith((".md", ".txt")):
            for m in pat.finditer(open(os.path.join(d, f)).read()):
                if m.group(1) == kernel and int(m.group(2)) == tokens and m.group(3) == sha:
                    return int(m.group(4))
    return None


def gpu_arm(args, rank, world, local_rank):
    import torch
    global LAYERS
    LAYERS = args.layers

    from w4a16_compact_expert_gb300 import build_ext, moe_w4a16, synth
    build_ext.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    T = tokens_of(args)
    steps = args.steps or (4000 if args.workload == "decode" else 100)
    warm = max(3, args.warmup)
    force = {"auto": 0, "gemv": moe_w4a16.FORCE_GEMV, "unfused": moe_w4a16.FORCE_GEMV | moe_w4a16.UNFUSED,
             "gemm": moe_w4a16.FORCE_GEMM}[args.force]

    layers, rws, xs, outs = [], [], [], []
    g = torch.Generator(device=dev)
    for l in range(LAYERS):
        m = moe_w4a16.MoELayer(H, I, E, K_TOP, max_tokens=T, device=local_rank)
        ex = synth.device_random_experts(synth.OLMOE, E, seed=synth.SEED_OLMOE_STACK * 1000 + l, device=dev)
        m.pack_experts(0, *ex)
        m.set_slot_table(list(range(E)))
        del ex
        g.manual_seed(10_000 + l)
        rws.append((torch.randn(E, H, device=dev, generator=g) * 0.02).half())
        xs.append([torch.randn(T, H, device=dev, generator=g).half() for _ in range(ROTATE)])
        outs.append(torch.empty(T, H, device=dev, dtype=torch.float16))
        layers.append(m)
    torch.cuda.synchronize()

    # Unique experts actually routed per (layer, batch): algorithmic bytes.
    uniq = [[0] * ROTATE for _ in range(LAYERS)]
    for l, m in enumerate(layers):
        for r in range(ROTATE):
            _, dbg = m.forward(xs[l][r], rws[l], None, force, out=outs[l], debug=True)
            uniq[l][r] = int(torch.unique(dbg["ids"]).numel())
    torch.cuda.synchronize()
    for m in layers:
        st, miss = m.get_status()
        assert st == moe_w4a16.OK and miss == 0

    def step(r, events=None):
        for l, m in enumerate(layers):
            if events is not None:
                m.set_stage_events(events[l])
            m.forward(xs[l][r], rws[l], None, force, out=outs[l])

    for i in range(warm):
        step(i % ROTATE)
    torch.cuda.synchronize()
    path, launches = layers[0].last_path()
    assert all(m.last_path() == (path, launches) for m in layers)

    stream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(stream):
        for r in range(ROTATE):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                step(r)
            graphs.append(gr)
    for gr in graphs:
        gr.replay()
    torch.cuda.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(steps):
                graphs[i % ROTATE].replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    tokens_total = LAYERS * T * steps * world
    value = tokens_total / (ms / 1e3)

    # Per-kernel durations: the same steps captured with stage events.
    prof_steps = ROTATE
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(LAYERS)] for _ in range(prof_steps)]
    for row in evs:
        for per_layer in row:
            for e in per_layer:
                e.record(stream)   # creates the underlying CUDA events before capture
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=stream):
            for r in range(prof_steps):
                step(r, evs[r])
        for m in layers:
            m.set_stage_events(None)
        gp.replay()
        gp.replay()
    torch.cuda.synchronize()
    stage_ms = [[], [], [], []]
    for r in range(prof_steps):
        for l in range(LAYERS):
            e = evs[r][l]
            for s in range(4):
                stage_ms[s].append(e[s].elapsed_time(e[s + 1]))
    stage_avg = [statistics.mean(v) for v in stage_ms]
    avg_u = statistics.mean(u for row in uniq for u in row)
    gate_up_bytes = 2 * (I * H // 2 + I * ((H + 255) // 256) * 2)
    down_bytes = H * I // 2 + H * ((I + 255) // 256) * 2
    P = T * K_TOP
    # algorithmic bytes of the three stages: router (router weight + x),
    # gate/up (unique experts' gate+up + x + h), down (unique experts' down + h + out)
    stage_bytes = [E * H * 2 + T * H * 2,
                   avg_u * gate_up_bytes + T * H * 2 + P * I * 2,
                   avg_u * down_bytes + P * I * 2 + T * H * 2]
    layer_bytes = sum(stage_bytes)
    layer_flops = 2.0 * P * (3 * H * I) + 2.0 * T * E * H
    pname = moe_w4a16.PATH_NAMES[path]
    layer_ms = ms / (steps * LAYERS)
    if path == moe_w4a16.PATH_DECODE_FUSED:
        # the timed graphs hold nothing but these launches, back to back: the
        # timed region's events give the average launch duration directly
        # (stage events inside a graph add their own gaps)
        kern = {"fused_decode_kernel": (layer_ms, layer_bytes, layer_flops)}
        srcs = ["decode_fused.cu", "route_dev.cuh", "gemv_dev.cuh", "common.cuh", "layout.h"]
    elif path == moe_w4a16.PATH_DECODE:
        kern = {"route": (stage_avg[0], stage_bytes[0], 2.0 * T * E * H),
                "gemv_gateup_kernel": (stage_avg[1], stage_bytes[1], 2.0 * P * 2 * H * I),
                "gemv_down_kernel": (stage_avg[2] + stage_avg[3], stage_bytes[2], 2.0 * P * H * I)}
        srcs = ["gemv.cu", "gemv_dev.cuh", "common.cuh", "layout.h"]
    else:
        kern = {"route": (stage_avg[0], stage_bytes[0], 2.0 * T * E * H),
                "grouped_gemm_kernel<gate_up>": (stage_avg[1], stage_bytes[1], 2.0 * P * 2 * H * I),
                "grouped_gemm_kernel<down>": (stage_avg[2], stage_bytes[2], 2.0 * P * H * I),
                "combine_kernel": (stage_avg[3], 0, 0.0)}
        srcs = ["gemm_tc.cu", "common.cuh", "layout.h"]
    dom = max(kern, key=lambda n: kern[n][0])
    dom_ms, dom_bytes, dom_flops = kern[dom]
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    tensor = path == moe_w4a16.PATH_GEMM
    if tensor:
        # FP16 dense peak = the measured BF16 cuBLAS figure (same nominal rate
        # for FP16 and BF16 on this part); the GEMM runs inside a long step.
        peak = peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops")
        peak_src = "measured bf16_tflops_sustained (fp16 nominal = bf16)" if peak else "fallback"
        peak = peak or 1700.0
        achieved = dom_flops / (dom_ms / 1e3) / 1e12
        unit, work = "TFLOP/s", {"algorithmic_flops_per_launch": dom_flops}
    else:
        peak = peaks.get("hbm_gbs")
        peak_src = "measured hbm_gbs" if peak else "fallback"
        peak = peak or 6800.0
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        unit, work = "GB/s", {"algorithmic_bytes_per_launch": dom_bytes}
    hbm = peaks.get("hbm_gbs") or 6800.0
    sha = src_hash(srcs)

    # End-to-end through the C ABI with host buffers (pinned), copies timed.
    e2e_steps = max(10, min(200, steps // 10))
    xh = [[xs[l][r].cpu().pin_memory() for r in range(ROTATE)] for l in range(LAYERS)]
    oh = [torch.empty(T, H, dtype=torch.float16).pin_memory() for _ in range(LAYERS)]
    for r in range(2):
        for l, m in enumerate(layers):
            m.forward_host(xh[l][r], rws[l], None, force, out_host=oh[l])
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        for l, m in enumerate(layers):
            m.forward_host(xh[l][i % ROTATE], rws[l], None, force, out_host=oh[l])
    e2e_s = time.perf_counter() - t0
    if world > 1:
        t = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_value = LAYERS * T * e2e_steps * world / e2e_s

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 weights x fp16 activations, fp32 accumulate", "data": "synthetic (seeded)",
        "config": workload_config(args, T) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                             "path": pname, "cuda_graph": True},
        "roofline": {"bound": "tensor" if tensor else "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "peak_source": peak_src,
                     "avg_launch_us": dom_ms * 1e3, "traffic": profiled_traffic(dom, T, sha)} | work,
        "layer_roofline": {"algorithmic_bytes_per_layer": layer_bytes, "us_per_layer": layer_ms * 1e3,
                           "achieved_gbs": layer_bytes / (layer_ms / 1e3) / 1e9,
                           "hbm_frac": layer_bytes / (layer_ms / 1e3) / 1e9 / hbm,
                           "achieved_tflops": layer_flops / (layer_ms / 1e3) / 1e12,
                           "avg_unique_experts": avg_u},
        "kernel_us": {n: v[0] * 1e3 for n, v in kern.items()},
        "stage_event_us": [v * 1e3 for v in stage_avg],
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": LAYERS * T * H * 2,
                "d2h_bytes_per_step": LAYERS * T * H * 2, "steps": e2e_steps},
        "gpu_launches": steps * LAYERS * launches,
        "launches_per_layer_forward": launches,
        "clocks": clk.summary(peaks.get("sm_max_mhz")),
        "kernel_src": sha,
    }
    for m in layers:
        m.close()
    return res


def main():
    args = parse()
    if args.cpu_leg:
        cpu_leg(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    T = tokens_of(args)
    if args.impl == "reference":
        if rank != 0:
            return
        steps = args.steps or 20
        leg = run_cpu_leg(args, seconds=150.0, max_steps=steps + args.warmup)
        res = {"impl": "reference", "metric": METRIC, "value": leg["value"], "unit": UNIT, "n_gpus": args.gpus,
               "steps": leg["steps"], "warmup": 0, "ms_per_step": leg["seconds"] * 1e3 / leg["steps"],
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic (seeded)", "config": workload_config(args, T),
               "cpu_baseline": {"value": leg["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{leg['steps']} float64-oracle forwards of one {args.workload} layer at "
                                          f"T={T} (bounded by steps and 150 s)"},
               "e2e": {"value": leg["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    # CPU baseline first, in its own process, before this process touches the GPU.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        leg = run_cpu_leg(args, seconds=args.cpu_seconds)
        cpu = {"value": leg["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{leg['steps']} float64-oracle forwards of one OLMoE-shaped layer at T={T} in "
                         f"{leg['seconds']:.1f} s, 1 thread"}
    res = gpu_arm(args, rank, world, local_rank)
    res["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
