#!/usr/bin/env python3
"""Throughput of the W4A16 routed-expert MoE layer on one GB300 (per rank).

Workloads (--workload):
  decode   (default) 16 independent OLMoE-shaped layers (H=2048, I=1024,
           E=64, top-8, all experts resident), each run on its own batch of T
           decode tokens (default T=4).  One step = one forward of each layer:
           the whole hot path (router top-k, permutation, gate/up with in-kernel
           int4 dequantisation, SiLU*up, down, top-k combine) 16 times over
           3.27 GB of distinct packed weights, so every step streams its experts
           from HBM (more than the 129 MB L2).  Activations rotate over 8 seeded
           batches per layer.
  prefill  the same 16 layers at T=2048 (--variant 2: per-expert logit bias
           ~ N(0, 1), a skewed expert load).
  qwen     8 independent Qwen-MoE-shaped partial-residency pools (H=2048,
           I=1408, E=60, top-4, 39 resident experts at permuted slots, -inf
           logit bias for the 21 absent ones; 1.37 GB), default T=8.
  stack    16 OLMoE-shaped layers run in sequence, x <- x + MoE(rmsnorm(x)),
           T tokens; --sweep times T in {1, 8, 16, 24, 32, 48, 64, 128, 512, 2048} with the decode
           kernels and the grouped GEMM forced in turn and reports the
           crossover.
Metric: MoE-layer tokens/s = layers * T * steps / time.  The default decode
line also carries "prefill": the OLMoE prefill layers (T = 2048, both
variants) timed in the same run, with their TFLOP/s against the measured
FP16/BF16 dense peak.  Every timed region records one event pair per CUDA
graph replay (median, min, max) and samples the SM clock and clock-event
reasons through NVML every 2 ms.

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

METRIC = "MoE-layer tokens/s (W4A16 routed-expert layer; packed-weight HBM roofline for decode, FP16 tensor roofline for prefill)"
UNIT = "tokens/s"
ROTATE = 8


class Shape:
    def __init__(self, name, H, I, E, k, slots):
        self.name, self.H, self.I, self.E, self.k, self.slots = name, H, I, E, k, slots
        self.nb_h = (H + 255) // 256
        self.nb_i = (I + 255) // 256
        self.gate_up_bytes = 2 * (I * H // 2 + I * self.nb_h * 2)
        self.down_bytes = H * I // 2 + H * self.nb_i * 2
        self.expert_bytes = self.gate_up_bytes + self.down_bytes


OLMOE = Shape("OLMoE", 2048, 1024, 64, 8, 64)
QWEN = Shape("Qwen-MoE", 2048, 1408, 60, 4, 39)
SWEEP_T = [1, 8, 16, 24, 32, 48, 64, 128, 512, 2048]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "prefill", "qwen", "stack"], default="decode")
    ap.add_argument("--variant", type=int, default=1, help="prefill: 1 = no bias, 2 = logit bias ~ N(0, 1)")
    ap.add_argument("--tokens", type=int, default=None, help="T per layer forward")
    ap.add_argument("--force", choices=["auto", "gemv", "unfused", "gemm", "offload"], default="auto",
                    help="gemv: decode kernels (single launch when it fits); unfused: decode kernels as "
                         "separate launches; gemm: tensor-core grouped GEMM; offload: the offload-qpacked "
                         "comparison (expansion into FP16 execution slots, then the dense grouped GEMM)")
    ap.add_argument("--offload-slots", type=int, default=16, help="FP16 execution slots for --force offload")
    ap.add_argument("--sweep", action="store_true", help="stack: T sweep with both kernel families")
    ap.add_argument("--cache", action="store_true",
                    help="qwen: partial residency through the expert cache (misses copied from host memory)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode: skip the OLMoE prefill legs (T = 2048, both variants) timed after the decode line")
    ap.add_argument("--layers", type=int, default=None, help="layers (pools) per step")
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-max-steps", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-warmup", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args()


def shape_of(args):
    return QWEN if args.workload == "qwen" else OLMOE


def tokens_of(args) -> int:
    if args.tokens:
        return args.tokens
    return {"decode": 4, "prefill": 2048, "qwen": 8, "stack": 8}[args.workload]


def layers_of(args) -> int:
    if args.layers:
        return args.layers
    return 8 if args.workload == "qwen" else 16


def flags_of(args) -> int:
    from w4a16_compact_expert_gb300 import moe_w4a16 as M
    return (M.RESIDUAL | M.PRENORM) if args.workload == "stack" else 0


def workload_config(args, T):
    s, L = shape_of(args), layers_of(args)
    desc = {
        "decode": f"{L} independent OLMoE-shaped W4A16 MoE layers, decode batch",
        "prefill": f"{L} independent OLMoE-shaped W4A16 MoE layers, prefill batch"
                   + (", per-expert logit bias ~ N(0,1)" if args.variant == 2 else ""),
        "qwen": f"{L} independent Qwen-MoE-shaped partial-residency pools ({s.slots} of {s.E} experts resident "
                f"at permuted slots, -inf bias for absent)",
        "stack": f"{L} OLMoE-shaped W4A16 MoE layers in sequence, x <- x + MoE(rmsnorm(x))",
    }[args.workload]
    total = L * s.slots * s.expert_bytes
    return {"workload": f"{desc}: H={s.H} I={s.I} E={s.E} top-{s.k}, T={T} tokens per layer forward",
            "tokens_per_layer": T, "layers_per_step": L, "hidden": s.H, "inter": s.I, "experts": s.E,
            "top_k": s.k, "resident_slots": s.slots,
            "weights": "int4 qpacked, 256-value blocks, FP16 scales",
            "l2": f"inputs larger than L2: {total / 1e9:.2f} GB of distinct packed weights per step",
            "activation_rotation": ROTATE}


# ------------------------------------------------------------ CPU oracle leg

def cpu_leg(args):
    """Times the float64 oracle (as it stands) on single layers of the workload."""
    from oracle import moe_oracle
    from w4a16_compact_expert_gb300 import synth
    T = tokens_of(args)
    if args.workload == "qwen":
        layer = synth.qwen_partial_layer()
        seed = synth.SEED_QWEN_PARTIAL
    elif args.workload == "prefill":
        layer = synth.olmoe_prefill_layer(args.variant)
        seed = synth.SEED_OLMOE_PREFILL
    else:
        layer = synth.olmoe_decode_layer()
        seed = synth.SEED_OLMOE_DECODE
    flags = (moe_oracle.FLAG_RESIDUAL | moe_oracle.FLAG_PRENORM) if args.workload == "stack" else 0
    xs = [synth.draw_x(seed + r, T, layer.shape.hidden) for r in range(ROTATE)]
    experts = layer.slot_experts().arrays()
    for w in range(args.cpu_warmup):   # untimed
        moe_oracle.moe_layer(xs[w % ROTATE], layer.router_w, layer.bias, experts, layer.shape.top_k, flags,
                             layer.expert_to_slot)
    done, t0 = 0, time.perf_counter()
    while True:
        moe_oracle.moe_layer(xs[done % ROTATE], layer.router_w, layer.bias, experts, layer.shape.top_k, flags,
                             layer.expert_to_slot)
        done += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds or (args.cpu_max_steps and done >= args.cpu_max_steps):
            break
    print(json.dumps({"value": T * done / el, "steps": done, "seconds": el, "tokens": T}))


def run_cpu_leg(args, seconds, max_steps=0, warmup=0):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-leg", "--workload", args.workload,
           "--variant", str(args.variant), "--tokens", str(tokens_of(args)), "--cpu-seconds", str(seconds),
           "--cpu-max-steps", str(max_steps), "--cpu-warmup", str(warmup)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=seconds * 4 + 300)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_sample_text(args, leg):
    T = tokens_of(args)
    return (f"{leg['steps']} float64-oracle forwards of one {shape_of(args).name}-shaped layer at T={T} "
            f"in {leg['seconds']:.1f} s, 1 thread")


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(args):
    """The oracle as it stands on the host cores: one process with one BLAS
    thread, then one such process per core at once (each on its own rotating
    batches: token-parallel work, since tokens are independent); the
    all-cores rate is the sum of the processes' rates."""
    import concurrent.futures
    single = run_cpu_leg(args, seconds=args.cpu_seconds)
    n = os.cpu_count() or 1
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        legs = list(ex.map(lambda _: run_cpu_leg(args, seconds=args.cpu_seconds), range(n)))
    total = sum(l["value"] for l in legs)
    steps = sum(l["steps"] for l in legs)
    return {"value": total, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": (f"{n} processes at once (one per host core, 1 BLAS thread each), {steps} float64-oracle "
                       f"forwards of one {shape_of(args).name}-shaped layer at T={tokens_of(args)} in "
                       f"{max(l['seconds'] for l in legs):.1f} s; rate = sum of the processes' rates"),
            "single_thread": {"value": single["value"], "cores": 1, "sample": cpu_sample_text(args, single)},
            "nproc": n, "cpu_model": cpu_model()}


# ------------------------------------------------------------------ clocks

REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (read-only
    queries) from a thread every ~2 ms while the timed region runs, so even
    a region of a few milliseconds gets several samples.  Falls back to
    nvidia-smi (100 ms period) when the NVML library cannot be loaded."""

    def __init__(self, local_rank, period_s=0.002):
        self.local_rank, self.period = local_rank, period_s
        self.samples, self.source = [], None
        self.nvml = self.dev = None
        self._smi = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            dev = ctypes.c_void_p()
            found = False
            try:
                import torch
                pr = torch.cuda.get_device_properties(local_rank)
                bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
                found = nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(dev)) == 0
            except Exception:   # noqa: BLE001 - older torch: no PCI ids
                found = False
            if not found and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(local_rank), ctypes.byref(dev)) != 0:
                raise OSError("no NVML handle")
            self.nvml, self.dev = nv, dev
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(dev, ctypes.c_int(1), ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            self.source = "nvml"
        except OSError:
            self.source = "nvidia-smi"

    def _read(self):
        import ctypes
        nv, dev = self.nvml, self.dev
        clk, mw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        nv.nvmlDeviceGetClockInfo(dev, ctypes.c_int(1), ctypes.byref(clk))   # NVML_CLOCK_SM
        nv.nvmlDeviceGetPowerUsage(dev, ctypes.byref(mw))
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(dev, ctypes.byref(rs))
        return float(clk.value), mw.value / 1000.0, int(rs.value)

    def _loop(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self._read())
            except Exception:   # noqa: BLE001 - a failed query ends sampling
                return
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        if self.nvml is not None:
            self._stop = threading.Event()
            self.samples = [self._read()]
            self._thr = threading.Thread(target=self._loop, daemon=True)
            self._thr.start()
        else:
            self._smi = ClockSampler(self.local_rank).__enter__()
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self._stop.set()
            self._thr.join()
            self.samples.append(self._read())
        else:
            self._smi.__exit__(*exc)

    def summary(self, max_mhz_fallback):
        if self.nvml is None:
            return self._smi.summary(max_mhz_fallback) | {"source": "nvidia-smi"}
        sm = [c for c, _, _ in self.samples]
        reasons = sorted({n for _, _, r in self.samples for n, b in REASON_BITS.items() if r & b})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(p for _, p, _ in self.samples), "reasons": reasons,
                "samples": len(sm), "source": "nvml, 2 ms period"}


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


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


class Workload:
    """The device-resident layers of one run: handles, router weights, biases,
    the rotating activations and the output buffers."""

    def __init__(self, args, T, dev, local_rank):
        import numpy as np
        import torch
        from w4a16_compact_expert_gb300 import moe_w4a16, synth
        s = shape_of(args)
        self.shape, self.T, self.L = s, T, layers_of(args)
        self.chain = args.workload == "stack"
        self.flags = flags_of(args)
        self.layers, self.rws, self.biases = [], [], []
        g = torch.Generator(device=dev)
        base_seed = synth.SEED_QWEN_PARTIAL if s is QWEN else synth.SEED_OLMOE_STACK
        for l in range(self.L):
            m = moe_w4a16.MoELayer(s.H, s.I, s.E, s.k, num_slots=s.slots, max_tokens=T, device=local_rank)
            ex = synth.device_random_experts(synth.QWEN if s is QWEN else synth.OLMOE, s.slots,
                                             seed=base_seed * 1000 + l, device=dev)
            m.pack_experts(0, *ex)
            del ex
            g.manual_seed(10_000 + l)
            self.rws.append((torch.randn(s.E, s.H, device=dev, generator=g) * 0.02).half())
            if s.slots < s.E:
                # seeded resident subset at a seeded permutation of the slots; -inf bias for the rest
                rng = np.random.Generator(np.random.PCG64(base_seed * 1000 + l))
                resident = np.sort(rng.choice(s.E, s.slots, replace=False))
                slots = rng.permutation(s.slots)
                table = np.full(s.E, -1, dtype=np.int32)
                table[resident] = slots
                bias = np.where(table >= 0, 0.0, -np.inf).astype(np.float32)
                m.set_slot_table(table.tolist())
                self.biases.append(torch.from_numpy(bias).to(dev))
            else:
                m.set_slot_table(list(range(s.E)))
                if args.workload == "prefill" and args.variant == 2:
                    self.biases.append(torch.randn(s.E, device=dev, generator=g).float())
                else:
                    self.biases.append(None)
            if getattr(args, "force", "auto") == "offload":
                m.offload_enable(args.offload_slots)
            self.layers.append(m)
        g.manual_seed(20_000)
        if self.chain:
            self.xs = [torch.randn(T, s.H, device=dev, generator=g).half() for _ in range(ROTATE)]
            self.bufs = [torch.empty(T, s.H, device=dev, dtype=torch.float16) for _ in range(2)]
        else:
            self.xs = [[torch.randn(T, s.H, device=dev, generator=g).half() for _ in range(ROTATE)]
                       for _ in range(self.L)]
            self.outs = [torch.empty(T, s.H, device=dev, dtype=torch.float16) for _ in range(self.L)]
        torch.cuda.synchronize()

    def _io(self, l, r):
        if self.chain:
            return (self.xs[r] if l == 0 else self.bufs[(l - 1) % 2]), self.bufs[l % 2]
        return self.xs[l][r], self.outs[l]

    def step(self, r, force, events=None):
        for l, m in enumerate(self.layers):
            if events is not None:
                m.set_stage_events(events[l])
            x, out = self._io(l, r)
            m.forward(x, self.rws[l], self.biases[l], self.flags | force, out=out)

    def unique_experts(self, force):
        """Mean number of distinct routed experts per layer forward (from the
        actual routing); also keeps layer 0's count for each activation batch
        (self.u_layer0, in launch order: the batches r = 0 .. ROTATE - 1)."""
        import torch
        n = []
        self.u_layer0 = []
        for r in range(ROTATE):
            for l, m in enumerate(self.layers):
                x, out = self._io(l, r)
                _, dbg = m.forward(x, self.rws[l], self.biases[l], self.flags | force, out=out, debug=True)
                u = int(torch.unique(dbg["ids"]).numel())
                n.append(u)
                if l == 0:
                    self.u_layer0.append(u)
        torch.cuda.synchronize()
        return statistics.mean(n)

    def close(self):
        for m in self.layers:
            m.close()


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the whole job is as slow as its
    slowest replica); the value itself on one rank.  `device`: where the
    reduction tensor lives (the rank's GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (weak scaling: each rank runs the same work)."""
    return units_per_rank * world / seconds


def time_graphs(wl, force, steps, warm, stream, world, local_rank, peaks):
    import torch
    for i in range(warm):
        wl.step(i % ROTATE, force)
    torch.cuda.synchronize()
    graphs = []
    with torch.cuda.stream(stream):
        for r in range(ROTATE):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                wl.step(r, force)
            graphs.append(gr)
    for gr in graphs:
        gr.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # one event before every replay and one after the last: the timed region
    # is first to last, each replay's own duration the gap between neighbours
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with NvmlSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            for i in range(steps):
                evs[i].record(stream)
                graphs[i % ROTATE].replay()
            evs[steps].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(evs[0].elapsed_time(evs[steps]), world, torch.device("cuda", local_rank))
    per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
    stats = {"n": steps, "median_ms": statistics.median(per), "min_ms": per[0], "max_ms": per[-1]}
    return ms, clk.summary(peaks.get("sm_max_mhz")), stats


def stage_times(wl, force, stream):
    """Per-stage durations from one more capture of the same steps with stage events."""
    import torch
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(wl.L)] for _ in range(ROTATE)]
    for row in evs:
        for per_layer in row:
            for e in per_layer:
                e.record(stream)   # creates the underlying CUDA events before capture
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=stream):
            for r in range(ROTATE):
                wl.step(r, force, evs[r])
        for m in wl.layers:
            m.set_stage_events(None)
        gp.replay()
        gp.replay()
    torch.cuda.synchronize()
    stage_ms = [[], [], [], []]
    for r in range(ROTATE):
        for l in range(wl.L):
            e = evs[r][l]
            for s in range(4):
                stage_ms[s].append(e[s].elapsed_time(e[s + 1]))
    return [statistics.mean(v) for v in stage_ms]


def e2e_rate(wl, force, steps, world, local_rank):
    """Same metric through the host-buffer entry point (forward_host_async):
    pinned host x in, host out, copies and the per-step synchronisation timed."""
    import torch
    T, H = wl.T, wl.shape.H
    if wl.chain:
        xh = [wl.xs[r].cpu().pin_memory() for r in range(ROTATE)]
    else:
        xh = [[wl.xs[l][r].cpu().pin_memory() for r in range(ROTATE)] for l in range(wl.L)]
    oh = [torch.empty(T, H, dtype=torch.float16).pin_memory() for _ in range(2 if wl.chain else wl.L)]

    # independent layers alternate over two streams, so one layer's copies
    # overlap another layer's kernels; a chained stack stays on one stream
    # (stream order carries a layer's host output into the next layer's input)
    streams = [torch.cuda.current_stream()] if wl.chain else [torch.cuda.Stream(), torch.cuda.Stream()]

    def one(i):
        # every layer's H2D copy, forward and D2H copy enqueued, then one
        # synchronisation: the step's outputs are on the host
        for l, m in enumerate(wl.layers):
            if wl.chain:
                src = xh[i % ROTATE] if l == 0 else oh[(l - 1) % 2]
                m.forward_host_async(src, wl.rws[l], oh[l % 2], wl.biases[l], wl.flags | force)
            else:
                m.forward_host_async(xh[l][i % ROTATE], wl.rws[l], oh[l], wl.biases[l], wl.flags | force,
                                     stream=streams[l % 2])
        torch.cuda.synchronize()

    for i in range(2):
        one(i)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    el = max_over_ranks(time.perf_counter() - t0, world, torch.device("cuda", local_rank))
    return job_rate(wl.L * T * steps, world, el)


def roofline(wl, path, layer_ms, stage_avg, avg_u, peaks):
    from w4a16_compact_expert_gb300 import moe_w4a16 as M
    s, T = wl.shape, wl.T
    P = T * s.k
    stage_bytes = [s.E * s.H * 2 + T * s.H * 2,
                   avg_u * s.gate_up_bytes + T * s.H * 2 + P * s.I * 2,
                   avg_u * s.down_bytes + P * s.I * 2 + T * s.H * 2]
    layer_bytes = sum(stage_bytes)
    layer_flops = 2.0 * P * (3 * s.H * s.I) + 2.0 * T * s.E * s.H
    if path == M.PATH_DECODE_FUSED:
        # the timed graphs hold nothing but these launches, back to back: the
        # timed region's events give the average launch duration directly
        kern = {"fused_decode_kernel": (layer_ms, layer_bytes, layer_flops)}
        srcs = ["decode_fused.cu", "route_dev.cuh", "gemv_dev.cuh", "common.cuh", "layout.h"]
    elif path == M.PATH_DECODE:
        kern = {"route": (stage_avg[0], stage_bytes[0], 2.0 * T * s.E * s.H),
                "gemv_gateup_kernel": (stage_avg[1], stage_bytes[1], 2.0 * P * 2 * s.H * s.I),
                "gemv_down_kernel": (stage_avg[2] + stage_avg[3], stage_bytes[2], 2.0 * P * s.H * s.I)}
        srcs = ["gemv.cu", "gemv_dev.cuh", "common.cuh", "layout.h"]
    else:
        kern = {"route + gather_rows": (stage_avg[0], stage_bytes[0], 2.0 * T * s.E * s.H),
                "grouped_gemm_kernel<gate_up>": (stage_avg[1], stage_bytes[1], 2.0 * P * 2 * s.H * s.I),
                "grouped_gemm_kernel<down>": (stage_avg[2], stage_bytes[2], 2.0 * P * s.H * s.I),
                "combine_kernel": (stage_avg[3], 0, 0.0)}
        srcs = ["gemm_tc.cu", "common.cuh", "layout.h"]
    dom = max(kern, key=lambda n: kern[n][0])
    dom_ms, dom_bytes, dom_flops = kern[dom]
    tensor = path == M.PATH_GEMM
    hbm = peaks.get("hbm_gbs") or 6800.0
    if tensor:
        # FP16 dense peak = the measured BF16 cuBLAS figure (same nominal rate
        # for FP16 and BF16 on this part); the GEMM runs inside a long step.
        peak = peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops")
        src = "measured bf16_tflops_sustained (fp16 nominal = bf16)" if peak else "fallback"
        peak = peak or 1700.0
        achieved = dom_flops / (dom_ms / 1e3) / 1e12
        unit, work = "TFLOP/s", {"algorithmic_flops_per_launch": dom_flops}
    else:
        peak = peaks.get("hbm_gbs")
        src = "measured hbm_gbs" if peak else "fallback"
        peak = peak or 6800.0
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        unit, work = "GB/s", {"algorithmic_bytes_per_launch": dom_bytes}
    sha = src_hash(srcs)
    roof = {"bound": "tensor" if tensor else "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
            "unit": unit, "frac": achieved / peak, "peak_source": src, "avg_launch_us": dom_ms * 1e3,
            "traffic": profiled_traffic(dom, T, sha)} | work
    per_batch = [u * (s.gate_up_bytes + s.down_bytes) + (layer_bytes - avg_u * (s.gate_up_bytes + s.down_bytes))
                 for u in getattr(wl, "u_layer0", [])]
    layer = {"algorithmic_bytes_per_layer": layer_bytes, "us_per_layer": layer_ms * 1e3,
             "layer0_unique_experts_per_batch": getattr(wl, "u_layer0", []),
             "layer0_algorithmic_bytes_per_batch": per_batch,
             "achieved_gbs": layer_bytes / (layer_ms / 1e3) / 1e9,
             "hbm_frac": layer_bytes / (layer_ms / 1e3) / 1e9 / hbm,
             "achieved_tflops": layer_flops / (layer_ms / 1e3) / 1e12, "avg_unique_experts": avg_u}
    return roof, layer, {n: v[0] * 1e3 for n, v in kern.items()}, sha


def prefill_legs(args, dev, local_rank, world, peaks, stream, steps=60):
    """OLMoE-shaped prefill (T = 2048), both variants, timed in the same run as
    the decode line: 16 layers per step, one CUDA-graph replay per step."""
    import torch
    from w4a16_compact_expert_gb300 import moe_w4a16 as M
    res = {}
    sus = peaks.get("bf16_tflops_sustained") or 1700.0
    burst = peaks.get("bf16_tflops") or 1900.0
    for variant in (1, 2):
        a = argparse.Namespace(**vars(args))
        a.workload, a.variant, a.tokens = "prefill", variant, 2048
        T = 2048
        wl = Workload(a, T, dev, local_rank)
        ms, clocks, replay = time_graphs(wl, 0, steps, 3, stream, world, local_rank, peaks)
        path, launches = wl.layers[0].last_path()
        stage_avg = stage_times(wl, 0, stream)
        for m in wl.layers:
            st, miss = m.get_status()
            assert st == M.OK and miss == 0, (st, miss)
        s = wl.shape
        P = T * s.k
        layer_s = ms / 1e3 / (steps * wl.L)
        flops = 2.0 * P * 3 * s.H * s.I + 2.0 * T * s.E * s.H
        gu_s = stage_avg[1] / 1e3
        gu_tf = 2.0 * P * 2 * s.H * s.I / gu_s / 1e12
        tf = flops / layer_s / 1e12
        res[f"variant{variant}"] = {
            "workload": workload_config(a, T)["workload"], "path": M.PATH_NAMES[path],
            "launches_per_layer_forward": launches, "steps": steps, "tokens_per_s": job_rate(wl.L * T * steps,
                                                                                              world, ms / 1e3),
            "us_per_layer": layer_s * 1e6, "algorithmic_flops_per_layer": flops, "tflops": tf,
            "frac_sustained": tf / sus, "frac_burst": tf / burst,
            "gemm_gate_up_us": stage_avg[1] * 1e3, "gemm_gate_up_tflops": gu_tf,
            "gemm_gate_up_frac_sustained": gu_tf / sus, "gemm_down_us": stage_avg[2] * 1e3,
            "route_gather_us": stage_avg[0] * 1e3, "combine_us": stage_avg[3] * 1e3,
            "step_replays": replay, "clocks": clocks,
            "peaks": {"sustained_tflops": sus, "burst_tflops": burst,
                      "source": "measured bf16 (fp16 nominal = bf16)"}}
        wl.close()
        del wl
        torch.cuda.empty_cache()
    return res


def force_flag(name):
    from w4a16_compact_expert_gb300 import moe_w4a16 as M
    return {"auto": 0, "gemv": M.FORCE_GEMV, "unfused": M.FORCE_GEMV | M.UNFUSED, "gemm": M.FORCE_GEMM,
            "offload": M.OFFLOAD}[name]


def gpu_arm(args, rank, world, local_rank):
    import torch
    from w4a16_compact_expert_gb300 import build_ext, moe_w4a16
    build_ext.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    T = tokens_of(args)
    steps = args.steps or (4000 if T <= 64 else 100)
    warm = max(3, args.warmup)
    force = force_flag(args.force)
    peaks = load_peaks()
    wl = Workload(args, T, dev, local_rank)
    avg_u = wl.unique_experts(force)
    for m in wl.layers:
        st, miss = m.get_status()
        assert st == moe_w4a16.OK and miss == 0, (st, miss)
    stream = torch.cuda.Stream(device=dev)
    ms, clocks, replay = time_graphs(wl, force, steps, warm, stream, world, local_rank, peaks)
    path, launches = wl.layers[0].last_path()
    assert all(m.last_path() == (path, launches) for m in wl.layers)
    value = job_rate(wl.L * T * steps, world, ms / 1e3)
    stage_avg = stage_times(wl, force, stream)
    layer_ms = ms / (steps * wl.L)
    roof, layer, kern_us, sha = roofline(wl, path, layer_ms, stage_avg, avg_u, peaks)
    e2e_steps = max(10, min(200, steps // 10))
    e2e = e2e_rate(wl, force, e2e_steps, world, local_rank)
    s = wl.shape
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded)",
        "config": workload_config(args, T) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                             "path": moe_w4a16.PATH_NAMES[path], "cuda_graph": True,
                                             "arithmetic": "int4 weights dequantised to f16 operands, "
                                                           "f16 activations, f32 accumulation"},
        "roofline": roof, "layer_roofline": layer, "kernel_us": kern_us,
        "stage_event_us": [v * 1e3 for v in stage_avg],
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": wl.L * T * s.H * 2,
                "d2h_bytes_per_step": wl.L * T * s.H * 2, "steps": e2e_steps},
        "gpu_launches": steps * wl.L * launches, "launches_per_layer_forward": launches,
        "clocks": clocks, "kernel_src": sha,
        "step_replays": replay | {"note": "one CUDA-graph replay = one step (every layer once); per-replay "
                                          "durations from an event pair around each replay"},
    }
    if args.workload == "decode" and args.force == "auto" and not args.tokens and not args.no_prefill:
        wl.close()
        del wl
        torch.cuda.empty_cache()
        res["prefill"] = prefill_legs(args, dev, local_rank, world, peaks, stream)
        return res
    if path == moe_w4a16.PATH_OFFLOAD:
        # what the expansion moves per layer, next to the compact path's weight bytes
        exp_bytes = avg_u * 3 * s.I * s.H * 2
        res["offload"] = {"execution_slots": args.offload_slots, "avg_active_experts": avg_u,
                          "expanded_fp16_bytes_written_per_layer": exp_bytes,
                          "fp16_weight_bytes_read_per_layer": exp_bytes,
                          "compact_weight_bytes_per_layer": avg_u * s.expert_bytes}
    wl.close()
    return res


def stack_sweep(args, rank, world, local_rank):
    """T sweep of the 16-layer stack with each kernel family forced; crossover T*."""
    import torch
    from w4a16_compact_expert_gb300 import build_ext, moe_w4a16
    build_ext.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    rows = []
    for T in SWEEP_T:
        a = argparse.Namespace(**vars(args))
        a.tokens = T
        wl = Workload(a, T, dev, local_rank)
        row = {"T": T}
        for fam in ("gemv", "gemm"):
            force = force_flag(fam)
            steps = args.steps or max(5, min(400, 4096 // T))
            ms, clocks, _ = time_graphs(wl, force, steps, 3, stream, world, local_rank, peaks)
            path, _ = wl.layers[0].last_path()
            row[fam] = {"tokens_per_s_per_layer": job_rate(T * steps, world, ms / 1e3),
                        "us_per_layer": ms * 1e3 / (steps * wl.L), "path": moe_w4a16.PATH_NAMES[path],
                        "sm_mhz": clocks["sm_mhz"], "reasons": clocks["reasons"]}
        for m in wl.layers:
            st, miss = m.get_status()
            assert st == moe_w4a16.OK and miss == 0, (st, miss)
        wl.close()
        del wl
        torch.cuda.empty_cache()
        rows.append(row)
    cross = next((r["T"] for r in rows if r["gemm"]["us_per_layer"] < r["gemv"]["us_per_layer"]), None)
    return {"metric": "per-layer tokens/s of the 16-layer OLMoE-shaped stack, decode kernels vs grouped GEMM",
            "unit": UNIT, "n_gpus": world, "config": workload_config(args, 0) | {"sweep_T": SWEEP_T},
            "rows": rows, "crossover_T": cross,
            "crossover_note": "smallest swept T at which the grouped GEMM is faster than the decode kernels"}


def cache_bench(args, rank, world, local_rank):
    """Qwen-shaped layer, 39 published slot rows over all 60 experts: each step
    routes T tokens on the GPU, reads the ids, acquires the routed group
    through the expert cache (misses stream from the host backing through
    pinned staging), runs the forward and releases the lease."""
    import numpy as np
    import torch
    from w4a16_compact_expert_gb300 import build_ext, moe_w4a16 as M, synth
    build_ext.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    s, T = QWEN, tokens_of(args)
    steps = args.steps or 200
    rng = np.random.Generator(np.random.PCG64(synth.SEED_QWEN_PARTIAL))
    E, H, I = s.E, s.H, s.I
    backing = (rng.integers(0, 256, (E, I, H // 2), dtype=np.uint8),
               (rng.uniform(0.002, 0.02, (E, I, s.nb_h)).astype(np.float16)).view(np.uint16),
               rng.integers(0, 256, (E, I, H // 2), dtype=np.uint8),
               (rng.uniform(0.002, 0.02, (E, I, s.nb_h)).astype(np.float16)).view(np.uint16),
               rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
               (rng.uniform(0.002, 0.02, (E, H, s.nb_i)).astype(np.float16)).view(np.uint16))
    group = min(E, T * s.k)
    m = M.MoELayer(H, I, E, s.k, num_slots=s.slots + group, max_tokens=T, device=local_rank)
    cache = M.ExpertCache(m, backing, staging_experts=4, spare_slots=group, max_group=group,
                          initial=list(range(s.slots)))
    g = torch.Generator(device=dev)
    g.manual_seed(30_000)
    rw = (torch.randn(E, H, device=dev, generator=g) * 0.02).half()
    xs = [torch.randn(T, H, device=dev, generator=g).half() for _ in range(ROTATE)]
    out = torch.empty(T, H, device=dev, dtype=torch.float16)

    def one(i):
        ids, _, _, _ = M.route_noalloc(xs[i % ROTATE], rw, None, E, s.k)
        grp = sorted(set(ids.cpu().numpy().ravel().tolist()))
        lease = cache.acquire(grp)
        m.forward(xs[i % ROTATE], rw, None, 0, out=out)
        cache.release(lease)

    for i in range(max(3, args.warmup)):
        one(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    s0 = cache.stats()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t0, world, torch.device("cuda", local_rank))
    s1 = cache.stats()
    st, miss = m.get_status()
    assert st == M.OK and miss == 0, (st, miss)
    misses = s1["misses"] - s0["misses"]
    hits = s1["hits"] - s0["hits"]
    h2d = s1["h2d_bytes"] - s0["h2d_bytes"]
    cfg = workload_config(args, T)
    cfg["workload"] = (f"one Qwen-MoE-shaped layer (H={H} I={I} E={E} top-{s.k}), {s.slots} published slot rows over "
                       f"all {E} experts through the expert cache, T={T} tokens per step")
    cfg["layers_per_step"] = 1
    cfg["l2"] = "misses copied from host memory; resident weights 171 MB"
    res = {"metric": "MoE-layer tokens/s with the expert cache's miss path in the loop",
           "value": job_rate(T * steps, world, el), "unit": UNIT, "n_gpus": world, "steps": steps,
           "ms_per_step": el * 1e3 / steps, "higher_is_better": True,
           "config": cfg | {"path": "route + acquire + forward + release per step",
                                                "published_rows": s.slots, "spare_rows": group,
                                                "staging_experts": 4, "backing": "host memory, all 60 experts"},
           "cache": {"misses_per_step": misses / steps, "hit_rate": hits / max(1, hits + misses),
                     "h2d_gbs": h2d / el / 1e9, "d2h_bytes": s1["d2h_bytes"], "evictions": s1["evictions"],
                     "lease_waits": s1["lease_waits"], "generation": s1["generation"]}}
    cache.close()
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
        leg = run_cpu_leg(args, seconds=150.0, max_steps=steps, warmup=args.warmup)
        res = {"impl": "reference", "metric": METRIC, "value": leg["value"], "unit": UNIT, "n_gpus": args.gpus,
               "steps": leg["steps"], "warmup": args.warmup, "ms_per_step": leg["seconds"] * 1e3 / leg["steps"],
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic (seeded)", "config": workload_config(args, T),
               "cpu_baseline": {"value": leg["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": cpu_sample_text(args, leg) + " (bounded by steps and 150 s)"},
               "e2e": {"value": leg["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if args.sweep:
        res = stack_sweep(args, rank, world, local_rank)
    elif args.cache:
        res = cache_bench(args, rank, world, local_rank)
    else:
        # CPU baseline first, in its own process, before this process touches the GPU.
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(args)
        res = gpu_arm(args, rank, world, local_rank)
        res["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
