#!/usr/bin/env python
"""Throughput benchmark of the SSD selective scan on one GB300 (or N replicas).

One step = one chunked SSD prefill of the Mamba-2-2.7B-shaped layer workload
(batch 8, L 2048, 80 heads, headdim 64, d_state 128, 1 group, bf16
x/dt/B/C/y with float32 state and accumulation, seeded synthetic inputs), at
the best static chunk of a 64/128/256 sweep. The timed region replays a CUDA
graph of exactly K steps; the steps rotate over copies of the inputs whose
total size exceeds the L2 cache, so every step reads its inputs from HBM.

Each of the other legs has its own timed region and is reported in the same
final JSON line: the 130M-shaped layer and the 2.7B-shaped layer at B1
L1024 / L4096 / L8192 (each with its chunk sweep), the decode step (batch 64,
80 heads, 1000 in-place steps in one graph), the decode-layer body, the
Mamba-1 diagonal scan (B8 L2048 D5120 N16, chunk sweep) and its softplus
timing shape, and the SSD backward. Every leg reports the mean and standard
deviation over 30 timed repetitions and a single-call latency, beside the
float64 oracle timed on the host cores on a bounded sample of the same
workload. A first JSON line ("details") carries the descriptions; the last
line is the result.

`--impl reference` times the float64 CPU oracle on the headline workload (a
bounded sample of tokens per step) and prints the same kind of line.
`--chunk-table` measures the best chunk over a grid of shapes (the table the
library's static chunk policy is built from) and prints it.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU (weak
scaling, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "ssd_m2_2p7b_B8_L2048"
PREFILL_LEGS = ("ssd_m2_130m_L4096", "ssd_m2_2p7b_L1024", "ssd_m2_2p7b_L4096", "ssd_m2_2p7b_L8192")
DECODE = "decode_B64_H80"
MAMBA1 = "mamba1_B8_L2048_D5120"
MAMBA1_SP = "mamba1_B1_L4096_D1024_softplus"
LEGS = ("headline", "prefill", "decode", "decode_layer", "mamba1", "mamba1_softplus", "backward")
METRIC = "SSD prefill tokens/s + % roofline; decode steps/s + state HBM GB/s"
# stages between the events of a staged call, per kernel path
STAGES = {"fused": ("flag_clear", "-", "chunk_fused"), "staged": ("chunk_state", "state_pass", "chunk_scan"),
          "simt": ("chunk_state", "state_pass", "chunk_scan")}
KERNELS_PER_STEP = {"fused": 2, "staged": 3, "simt": 3}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
REPS = 30  # timed repetitions behind every mean and standard deviation


# ----------------------------------------------------------------- helpers

def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int, device="cpu") -> float:
    """Max of a float over ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def file_hash(*paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def host_cpu() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def ssd_compulsory_bytes(w: dict, io_bytes: int = 2) -> dict:
    """Algorithmic bytes of one prefill: every input read once, y and the final
    state written once (no initial state in these workloads)."""
    Bz, L, H, P, N, G = w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    tok = Bz * L
    x = tok * H * P * io_bytes
    dt = tok * H * io_bytes
    bc = tok * G * N * io_bytes
    return {"x": x, "dt": dt, "B": bc, "C": bc, "y": x, "final_state": Bz * H * P * N * 4,
            "total": 2 * x + dt + 2 * bc + Bz * H * P * N * 4}


def stage_algorithmic_bytes(w: dict, stage: str) -> int:
    """Compulsory bytes each stage kernel must move (intermediate workspace
    traffic is overhead, not credited)."""
    b = ssd_compulsory_bytes(w)
    if stage == "chunk_state":
        return b["x"] + b["dt"] + b["B"]
    if stage == "state_pass":
        return b["final_state"]
    if stage == "chunk_fused":
        return b["total"]
    if stage == "flag_clear":
        return 0
    return b["x"] + b["dt"] + b["B"] + b["C"] + b["y"]


def ssd_flops(w: dict, Q: int) -> float:
    """Useful flops (causal MACs x2 of intra-chunk, chunk-state and output
    contractions, C.B^T once per group)."""
    Bz, L, H, P, N, G = w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    return float(Bz * L * (H * (Q * P + 4 * N * P) + G * Q * N))


def mean_std(xs):
    return float(statistics.mean(xs)), float(statistics.stdev(xs)) if len(xs) > 1 else 0.0


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def _traffic_record(key: str):
    """ncu DRAM bytes (read + write) recorded in profiles/traffic.json under
    `key`, only if none of its kernels' sources changed since the capture;
    else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    srcs = [os.path.join(ROOT, "mamba_ssd_selective_gb300", "csrc", s) for s in rec.get("sources", [])]
    if not srcs or not all(os.path.exists(s) for s in srcs) or file_hash(*srcs) != rec.get("source_hash"):
        return None
    return rec


# --------------------------------------------------------------- prefill legs

class Prefill:
    """One prefill workload on the device: inputs rotating over copies whose
    total exceeds 3x the L2 cache, a workspace per copy."""

    def __init__(self, torch, binding, inputs, dev, name, l2):
        self.torch, self.binding, self.dev, self.name = torch, binding, dev, name
        w = self.w = dict(inputs.WORKLOADS[name])
        Bz, L, H, P, N, G = w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
        self.shape = (Bz, L, H, P, N, G)
        bf = torch.bfloat16
        d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=0)

        def t_(a, dtype=torch.float32):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

        self.base = {"x": t_(d["x"], bf), "dt": t_(d["dt"], bf), "B": t_(d["B"], bf), "C": t_(d["C"], bf)}
        self.A, self.D = t_(d["A"]), t_(d["D"])
        del d
        self.ws_max = max(binding.ssd_workspace_size(Bz, L, H, P, N, G, bf, q) for q in (64, 128, 256))
        in_bytes = sum(v.numel() * v.element_size() for v in self.base.values())
        self.per_set = 2 * in_bytes + self.ws_max + Bz * H * P * N * 4
        self.n_sets = max(2, math.ceil(3 * l2 / self.per_set))
        self.sets = []
        for _ in range(self.n_sets):
            s = {k: v.clone() for k, v in self.base.items()}
            s["y"] = torch.empty_like(self.base["x"])
            s["final"] = torch.empty((Bz, H, P, N), dtype=torch.float32, device=dev)
            s["ws"] = torch.empty(self.ws_max, dtype=torch.uint8, device=dev)
            self.sets.append(s)

    def step(self, i, q, stream=None):
        s = self.sets[i % self.n_sets]
        self.binding.ssd_scan_chunked(s["x"], s["dt"], self.A, s["B"], s["C"], self.D, None, chunk_size=q,
                                      y=s["y"], final_state=s["final"], workspace=s["ws"], stream=stream)

    def path(self, q):
        Bz, L, H, P, N, G = self.shape
        return self.binding.ssd_scan_path(Bz, L, H, P, N, G, self.torch.bfloat16, q)

    def capture(self, nsteps, q, stage_events=None):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream(device=self.dev)
        stream.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(stream):
            for i in range(min(nsteps, self.n_sets)):  # eager warm-up on the capture stream
                self.step(i, q)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for i in range(nsteps):
                if stage_events is not None:
                    self.binding.ssd_record_stage_events(stage_events[i])
                self.step(i, q)
        return g

    def replay_ms(self, g, reps=1):
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1)

    def sweep(self, W):
        """ms per step at chunk 64 / 128 / 256, graph of back-to-back steps."""
        out = {}
        S = 4 * self.n_sets
        for q in (64, 128, 256):
            g = self.capture(S, q)
            for _ in range(max(W, 3)):
                g.replay()
            out[q] = self.replay_ms(g, reps=3) / (3 * S)
            del g
        return out

    def rep_stats(self, q, W):
        """Mean and standard deviation of the per-step time over REPS replays of
        a graph of back-to-back steps, and the single-call latency (one eager
        call between events, REPS times)."""
        torch = self.torch
        S = 2 * self.n_sets
        g = self.capture(S, q)
        for _ in range(max(W, 3)):
            g.replay()
        per = [self.replay_ms(g) / S for _ in range(REPS)]
        del g
        one = []
        for r in range(REPS):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(self.dev)
            e0.record()
            self.step(r, q)
            e1.record()
            torch.cuda.synchronize(self.dev)
            one.append(e0.elapsed_time(e1))
        m, sd = mean_std(per)
        return {"mean_ms": m, "std_ms": sd, "reps": REPS, "single_call_ms": statistics.median(one)}

    def stage_ms(self, q, nsteps):
        """Per-stage kernel times: events between the stages of every step of a
        graph of nsteps steps; the stages then run without programmatic overlap,
        so each kernel is timed alone."""
        torch = self.torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nsteps)]
        for row in evs:
            for e in row:
                e.record()
        torch.cuda.synchronize(self.dev)
        g = self.capture(nsteps, q, stage_events=evs)
        g.replay()
        torch.cuda.synchronize(self.dev)
        names = STAGES[self.path(q)]
        out = {nm: statistics.mean(r[i].elapsed_time(r[i + 1]) for r in evs) for i, nm in enumerate(names)
               if nm != "-"}
        del g
        return out

    def close(self):
        del self.sets, self.base
        self.torch.cuda.empty_cache()


def prefill_leg(torch, binding, inputs, dev, name, W, hbm_peak, l2):
    """A prefill leg: chunk sweep, best chunk, REPS-repetition statistics and
    single-call latency at that chunk, fraction of the HBM roofline."""
    pf = Prefill(torch, binding, inputs, dev, name, l2)
    try:
        sweep = pf.sweep(W)
        q = min(sweep, key=sweep.get)
        st = pf.rep_stats(q, W)
        comp = ssd_compulsory_bytes(pf.w)["total"]
        tokens = pf.w["batch"] * pf.w["seqlen"]
        return {"w": name.replace("ssd_m2_", ""), "q": q, "path": pf.path(q), "us": round(st["mean_ms"] * 1e3, 1),
                "std": round(st["std_ms"] * 1e3, 1), "one_us": round(st["single_call_ms"] * 1e3, 1),
                "Mtok_s": round(tokens / st["mean_ms"] / 1e3, 1),
                "frac": round(comp / (st["mean_ms"] / 1e3) / 1e9 / hbm_peak, 4),
                "sweep_us": [round(sweep[k] * 1e3, 1) for k in (64, 128, 256)]}
    finally:
        pf.close()


# ------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    from mamba_ssd_selective_gb300 import binding, inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    binding.load()
    peaks = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0)) or 129 * 2 ** 20
    K, W = args.steps, args.warmup
    legs = set(args.legs.split(",")) if args.legs else set(LEGS)
    if args.skip_extra:
        legs = {"headline"}
    details, compact = {}, {}
    line = None

    sampler = ClockSampler(local).start() if rank == 0 else None

    # ---------------- the headline: B8 L2048 H80 prefill
    if "headline" in legs:
        pf = Prefill(torch, binding, inputs, dev, HEADLINE, l2)
        w = pf.w
        Bz, L, H, P, N, G = pf.shape
        sweep = pf.sweep(W)
        best_q = args.chunk or min(sweep, key=sweep.get)
        path = pf.path(best_q)

        # the timed region: exactly K steps in one graph
        g = pf.capture(K, best_q)
        gw = pf.capture(max(W, 3), best_q)
        for _ in range(2):
            gw.replay()
        # keep the GPU busy ~1 s before the timed region so that the clock
        # samples describe the clocks under this load
        if rank == 0:
            t_end = time.time() + 1.0
            while time.time() < t_end:
                gw.replay()
                torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("timed_region")
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        barrier(world)
        ms_total = reduce_max(e0.elapsed_time(e1), world, device=dev)
        ms_step = ms_total / K
        tokens = Bz * L
        value = world * tokens * K / (ms_total / 1e3)
        del g, gw

        stats = pf.rep_stats(best_q, W)
        stage_ms = pf.stage_ms(best_q, min(K, 64))
        dom = max(stage_ms, key=stage_ms.get)
        dom_bytes = stage_algorithmic_bytes(w, dom)
        achieved = dom_bytes / (stage_ms[dom] / 1e3) / 1e9
        comp = ssd_compulsory_bytes(w)
        traffic = _traffic_record(f"step:{HEADLINE}:{path}:{best_q}")
        step_gbs = comp["total"] / (ms_step / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4), "launch_ms": round(stage_ms[dom], 5),
                    "alg_bytes": dom_bytes,
                    "traffic": traffic["read"] + traffic["write"] if traffic else None,
                    "tr_ratio": round((traffic["read"] + traffic["write"]) / comp["total"], 3) if traffic
                    else None,
                    "step_frac": round(step_gbs / hbm_peak, 4), "peak_src": peaks["source"]}
        details["headline"] = {
            "workload": HEADLINE, "path": path, "chunk_sweep_ms_per_step": {str(k): round(v, 5) for k, v in sweep.items()},
            "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
            "tflops": round(ssd_flops(w, best_q) / (ms_step / 1e3) / 1e12, 2),
            "chunk_policy": binding.ssd_best_chunk(Bz, L, H, P, N, G, torch.bfloat16),
            "l2": f"inputs rotate over {pf.n_sets} copies ({pf.n_sets * pf.per_set / 2**20:.0f} MiB > L2 "
                  f"{l2 / 2**20:.0f} MiB)",
            "traffic_record": traffic,
            "roofline_note": "frac: the dominant kernel alone (stages launched without programmatic overlap, CUDA "
                             "events between them) against its algorithmic bytes; step_frac: the whole step "
                             "(graph of K steps) against the compulsory bytes; traffic: ncu DRAM read + write "
                             "bytes of one step's kernels, in steady state (cache control off, the next step "
                             "evicts the previous one's written lines)",
        }
        e2e = e2e_headline(torch, binding, pf, best_q, K, W, world, tokens)
        pf.close()
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": HEADLINE, "batch": Bz, "seqlen": L, "nheads": H, "headdim": P, "dstate": N,
                       "ngroups": G, "chunk": best_q, "path": path, "l2": "inputs > L2",
                       "parallelism": "replicas" if world == 1 else f"replicas x{world}"},
            "timing": {"mean_ms": round(stats["mean_ms"], 5), "std_ms": round(stats["std_ms"], 5), "reps": REPS,
                       "single_call_ms": round(stats["single_call_ms"], 5)},
            "roofline": roofline,
            "gpu_launches": KERNELS_PER_STEP[path] * K,
            "e2e": {k: v for k, v in e2e.items() if k not in ("pipeline", "steps")},
        }
        details["e2e"] = e2e

    # ---------------- the other legs
    if "prefill" in legs:
        compact["prefill"] = [prefill_leg(torch, binding, inputs, dev, nm, W, hbm_peak, l2) for nm in PREFILL_LEGS]
    if "decode" in legs:
        compact["decode"] = bench_decode(torch, binding, inputs, dev, hbm_peak, W)
    if "decode_layer" in legs:
        compact["decode_layer"] = [bench_decode_layer(torch, binding, inputs, dev, hbm_peak, nm, W)
                                   for nm in ("decode_layer_B64_H80", "decode_layer_B1_H128_G8")]
    if "mamba1" in legs:
        compact["mamba1"] = bench_mamba1(torch, binding, inputs, dev, hbm_peak, K, W)
    if "mamba1_softplus" in legs:
        compact["mamba1_softplus"] = bench_mamba1_softplus(torch, binding, inputs, dev, hbm_peak, K, W)
    if "backward" in legs:
        compact["backward"] = bench_backward(torch, binding, inputs, dev, hbm_peak, W, bwd_shape(args))
        if getattr(args, "bwd_shape", None) is None:
            # and the 2.7B-shaped layer at B4 L2048, where the chunk states and parts cross HBM
            compact["backward_2p7b"] = bench_backward(torch, binding, inputs, dev, hbm_peak, W, (4, 2048, 80))

    clocks = sampler.stop() if sampler else None
    if rank != 0:
        return
    if not args.skip_cpu:
        oracle_beside(compact, details)
    if line is None:  # no headline leg: a line of the other legs alone
        line = {"metric": METRIC, "value": None, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": "legs only"}}
    line["legs"] = compact
    if not args.skip_cpu and "headline" in legs:
        line["cpu_baseline"] = cpu_baseline(inputs_workload(HEADLINE))
    if clocks is not None:
        line["clocks"] = clocks
    print(json.dumps({"details": details}), flush=True)
    print(json.dumps(line), flush=True)


def inputs_workload(name):
    from mamba_ssd_selective_gb300 import inputs
    return dict(inputs.WORKLOADS[name])


def e2e_headline(torch, binding, pf, q, K, W, world, tokens):
    """The headline metric end to end through the C ABI with host buffers:
    every step copies its inputs from pinned host memory and its results (y
    and the final state) back. The inputs of a step are one packed host
    buffer (one copy in), its outputs one packed device buffer (one copy
    out); three streams overlap the copy in of step i + 1, the scan of step i
    and the copy out of step i - 1 over two device buffer sets."""
    dev, bf = pf.dev, torch.bfloat16
    Bz, L, H, P, N, G = pf.shape
    base = pf.base
    in_parts = [("x", base["x"]), ("dt", base["dt"]), ("B", base["B"]), ("C", base["C"]), ("A", pf.A), ("D", pf.D)]

    def carve(buf, parts):
        views, off = {}, 0
        for name, like in parts:
            nbytes = like.numel() * like.element_size()
            views[name] = buf[off:off + nbytes].view(like.dtype).view(like.shape)
            off += (nbytes + 255) // 256 * 256
        return views

    def packed_bytes(parts):
        return sum((t.numel() * t.element_size() + 255) // 256 * 256 for _, t in parts)

    y_like = torch.empty(base["x"].shape, dtype=bf, device=dev)
    f_like = torch.empty((Bz, H, P, N), dtype=torch.float32, device=dev)
    out_parts = [("y", y_like), ("final", f_like)]
    hin = torch.empty(packed_bytes(in_parts), dtype=torch.uint8).pin_memory()
    hout = torch.empty(packed_bytes(out_parts), dtype=torch.uint8).pin_memory()
    hv = carve(hin, in_parts)
    for name, t in in_parts:
        hv[name].copy_(t.cpu())
    dsets = []
    for _ in range(2):
        din = torch.empty(hin.numel(), dtype=torch.uint8, device=dev)
        dout = torch.empty(hout.numel(), dtype=torch.uint8, device=dev)
        dsets.append({"din": din, "dout": dout, "in": carve(din, in_parts), "out": carve(dout, out_parts),
                      "ws": torch.empty(pf.ws_max, dtype=torch.uint8, device=dev)})
    s_cap, s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(4))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "run", "out")}

    def e2e_step(i):
        d = dsets[i & 1]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["run"][i & 1])  # the scan two steps back has read these inputs
            d["din"].copy_(hin, non_blocking=True)
            ev["in"][i & 1].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev["in"][i & 1])
            if i >= 2:
                s_run.wait_event(ev["out"][i & 1])  # the outputs two steps back have been copied out
            v, o = d["in"], d["out"]
            binding.ssd_scan_chunked(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], None, chunk_size=q,
                                     y=o["y"], final_state=o["final"], workspace=d["ws"], stream=s_run)
            ev["run"][i & 1].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["run"][i & 1])
            hout.copy_(d["dout"], non_blocking=True)
            ev["out"][i & 1].record(s_out)

    def capture_e2e(nsteps):
        g = torch.cuda.CUDAGraph()
        s_cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.graph(g, stream=s_cap, capture_error_mode="relaxed"):
            fork = torch.cuda.Event()
            fork.record(s_cap)
            for st in (s_in, s_run, s_out):
                st.wait_event(fork)
            for i in range(nsteps):
                e2e_step(i)
            for st in (s_in, s_run, s_out):
                s_cap.wait_stream(st)
        return g

    Ke = max(1, min(K, 200))
    for i in range(max(W, 3)):  # eager warm-up (tensor maps, lazy loading)
        e2e_step(i)
    torch.cuda.synchronize(dev)
    ge = capture_e2e(Ke)
    ge.replay()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_cap):
        e0.record(s_cap)
        ge.replay()
        e1.record(s_cap)
    torch.cuda.synchronize(dev)
    ms_e2e = reduce_max(e0.elapsed_time(e1), world, device=dev)
    del ge, dsets
    h2d = sum(t.numel() * t.element_size() for _, t in in_parts)
    d2h = sum(t.numel() * t.element_size() for _, t in out_parts)
    return {"value": round(world * tokens * Ke / (ms_e2e / 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": Ke,
            "pipeline": "packed pinned buffers; copy in / scan / copy out overlapped on three streams; K steps in "
                        "one CUDA graph"}


def graph_rep_stats(torch, g, steps_per_replay, reps=REPS):
    """Mean and standard deviation (ms per step) over `reps` replays of a graph."""
    per = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) / steps_per_replay)
    return mean_std(per)


def batch_rep_stats(torch, fn, per_batch=10, reps=REPS):
    """Mean and standard deviation (ms per call) over `reps` batches of
    `per_batch` back-to-back calls, each batch between events."""
    per = []
    for r in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for i in range(per_batch):
            fn(r * per_batch + i)
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) / per_batch)
    return mean_std(per)


def call_rep_stats(torch, fn, reps=REPS):
    """Mean and standard deviation (ms) of single calls, each between events."""
    per = []
    for i in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        fn(i)
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1))
    return mean_std(per)


def bench_decode_layer(torch, binding, inputs, dev, hbm_peak, name, W):
    """The decode layer body (conv step, SSD decode step, gated norm) over
    `steps` tokens as one CUDA graph the library captures; per-step inputs are
    separate slices (16 generated steps repeated, > L2 in total)."""
    w = inputs.WORKLOADS[name]
    Bz, H, P, N, G, Wc, steps = (w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["width"],
                                 w["steps"])
    bf = torch.bfloat16
    Cc = H * P + 2 * G * N

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    prm = inputs.decode_layer_params(Bz, H, P, N, G, Wc, seed=0)
    pool = [inputs.decode_layer_step_inputs(k, Bz, H, P, N, G, io_dtype="bf16", seed=0) for k in range(16)]
    xBC = torch.empty((steps, Bz, Cc), dtype=bf, device=dev)
    dts = torch.empty((steps, Bz, H), dtype=bf, device=dev)
    zs = torch.empty((steps, Bz, H * P), dtype=bf, device=dev)
    for k, src in enumerate(pool):
        xBC[k].copy_(t_(src["xBC"], bf))
        dts[k].copy_(t_(src["dt"], bf))
        zs[k].copy_(t_(src["z"], bf))
    for k in range(len(pool), steps):
        for buf in (xBC, dts, zs):
            buf[k].copy_(buf[k % len(pool)])
    cst, sst = t_(prm["conv_state"]), t_(prm["ssm_state"])
    cw, cb, A, Dv, nw = t_(prm["conv_w"]), t_(prm["conv_b"]), t_(prm["A"]), t_(prm["D"]), t_(prm["norm_w"])
    graph = binding.DecodeGraph(xBC, cst, cw, cb, dts, A, Dv, sst, zs, nw, norm_group=w["norm_group"])
    try:
        for _ in range(max(W, 3)):
            graph.launch()
        torch.cuda.synchronize(dev)
        per = []
        for _ in range(REPS):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record()
            graph.launch()
            e1.record()
            torch.cuda.synchronize(dev)
            per.append(e0.elapsed_time(e1) * 1e3 / steps)
        us, sd = mean_std(per)
    finally:
        graph.close()
    one, _ = call_rep_stats(torch, lambda i: binding.decode_layer_step(xBC[i], cst, cw, cb, dts[i], A, Dv, sst, zs[i],
                                                                       nw, norm_group=w["norm_group"]))
    nbytes = (2 * Bz * H * P * N * 4 + 2 * Bz * Cc * Wc * 4 + Bz * Cc * 2 + Cc * Wc * 4 + Cc * 4
              + Bz * H * 2 + 2 * Bz * H * P * 2 + H * P * 4 + 2 * H * 4)
    gbs = nbytes / (us / 1e6) / 1e9
    return {"w": name.replace("decode_layer_", "layer_"), "us": round(us, 2), "std": round(sd, 2),
            "one_us": round(one * 1e3, 1), "steps_s": round(1e6 / us, 1), "frac": round(gbs / hbm_peak, 4)}


def bench_decode(torch, binding, inputs, dev, hbm_peak, W):
    w = inputs.WORKLOADS[DECODE]
    Bz, H, P, N, G, steps = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["steps"]
    bf = torch.bfloat16

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    state = t_(inputs.decode_state(Bz, H, P, N, seed=0))
    prm = inputs.decode_params(H, seed=0)
    A, Dv = t_(prm["A"]), t_(prm["D"])
    xs = torch.empty((steps, Bz, H, P), dtype=bf, device=dev)
    dts = torch.empty((steps, Bz, H), dtype=bf, device=dev)
    Bs = torch.empty((steps, Bz, G, N), dtype=bf, device=dev)
    Cs = torch.empty((steps, Bz, G, N), dtype=bf, device=dev)
    for s in range(steps):
        di = inputs.decode_step_inputs(s, Bz, H, P, N, G, io_dtype="bf16", seed=0)
        xs[s], dts[s], Bs[s], Cs[s] = t_(di["x"], bf), t_(di["dt"], bf), t_(di["B"], bf), t_(di["C"], bf)
    ys = torch.empty_like(xs)
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        binding.ssd_decode_step(state, xs[0], dts[0], A, Bs[0], Cs[0], Dv, y=ys[0])
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for s in range(steps):
            binding.ssd_decode_step(state, xs[s], dts[s], A, Bs[s], Cs[s], Dv, y=ys[s])
    for _ in range(max(W, 3) // 3 + 1):
        g.replay()
    torch.cuda.synchronize(dev)
    ms, sd = graph_rep_stats(torch, g, steps)
    del g
    one, _ = call_rep_stats(torch, lambda i: binding.ssd_decode_step(state, xs[i], dts[i], A, Bs[i], Cs[i], Dv,
                                                                     y=ys[i]))
    state_bytes = 2 * Bz * H * P * N * 4
    step_bytes = state_bytes + Bz * H * P * 2 * 2 + Bz * H * 2 + 2 * Bz * G * N * 2
    gbs = step_bytes / (ms / 1e3) / 1e9
    tr = _traffic_record("kernel:decode_step")
    return {"w": DECODE, "us": round(ms * 1e3, 2), "std": round(sd * 1e3, 2), "one_us": round(one * 1e3, 1),
            "steps_s": round(1e3 / ms, 1), "state_gbs": round(state_bytes / (ms / 1e3) / 1e9, 1),
            "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4), "frac_8tbs": round(gbs / 8000.0, 4),
            "tr_ratio": round((tr["read"] + tr["write"]) / step_bytes, 3) if tr else None}


MAMBA1_PROBE_MHZ = 2070.0  # the SM clock the pipe-rate probe's rates are per (the GB300's maximum)


def bench_mamba1(torch, binding, inputs, dev, hbm_peak, K, W):
    w = inputs.WORKLOADS[MAMBA1]
    Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
    bf = torch.bfloat16
    d = inputs.diag_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=0)

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    x, dt, Bm, Cm = t_(d["x"], bf), t_(d["dt"], bf), t_(d["B"], bf), t_(d["C"], bf)
    A, Dv = t_(d["A"]), t_(d["D"])
    del d
    y = torch.empty_like(x)
    hT = torch.empty((Bz, Dm, N), dtype=torch.float32, device=dev)
    reps = max(5, min(K, 50))

    def run(i, chunk):
        binding.selective_scan_diag(x, dt, A, Bm, Cm, Dv, None, chunk_size=chunk, y=y, final_state=hT)

    sweep = {}
    for chunk in (256, 512, 1024, 2048):
        for i in range(max(W, 3)):
            run(i, chunk)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            run(i, chunk)
        e1.record()
        torch.cuda.synchronize(dev)
        sweep[chunk] = e0.elapsed_time(e1) / reps
    best = min(sweep, key=sweep.get)
    ms, sd = batch_rep_stats(torch, lambda i: run(i, best), per_batch=5)
    one, _ = call_rep_stats(torch, lambda i: run(i, best))
    nbytes = 3 * Bz * L * Dm * 2 + 2 * Bz * L * N * 2 + Dm * N * 4 + Dm * 4 + Bz * Dm * N * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    tr = _traffic_record("kernel:diag_scan")
    # The scan's pipe floor beside its HBM fraction: one ex2 and two packed
    # float32 FMA-pipe instructions per state update, at the rates the probe
    # tests/probes/xu_fma_rates.cu measured on GB300 (29.4 ex2 and 59.4
    # fma.rn.f32x2 per SM per clock), at the device's SM count and maximum clock
    props = torch.cuda.get_device_properties(dev)
    sm_hz = MAMBA1_PROBE_MHZ * 1e6
    per_update = max(1.0 / 29.4, 2.0 / 59.4)  # SM clocks per state update on the busier pipe
    pipe_floor_s = Bz * L * Dm * N * per_update / (props.multi_processor_count * sm_hz)
    return {"w": MAMBA1, "q": best, "us": round(ms * 1e3, 1), "std": round(sd * 1e3, 1), "one_us": round(one * 1e3, 1),
            "Mtok_s": round(Bz * L / ms / 1e3, 2), "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
            "pipe_floor_us": round(pipe_floor_s * 1e6, 1), "pipe_frac": round(pipe_floor_s / (ms / 1e3), 4),
            "tr_ratio": round((tr["read"] + tr["write"]) / nbytes, 3) if tr else None,
            "sweep_us": [round(sweep[k] * 1e3, 1) for k in (256, 512, 1024, 2048)]}


def bench_mamba1_softplus(torch, binding, inputs, dev, hbm_peak, K, W):
    """selective_scan_fn's kernel-level timing shape with delta_softplus: B1
    L4096 D1024 N16 (24 MB of I/O), inputs rotated over 8 copies (> L2)."""
    w = inputs.WORKLOADS[MAMBA1_SP]
    Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
    bf = torch.bfloat16
    d = inputs.diag_option_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=0, bias=False, z=False)

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    n_sets = 8
    sets = [dict(x=t_(d["x"], bf), dt=t_(d["dt"], bf), B=t_(d["B"], bf), C=t_(d["C"], bf),
                 y=torch.empty((Bz, L, Dm), dtype=bf, device=dev)) for _ in range(n_sets)]
    A, Dv = t_(d["A"]), t_(d["D"])
    hT = torch.empty((Bz, Dm, N), dtype=torch.float32, device=dev)
    ws_bytes = binding.selective_scan_diag_workspace_size(Bz, L, Dm, N, bf)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    launches = 3 if ws_bytes else 1   # segment-local scan, segment pass, output scan

    def run(i, chunk):
        s_ = sets[i % n_sets]
        binding.selective_scan_diag(s_["x"], s_["dt"], A, s_["B"], s_["C"], Dv, None, chunk_size=chunk, y=s_["y"],
                                    final_state=hT, delta_softplus=True, workspace=ws)

    for i in range(max(W, 3)):
        run(i, 2048)
    torch.cuda.synchronize(dev)
    ms, sd = batch_rep_stats(torch, lambda i: run(i, 2048))
    one, _ = call_rep_stats(torch, lambda i: run(i, 2048))
    nbytes = 3 * Bz * L * Dm * 2 + 2 * Bz * L * N * 2 + Dm * N * 4 + Dm * 4 + Bz * Dm * N * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"w": MAMBA1_SP, "q": 2048, "us": round(ms * 1e3, 1), "std": round(sd * 1e3, 1), "one_us": round(one * 1e3, 1),
            "Mtok_s": round(Bz * L / ms / 1e3, 2), "frac": round(gbs / hbm_peak, 4), "kernels": launches}


def bwd_shape(args):
    """(B, L, H) of the backward leg: the 130M-shaped layer at L 2048 unless
    --bwd-shape names another."""
    return tuple(int(v) for v in (getattr(args, "bwd_shape", None) or "1,2048,24").split(","))


def bench_backward(torch, binding, inputs, dev, hbm_peak, W, shape=(1, 2048, 24)):
    """SSD backward (recompute, adjoint states, per-chunk gradients) on the
    130M-shaped layer at L 2048 (or another (B, L, H) with P 64, N 128, one
    group), bf16 inputs, float32 gradients; input copies rotate past L2."""
    Bz, L, H = shape
    P, N, G = 64, 128, 1
    bf = torch.bfloat16
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=0)
    rng = np.random.default_rng(1)
    dy = inputs.round_to(rng.standard_normal(d["x"].shape), "bf16")

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    n_sets = 8
    sets = [dict(x=t_(d["x"], bf), dt=t_(d["dt"], bf), B=t_(d["B"], bf), C=t_(d["C"], bf), dy=t_(dy, bf))
            for _ in range(n_sets)]
    A, Dv = t_(d["A"]), t_(d["D"])
    dims = binding._dims(Bz, L, H, P, N, G, binding.SSD_BF16)
    ws = torch.empty(int(binding.load().ssd_scan_chunked_bwd_workspace_size(binding.ctypes.byref(dims))),
                     dtype=torch.uint8, device=dev)

    def run(i):
        s_ = sets[i % n_sets]
        return binding.ssd_scan_chunked_bwd(s_["x"], s_["dt"], A, s_["B"], s_["C"], s_["dy"], Dv, workspace=ws)

    for i in range(max(W, 3)):
        run(i)
    torch.cuda.synchronize(dev)
    ms, sd = batch_rep_stats(torch, run, per_batch=5)
    # compulsory bytes: x, dt, B, C, dy read (bf16); dx, ddt, dB, dC written (float32)
    nbytes = Bz * L * (2 * H * P + H + 2 * G * N) * 2 + Bz * L * (H * P + H + 2 * G * N) * 4
    name = "bwd_130m_L2048" if shape == (1, 2048, 24) else f"bwd_B{Bz}_L{L}_H{H}"
    return {"w": name, "shape": [Bz, L, H], "us": round(ms * 1e3, 1), "std": round(sd * 1e3, 1),
            "Mtok_s": round(Bz * L / ms / 1e3, 2), "frac": round(nbytes / (ms / 1e3) / 1e9 / hbm_peak, 4)}


# ------------------------------------------------------------ CPU oracle

def oracle_sample_tokens(w: dict, seconds: float, threads: int) -> int:
    """Tokens of the workload (from the start of the sequence, all batches and
    heads) the oracle processes in about `seconds`, measured on a short probe."""
    import oracle
    from mamba_ssd_selective_gb300 import inputs
    probe = min(64, w["seqlen"])
    d = inputs.ssd_inputs(w["batch"], probe, w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                          io_dtype="bf16", seed=0)
    t0 = time.perf_counter()
    oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=threads)
    dt_probe = max(time.perf_counter() - t0, 1e-4)
    return int(max(16, min(w["seqlen"], probe * seconds / dt_probe)))


def cpu_baseline(w: dict, seconds: float = 10.0) -> dict:
    """The float64 oracle, as it stands, on a bounded sample of the workload."""
    import oracle
    from mamba_ssd_selective_gb300 import inputs
    threads = oracle.default_threads()
    Ls = oracle_sample_tokens(w, seconds / 2, threads)
    d = inputs.ssd_inputs(w["batch"], Ls, w["nheads"], w["headdim"], w["dstate"], w["ngroups"], io_dtype="bf16",
                          seed=0)
    # repeat the sample until about `seconds` of host time have been spent
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 10000:
            break
    return {"value": round(w["batch"] * Ls * reps / el, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "cpu": host_cpu(),
            "sample": f"first {Ls} of {w['seqlen']} tokens of all {w['batch']} sequences and {w['nheads']} heads, "
                      f"float64 token loop, {reps} rep(s) in {el:.1f} s"}


def _timed(fn, seconds):
    """Seconds per call of fn, repeated for about `seconds` (at least once)."""
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            return el / reps, reps


def oracle_beside(compact: dict, details: dict, seconds: float = 2.0) -> None:
    """The float64 oracle, as it stands, timed on the host cores beside each
    leg on a bounded sample of its workload, in the leg's own unit: the value
    goes into the leg as "cpu", the sample's description into the details."""
    import oracle
    from mamba_ssd_selective_gb300 import inputs
    thr = oracle.default_threads()
    notes = details.setdefault("oracle_samples", {"cores": thr, "cpu": host_cpu()})

    for leg in compact.get("prefill", []):
        w = inputs.WORKLOADS["ssd_m2_" + leg["w"]]
        Ls = oracle_sample_tokens(w, seconds / 2, thr)
        d = inputs.ssd_inputs(w["batch"], Ls, w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                              io_dtype="bf16", seed=0)
        per, reps = _timed(lambda: oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=thr),
                           seconds)
        leg["cpu"] = round(w["batch"] * Ls / per, 1)
        notes[leg["w"]] = f"first {Ls} tokens, all heads, {reps} rep(s)"
    if "decode" in compact:
        w = inputs.WORKLOADS[DECODE]
        Bz, H, P, N, G = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
        st = inputs.decode_state(Bz, H, P, N, seed=0)
        prm = inputs.decode_params(H, seed=0)
        di = inputs.decode_step_inputs(0, Bz, H, P, N, G, io_dtype="bf16", seed=0)
        per, reps = _timed(lambda: oracle.ssd_decode(st, di["x"], di["dt"], prm["A"], di["B"], di["C"], prm["D"],
                                                     threads=thr), seconds)
        compact["decode"]["cpu"] = round(1.0 / per, 2)
        notes[DECODE] = f"one full step, {reps} rep(s)"
    for leg in compact.get("decode_layer", []):
        w = inputs.WORKLOADS[leg["w"].replace("layer_", "decode_layer_")]
        Bz, H, P, N, G, Wc = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["width"]
        prm = inputs.decode_layer_params(Bz, H, P, N, G, Wc, seed=0)
        li = inputs.decode_layer_step_inputs(0, Bz, H, P, N, G, io_dtype="bf16", seed=0)
        cst, sst = prm["conv_state"].copy(), prm["ssm_state"].copy()
        per, reps = _timed(lambda: oracle.decode_layer_step(cst, sst, li["xBC"], prm["conv_w"], prm["conv_b"],
                                                            li["dt"], prm["A"], prm["D"], li["z"], prm["norm_w"],
                                                            H, P, N, G, group=w["norm_group"]), seconds)
        leg["cpu"] = round(1.0 / per, 2)
        notes[leg["w"]] = f"one full layer step, {reps} rep(s)"
    if "mamba1" in compact:
        w = inputs.WORKLOADS[MAMBA1]
        Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
        ch = 64  # a 64-channel sample of the workload, same distributions
        d = inputs.diag_inputs(Bz, L, ch, N, io_dtype="bf16", seed=0)
        per, reps = _timed(lambda: oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=thr),
                           seconds)
        compact["mamba1"]["cpu"] = round(Bz * L / (per * Dm / ch), 1)
        notes[MAMBA1] = f"{ch} of {Dm} channels, all tokens, {reps} rep(s), scaled to all channels"
    if "mamba1_softplus" in compact:
        w = inputs.WORKLOADS[MAMBA1_SP]
        Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
        ch = 128
        d = inputs.diag_option_inputs(Bz, L, ch, N, io_dtype="bf16", seed=0, bias=False, z=False)
        per, reps = _timed(lambda: oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=thr,
                                                   delta_softplus=True), seconds)
        compact["mamba1_softplus"]["cpu"] = round(Bz * L / (per * Dm / ch), 1)
        notes[MAMBA1_SP] = f"{ch} of {Dm} channels, all tokens, {reps} rep(s), scaled to all channels"
    if "backward" in compact:
        (Bz, L, H), (P, N, G) = compact["backward"].get("shape", (1, 2048, 24)), (64, 128, 1)
        hs = 2
        d = inputs.ssd_inputs(Bz, L, hs, P, N, G, io_dtype="bf16", seed=0)
        dy = inputs.round_to(np.random.default_rng(1).standard_normal(d["x"].shape), "bf16")
        per, reps = _timed(lambda: oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"],
                                                      threads=thr), seconds)
        compact["backward"]["cpu"] = round(Bz * L / (per * H / hs), 1)
        notes["backward"] = f"{hs} of {H} heads (one host thread), all {L} tokens, {reps} rep(s), scaled to all heads"


def run_reference(args):
    """The oracle as the reference arm: same workload, metric and unit."""
    world, rank, _ = dist_env()
    if rank != 0:
        return  # rank 0 alone runs and prints
    import oracle
    from mamba_ssd_selective_gb300 import inputs
    w = inputs.WORKLOADS[args.workload or HEADLINE]
    K, W = args.steps, args.warmup
    threads = oracle.default_threads()
    budget = float(args.ref_budget_s)
    Ls = oracle_sample_tokens(w, budget / max(1, K + W), threads)
    d = inputs.ssd_inputs(w["batch"], Ls, w["nheads"], w["headdim"], w["dstate"], w["ngroups"], io_dtype="bf16",
                          seed=0)
    for _ in range(W):
        oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=threads)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=threads)
    el = time.perf_counter() - t0
    tokens = w["batch"] * Ls
    value = tokens * K / el
    sample = f"first {Ls} of {w['seqlen']} tokens of all {w['batch']} sequences per step, all {w['nheads']} heads, float64"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(el / K * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": args.workload or HEADLINE, "batch": w["batch"], "seqlen": w["seqlen"],
                   "nheads": w["nheads"], "headdim": w["headdim"], "dstate": w["dstate"], "ngroups": w["ngroups"],
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "cpu": host_cpu(), "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ chunk table

CT_CHUNKS = (64, 128, 256)
CT_BATCHES = (1, 2, 4, 8)
CT_LENGTHS = (512, 1024, 2048, 4096, 8192)
CT_HEADS = (24, 48, 80)


def run_chunk_table(args):
    """The fastest chunk size per shape over a grid of batch, length and head
    count (bf16, headdim 64, d_state 128, one group), each shape in a graph of
    back-to-back calls whose inputs rotate past L2 (random device tensors:
    timing only). Prints one JSON line per shape, then the C table of the
    static chunk policy (ssd_best_chunk) -- the pages' static-oracle /
    learned-table policy ("COREY ...", section 5.2)."""
    import torch
    from mamba_ssd_selective_gb300 import binding
    binding.load()
    dev, bf = torch.device("cuda"), torch.bfloat16
    P, N = 64, 128
    rows = []
    for H in CT_HEADS:
        for Bz in CT_BATCHES:
            for L in CT_LENGTHS:
                g = torch.Generator(device=dev).manual_seed(0)
                per = Bz * L * (2 * H * P + H + 2 * N) * 2
                nsets = max(2, math.ceil(3 * 129e6 / per))
                ws_max = max(binding.ssd_workspace_size(Bz, L, H, P, N, 1, bf, q) for q in CT_CHUNKS)
                A = -torch.exp(torch.rand(H, generator=g, device=dev) * math.log(16.0))
                Dv = torch.rand(H, generator=g, device=dev) + 0.5
                sets = []
                for _ in range(nsets):
                    sets.append(dict(
                        x=torch.randn(Bz, L, H, P, generator=g, device=dev).to(bf),
                        dt=torch.nn.functional.softplus(torch.randn(Bz, L, H, generator=g, device=dev) * 0.5 - 4).to(bf),
                        B=torch.randn(Bz, L, 1, N, generator=g, device=dev).to(bf),
                        C=torch.randn(Bz, L, 1, N, generator=g, device=dev).to(bf),
                        y=torch.empty(Bz, L, H, P, dtype=bf, device=dev), f=torch.empty(Bz, H, P, N, device=dev),
                        ws=torch.empty(ws_max, dtype=torch.uint8, device=dev)))
                us = {}
                for q in CT_CHUNKS:
                    def step(s):
                        binding.ssd_scan_chunked(s["x"], s["dt"], A, s["B"], s["C"], Dv, None, chunk_size=q,
                                                 y=s["y"], final_state=s["f"], workspace=s["ws"])
                    st = torch.cuda.Stream()
                    st.wait_stream(torch.cuda.current_stream())
                    with torch.cuda.stream(st):
                        for s in sets:
                            step(s)
                    st.synchronize()
                    steps = max(4, 2 * nsets)
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=st, capture_error_mode="relaxed"):
                        for i in range(steps):
                            step(sets[i % nsets])
                    for _ in range(2):
                        graph.replay()
                    ms, _ = graph_rep_stats(torch, graph, steps, reps=3)
                    us[q] = ms * 1e3
                    del graph
                del sets
                torch.cuda.empty_cache()
                best = min(us, key=us.get)
                rows.append({"batch": Bz, "seqlen": L, "nheads": H, "best": best,
                             "us": {str(q): round(v, 2) for q, v in us.items()}})
                print(json.dumps(rows[-1]), flush=True)
    print("// {batch, seqlen, nheads, best chunk}: measured by bench.py --chunk-table")
    print("const ChunkEntry kChunkTable[] = {")
    for r in rows:
        print(f"    {{{r['batch']}, {r['seqlen']}, {r['nheads']}, {r['best']}}},")
    print("};")


def run_profile_calls(args):
    """N plain calls of each selected leg's workload (prefill legs at chunk 128,
    the headline at its chunk argument or 128), no timing, for profiler launch
    lists; inputs as in the timed legs."""
    import torch
    from mamba_ssd_selective_gb300 import binding, inputs
    binding.load()
    dev = torch.device("cuda")
    bf = torch.bfloat16
    legs = set(args.legs.split(",")) if args.legs else set(LEGS)
    n = args.profile_calls

    def t_(a, dtype=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    names = ([HEADLINE] if "headline" in legs else []) + (list(PREFILL_LEGS) if "prefill" in legs else [])
    for nm in names:
        w = inputs.WORKLOADS[nm]
        d = inputs.ssd_inputs(w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                              io_dtype="bf16", seed=0)
        a = (t_(d["x"], bf), t_(d["dt"], bf), t_(d["A"]), t_(d["B"], bf), t_(d["C"], bf), t_(d["D"]))
        del d
        q = (args.chunk or 128) if nm == HEADLINE else 128
        for _ in range(n):
            binding.ssd_scan_chunked(*a, None, chunk_size=q)
        torch.cuda.synchronize()
        del a
    if "decode" in legs:
        w = inputs.WORKLOADS[DECODE]
        Bz, H, P, N, G = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
        st = t_(inputs.decode_state(Bz, H, P, N, seed=0))
        prm = inputs.decode_params(H, seed=0)
        for s in range(n):
            di = inputs.decode_step_inputs(s, Bz, H, P, N, G, io_dtype="bf16", seed=0)
            binding.ssd_decode_step(st, t_(di["x"], bf), t_(di["dt"], bf), t_(prm["A"]), t_(di["B"], bf),
                                    t_(di["C"], bf), t_(prm["D"]))
        torch.cuda.synchronize()
    if "decode_layer" in legs:
        w = inputs.WORKLOADS["decode_layer_B64_H80"]
        Bz, H, P, N, G, Wc = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["width"]
        prm = inputs.decode_layer_params(Bz, H, P, N, G, Wc, seed=0)
        li = inputs.decode_layer_step_inputs(0, Bz, H, P, N, G, io_dtype="bf16", seed=0)
        cst, sst = t_(prm["conv_state"]), t_(prm["ssm_state"])
        for _ in range(n):
            binding.decode_layer_step(t_(li["xBC"], bf), cst, t_(prm["conv_w"]), t_(prm["conv_b"]), t_(li["dt"], bf),
                                      t_(prm["A"]), t_(prm["D"]), sst, t_(li["z"], bf), t_(prm["norm_w"]),
                                      norm_group=w["norm_group"])
        torch.cuda.synchronize()
    if "mamba1" in legs:
        w = inputs.WORKLOADS[MAMBA1]
        d = inputs.diag_inputs(w["batch"], w["seqlen"], w["dim"], w["dstate"], io_dtype="bf16", seed=0)
        a = (t_(d["x"], bf), t_(d["dt"], bf), t_(d["A"]), t_(d["B"], bf), t_(d["C"], bf), t_(d["D"]))
        del d
        for _ in range(n):
            binding.selective_scan_diag(*a, None, chunk_size=w["chunk"])
        torch.cuda.synchronize()
        del a
    if "mamba1_softplus" in legs:
        w = inputs.WORKLOADS[MAMBA1_SP]
        d = inputs.diag_option_inputs(w["batch"], w["seqlen"], w["dim"], w["dstate"], io_dtype="bf16", seed=0,
                                      bias=False, z=False)
        a = (t_(d["x"], bf), t_(d["dt"], bf), t_(d["A"]), t_(d["B"], bf), t_(d["C"], bf), t_(d["D"]))
        for _ in range(n):
            binding.selective_scan_diag(*a, None, chunk_size=w["chunk"], delta_softplus=True)
        torch.cuda.synchronize()
    if "backward" in legs:
        Bz, L, H = bwd_shape(args)
        d = inputs.ssd_inputs(Bz, L, H, 64, 128, 1, io_dtype="bf16", seed=0)
        dy = inputs.round_to(np.random.default_rng(1).standard_normal(d["x"].shape), "bf16")
        a = (t_(d["x"], bf), t_(d["dt"], bf), t_(d["A"]), t_(d["B"], bf), t_(d["C"], bf), t_(dy, bf), t_(d["D"]))
        for _ in range(n):
            binding.ssd_scan_chunked_bwd(*a)
        torch.cuda.synchronize()
    print(json.dumps({"profile_calls": n, "legs": sorted(legs)}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--chunk", type=int, default=0, help="force the headline's chunk size (default: best of 64/128/256)")
    ap.add_argument("--legs", default=None, help=f"comma-separated subset of {','.join(LEGS)} (default: all)")
    ap.add_argument("--bwd-shape", default=None, help="B,L,H of the backward leg (default 1,2048,24; P 64, N 128)")
    ap.add_argument("--workload", default=None, help="reference arm: workload name (default: the headline)")
    ap.add_argument("--ref-budget-s", type=float, default=60.0, help="reference arm: total oracle seconds")
    ap.add_argument("--skip-extra", action="store_true", help="the headline leg only")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU oracle baselines")
    ap.add_argument("--chunk-table", action="store_true", help="measure the chunk-policy table and print it")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="make this many plain calls of each selected leg's workload (for profiler launch lists)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3  # at least three warm-up steps
    if args.legs:
        bad = set(args.legs.split(",")) - set(LEGS)
        if bad:
            ap.error(f"unknown legs: {sorted(bad)}")
    if args.chunk_table:
        run_chunk_table(args)
    elif args.profile_calls > 0:
        run_profile_calls(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    world, _, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
