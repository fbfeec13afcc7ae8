#!/usr/bin/env python
"""Throughput benchmark of the SSD selective scan on one GB300 (or N replicas).

One step = one chunked SSD prefill (chunk state -> state passing -> chunk scan,
with the in-chunk cumulative sums fused into both chunk kernels) of the
Mamba-2-130M-shaped layer workload: batch 1, L 4096, 24 heads, headdim 64,
d_state 128, 1 group, bf16 x/dt/B/C/y with float32 state and accumulation,
seeded synthetic inputs. The timed region replays a CUDA graph of exactly K
steps; the steps rotate over copies of the inputs whose total size exceeds
the L2 cache, so every step reads its inputs from HBM.

The same JSON line also carries, each in its own timed region: the decode
workload (batch 64, 80 heads, 64 x 128 fp32 state, 1000 in-place steps, one
CUDA graph), the Mamba-1 diagonal scan (batch 8, L 2048, 5120 channels,
d_state 16, chunk sweep), the per-stage kernel times, the end-to-end number
through the C ABI with host buffers, and the float64 CPU oracle timed on the
host cores.

`--impl reference` times the float64 CPU oracle on the same workload (a
bounded sample of tokens per step) and prints the same kind of line.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU (weak
scaling, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "ssd_m2_130m_L4096"
DECODE = "decode_B64_H80"
MAMBA1 = "mamba1_B8_L2048_D5120"
MAMBA1_SP = "mamba1_B1_L4096_D1024_softplus"
METRIC = "SSD prefill tokens/s + % roofline; decode steps/s + state HBM GB/s"
STAGES = ("chunk_state", "state_pass", "chunk_scan")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


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
    return b["x"] + b["dt"] + b["B"] + b["C"] + b["y"]


def ssd_flops(w: dict, Q: int) -> float:
    """Useful flops (causal MACs x2 of intra-chunk, chunk-state and output
    contractions, C.B^T once per group)."""
    Bz, L, H, P, N, G = w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    return float(Bz * L * (H * (Q * P + 4 * N * P) + G * Q * N))


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


# -------------------------------------------------------------- our arm

def _traffic_for(kernel: str):
    """ncu DRAM bytes per launch recorded in profiles/traffic.json, only if the
    kernel's source is unchanged since the capture; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "mamba_ssd_selective_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or file_hash(src) != rec.get("source_hash"):
        return None
    return rec.get("bytes_per_launch")


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
    bf = torch.bfloat16
    K, W = args.steps, args.warmup
    out = {}

    sampler = ClockSampler(local).start() if rank == 0 else None

    # ---------------- prefill (headline)
    w = dict(inputs.WORKLOADS[HEADLINE])
    d = inputs.ssd_inputs(w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                          io_dtype="bf16", seed=0)

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    base = {"x": t_(d["x"], bf), "dt": t_(d["dt"], bf), "B": t_(d["B"], bf), "C": t_(d["C"], bf)}
    A, Dv = t_(d["A"]), t_(d["D"])
    Bz, L, H, P, N, G = w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    ws_max = max(binding.ssd_workspace_size(Bz, L, H, P, N, G, bf, q) for q in (64, 128, 256))
    per_set = sum(v.numel() * v.element_size() for v in base.values()) * 2 + ws_max + Bz * H * P * N * 4
    n_sets = max(2, math.ceil(3 * l2 / per_set))
    sets = []
    for _ in range(n_sets):
        s = {k: v.clone() for k, v in base.items()}
        s["y"] = torch.empty_like(base["x"])
        s["final"] = torch.empty((Bz, H, P, N), dtype=torch.float32, device=dev)
        s["ws"] = torch.empty(ws_max, dtype=torch.uint8, device=dev)
        sets.append(s)

    def step(s, q):
        binding.ssd_scan_chunked(s["x"], s["dt"], A, s["B"], s["C"], Dv, None, chunk_size=q, y=s["y"],
                                 final_state=s["final"], workspace=s["ws"])

    def capture(nsteps, q, stage_events=None):
        g = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream(device=dev)
        stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(stream):
            for i in range(min(nsteps, n_sets)):  # eager warm-up on the capture stream
                step(sets[i % n_sets], q)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for i in range(nsteps):
                if stage_events is not None:
                    binding.ssd_record_stage_events(stage_events[i])
                step(sets[i % n_sets], q)
        return g

    def time_graph(g, reps=1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    # chunk sweep: the best static chunk per workload is the one reported
    sweep = {}
    S = 8 * n_sets
    for q in (64, 128, 256):
        g = capture(S, q)
        for _ in range(max(W, 3)):
            g.replay()
        ms = time_graph(g, reps=5) / (5 * S)
        sweep[q] = ms
        del g
    best_q = args.chunk or min(sweep, key=sweep.get)

    # the timed region: exactly K steps in one graph
    g = capture(K, best_q)
    gw = capture(max(W, 3), best_q)
    for _ in range(2):
        gw.replay()
    # keep the GPU busy ~1 s before the timed region so that the clock samples
    # describe the clocks under this load
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

    # per-stage kernel times, CUDA events between the stages of every step of a
    # second K'-step graph of the same workload
    Ks = min(K, 256)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Ks)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize(dev)
    gs = capture(Ks, best_q, stage_events=evs)
    gs.replay()
    torch.cuda.synchronize(dev)
    stage_ms = {nm: statistics.mean(r[i].elapsed_time(r[i + 1]) for r in evs) for i, nm in enumerate(STAGES)}
    del gs
    dom = max(stage_ms, key=stage_ms.get)
    dom_bytes = stage_algorithmic_bytes(w, dom)
    achieved = dom_bytes / (stage_ms[dom] / 1e3) / 1e9
    comp = ssd_compulsory_bytes(w)
    src_of = {"chunk_state": "chunked_tc.cu", "state_pass": "chunked_simt.cu", "chunk_scan": "chunked_tc.cu"}
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "traffic": _traffic_for(dom), "algorithmic_bytes": dom_bytes,
                "launch_ms": round(stage_ms[dom], 5), "peak_source": peaks["source"]}
    step_gbs = comp["total"] / (ms_step / 1e3) / 1e9
    out["prefill"] = {
        "step_roofline": {"bound": "hbm", "compulsory_bytes": comp["total"], "achieved": round(step_gbs, 1),
                          "peak": hbm_peak, "unit": "GB/s", "frac": round(step_gbs / hbm_peak, 4)},
        "tflops": round(ssd_flops(w, best_q) / (ms_step / 1e3) / 1e12, 2),
        "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
        "chunk_sweep_ms_per_step": {str(k): round(v, 5) for k, v in sweep.items()},
        "chunk_policy": binding.ssd_best_chunk(Bz, L, H, P, N, G, torch.bfloat16),
    }

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its inputs from pinned host memory and its results
    # (y and the final state) back, as a serving loop would: the inputs of a
    # step are one packed host buffer (one copy in), its outputs one packed
    # device buffer (one copy out), and three streams overlap the copy in of
    # step i + 1, the scan of step i and the copy out of step i - 1 over two
    # device buffer sets.
    in_parts = [("x", base["x"]), ("dt", base["dt"]), ("B", base["B"]), ("C", base["C"]), ("A", A), ("D", Dv)]

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
                      "ws": torch.empty(ws_max, dtype=torch.uint8, device=dev)})
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
            binding.ssd_scan_chunked(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], None, chunk_size=best_q,
                                     y=o["y"], final_state=o["final"], workspace=d["ws"], stream=s_run)
            ev["run"][i & 1].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["run"][i & 1])
            hout.copy_(d["dout"], non_blocking=True)
            ev["out"][i & 1].record(s_out)

    def capture_e2e(nsteps):
        # K steps in one graph: s_cap forks to the three stage streams and joins them
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
    del ge
    h2d = sum(t.numel() * t.element_size() for _, t in in_parts)
    d2h = sum(t.numel() * t.element_size() for _, t in out_parts)
    e2e = {"value": world * tokens * Ke / (ms_e2e / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": Ke,
           "pipeline": "packed pinned buffers; copy in / scan / copy out overlapped on three streams; K steps in "
                       "one CUDA graph"}
    del sets, dsets

    # ---------------- decode workload
    if not args.skip_extra:
        out["decode"] = bench_decode(torch, binding, inputs, dev, hbm_peak, peaks["source"], W)
        out["decode_layer"] = [bench_decode_layer(torch, binding, inputs, dev, hbm_peak, name, W)
                               for name in ("decode_layer_B64_H80", "decode_layer_B1_H128_G8")]
        out["mamba1"] = bench_mamba1(torch, binding, inputs, dev, hbm_peak, peaks["source"], K, W)
        out["mamba1_softplus"] = bench_mamba1_softplus(torch, binding, inputs, dev, hbm_peak, K, W)
        out["backward"] = bench_backward(torch, binding, inputs, dev, hbm_peak, W)

    clocks = sampler.stop() if sampler else None

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded: x,B,C~N(0,1); dt=softplus(N(0,.5)+b), A=-exp(U(0,ln16)))",
        "config": {"workload": HEADLINE, "batch": Bz, "seqlen": L, "nheads": H, "headdim": P, "dstate": N,
                   "ngroups": G, "chunk": best_q, "io": "bf16 x/dt/B/C/y, fp32 state and accumulation",
                   "l2": f"inputs rotate over {n_sets} copies ({n_sets * per_set / 2**20:.0f} MiB > L2 "
                         f"{l2 / 2**20:.0f} MiB)", "graph": "K steps in one CUDA graph",
                   "parallelism": "replicas" if world == 1 else f"replicas x{world}"},
        "roofline": roofline,
        "gpu_launches": 3 * K,
        "e2e": e2e,
    }
    if not args.skip_cpu and not args.skip_extra:
        oracle_beside(out)
    line.update(out)
    if not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(w)
    if clocks is not None:
        line["clocks"] = clocks
    print(json.dumps(line), flush=True)


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
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        e0.record()
        for _ in range(reps):
            graph.launch()
        e1.record()
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / (reps * steps)
    finally:
        graph.close()
    nbytes = (2 * Bz * H * P * N * 4 + 2 * Bz * Cc * Wc * 4 + Bz * Cc * 2 + Cc * Wc * 4 + Cc * 4
              + Bz * H * 2 + 2 * Bz * H * P * 2 + H * P * 4 + 2 * H * 4)
    gbs = nbytes / (us / 1e6) / 1e9
    return {"workload": name, "us_per_step": round(us, 3), "steps_per_s": round(1e6 / us, 1),
            "kernels_per_step": 3, "gpu_launches": 3 * steps * reps, "algorithmic_bytes_per_step": nbytes,
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
            "graph": f"{steps} steps captured by ssd_decode_graph_create, one launch"}


def bench_decode(torch, binding, inputs, dev, hbm_peak, peak_src, W):
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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    state_bytes = 2 * Bz * H * P * N * 4
    step_bytes = state_bytes + Bz * H * P * 2 * 2 + Bz * H * 2 + 2 * Bz * G * N * 2
    gbs = step_bytes / (ms / 1e3) / 1e9
    return {"workload": DECODE, "steps": steps, "ms_per_step": round(ms, 6), "steps_per_s": round(1e3 / ms, 1),
            "state_gbs": round(state_bytes / (ms / 1e3) / 1e9, 1), "gpu_launches": steps,
            "roofline": {"bound": "hbm", "kernel": "decode_step", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "algorithmic_bytes": step_bytes,
                         "traffic": _traffic_for("decode_step"), "frac_of_8tbs": round(gbs / 8000.0, 4),
                         "peak_source": peak_src}}


def bench_mamba1(torch, binding, inputs, dev, hbm_peak, peak_src, K, W):
    w = inputs.WORKLOADS[MAMBA1]
    Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
    bf = torch.bfloat16
    d = inputs.diag_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=0)

    def t_(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype)

    x, dt, Bm, Cm = t_(d["x"], bf), t_(d["dt"], bf), t_(d["B"], bf), t_(d["C"], bf)
    A, Dv = t_(d["A"]), t_(d["D"])
    y = torch.empty_like(x)
    hT = torch.empty((Bz, Dm, N), dtype=torch.float32, device=dev)
    reps = max(5, min(K, 50))
    sweep = {}
    for chunk in (256, 512, 1024, 2048):
        for _ in range(max(W, 3)):
            binding.selective_scan_diag(x, dt, A, Bm, Cm, Dv, None, chunk_size=chunk, y=y, final_state=hT)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            binding.selective_scan_diag(x, dt, A, Bm, Cm, Dv, None, chunk_size=chunk, y=y, final_state=hT)
        e1.record()
        torch.cuda.synchronize(dev)
        sweep[chunk] = e0.elapsed_time(e1) / reps
    best = min(sweep, key=sweep.get)
    ms = sweep[best]
    nbytes = 3 * Bz * L * Dm * 2 + 2 * Bz * L * N * 2 + Dm * N * 4 + Dm * 4 + Bz * Dm * N * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    n_exp = Bz * L * Dm * N
    return {"workload": MAMBA1, "chunk": best, "ms": round(ms, 5), "tokens_per_s": round(Bz * L / (ms / 1e3), 1),
            "chunk_sweep_ms": {str(k): round(v, 5) for k, v in sweep.items()},
            "exp_per_s": round(n_exp / (ms / 1e3), 1), "gpu_launches": reps,
            "roofline": {"bound": "hbm", "kernel": "diag_scan", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "algorithmic_bytes": nbytes,
                         "traffic": _traffic_for("diag_scan"), "peak_source": peak_src}}


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
    reps = max(8, min(K, 200))
    ws_bytes = binding.selective_scan_diag_workspace_size(Bz, L, Dm, N, bf)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    launches = 3 if ws_bytes else 1   # segment-local scan, segment pass, output scan

    def run(i, chunk):
        s_ = sets[i % n_sets]
        binding.selective_scan_diag(s_["x"], s_["dt"], A, s_["B"], s_["C"], Dv, None, chunk_size=chunk, y=s_["y"],
                                    final_state=hT, delta_softplus=True, workspace=ws)

    sweep = {}
    for chunk in (256, 2048):
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
    ms = sweep[best]
    nbytes = 3 * Bz * L * Dm * 2 + 2 * Bz * L * N * 2 + Dm * N * 4 + Dm * 4 + Bz * Dm * N * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": MAMBA1_SP, "chunk": best, "ms": round(ms, 5),
            "tokens_per_s": round(Bz * L / (ms / 1e3), 1),
            "chunk_sweep_ms": {str(k): round(v, 5) for k, v in sweep.items()}, "gpu_launches": reps * launches,
            "time_segments": ws_bytes > 0,
            "l2": f"inputs rotate over {n_sets} copies", "hbm_frac": round(gbs / hbm_peak, 4),
            "pages_time_ms": {"value": 0.3204, "hardware": "RTX 3070, fp16, selective_scan_fn, delta_softplus"}}


def bench_backward(torch, binding, inputs, dev, hbm_peak, W):
    """SSD backward (recompute, adjoint states, per-chunk gradients) on the
    130M-shaped layer at L 2048, bf16 inputs, float32 gradients; input copies
    rotate past L2."""
    Bz, L, H, P, N, G = 1, 2048, 24, 64, 128, 1
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
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        run(i)
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / reps
    # compulsory bytes: x, dt, B, C, dy read (bf16); dx, ddt, dB, dC written (float32)
    nbytes = Bz * L * (2 * H * P + H + 2 * G * N) * 2 + Bz * L * (H * P + H + 2 * G * N) * 4
    return {"workload": "ssd_bwd_m2_130m_L2048", "ms": round(ms, 4), "tokens_per_s": round(Bz * L / (ms / 1e3), 1),
            "kernels_per_call": 6, "gpu_launches": 6 * reps, "hbm_frac": round(nbytes / (ms / 1e3) / 1e9 / hbm_peak, 4),
            "arith": "float32 CUDA cores, chunks of 64", "l2": f"inputs rotate over {n_sets} copies",
            "pages_context": "Table 13 (L40S): whole-model forward + backward, not comparable"}


# ------------------------------------------------------------ CPU oracle

def oracle_sample_tokens(w: dict, seconds: float, threads: int) -> int:
    """Tokens of the workload (from the start of the sequence, all heads) the
    oracle processes in about `seconds`, measured on a short probe run."""
    import oracle
    from mamba_ssd_selective_gb300 import inputs
    probe = min(256, w["seqlen"])
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
    Ls = oracle_sample_tokens(w, seconds, threads)
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
            "sample": f"first {Ls} of {w['seqlen']} tokens, all {w['nheads']} heads, float64 token-by-token "
                      f"recurrence, {reps} repetition(s) in {el:.2f} s"}


def _timed(fn, seconds):
    """Seconds per call of fn, repeated for about `seconds` (at least once)."""
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            return el / reps, reps


def oracle_beside(out: dict, seconds: float = 2.0) -> None:
    """The float64 oracle, as it stands, timed on the host cores beside each
    extra leg on a bounded sample of its workload, in the leg's own unit."""
    import oracle
    from mamba_ssd_selective_gb300 import inputs
    thr = oracle.default_threads()

    def rec(value, unit, sample):
        return {"value": round(value, 2), "unit": unit, "cores": thr, "kind": "oracle", "sample": sample}

    if "decode" in out:
        w = inputs.WORKLOADS[DECODE]
        Bz, H, P, N, G = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
        st = inputs.decode_state(Bz, H, P, N, seed=0)
        prm = inputs.decode_params(H, seed=0)
        di = inputs.decode_step_inputs(0, Bz, H, P, N, G, io_dtype="bf16", seed=0)
        per, reps = _timed(lambda: oracle.ssd_decode(st, di["x"], di["dt"], prm["A"], di["B"], di["C"], prm["D"],
                                                     threads=thr), seconds)
        out["decode"]["oracle"] = rec(1.0 / per, "steps/s", f"one full step, {reps} repetition(s)")
    for leg in out.get("decode_layer", []):
        w = inputs.WORKLOADS[leg["workload"]]
        Bz, H, P, N, G, Wc = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["width"]
        prm = inputs.decode_layer_params(Bz, H, P, N, G, Wc, seed=0)
        li = inputs.decode_layer_step_inputs(0, Bz, H, P, N, G, io_dtype="bf16", seed=0)
        cst, sst = prm["conv_state"].copy(), prm["ssm_state"].copy()
        per, reps = _timed(lambda: oracle.decode_layer_step(cst, sst, li["xBC"], prm["conv_w"], prm["conv_b"],
                                                            li["dt"], prm["A"], prm["D"], li["z"], prm["norm_w"],
                                                            H, P, N, G, group=w["norm_group"]), seconds)
        leg["oracle"] = rec(1.0 / per, "steps/s", f"one full layer step, {reps} repetition(s)")
    if "mamba1" in out:
        w = inputs.WORKLOADS[MAMBA1]
        Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
        ch = 64  # a 64-channel sample of the workload, same distributions
        d = inputs.diag_inputs(Bz, L, ch, N, io_dtype="bf16", seed=0)
        per, reps = _timed(lambda: oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=thr),
                           seconds)
        out["mamba1"]["oracle"] = rec(Bz * L / (per * Dm / ch), "tokens/s",
                                      f"{ch} of {Dm} channels, all {Bz}x{L} tokens, {reps} repetition(s), "
                                      f"scaled to all channels")
    if "mamba1_softplus" in out:
        w = inputs.WORKLOADS[MAMBA1_SP]
        Bz, L, Dm, N = w["batch"], w["seqlen"], w["dim"], w["dstate"]
        ch = 128  # a 128-channel sample of the workload, same distributions
        d = inputs.diag_option_inputs(Bz, L, ch, N, io_dtype="bf16", seed=0, bias=False, z=False)
        per, reps = _timed(lambda: oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], threads=thr,
                                                   delta_softplus=True), seconds)
        out["mamba1_softplus"]["oracle"] = rec(Bz * L / (per * Dm / ch), "tokens/s",
                                               f"{ch} of {Dm} channels, all tokens, {reps} repetition(s), "
                                               f"scaled to all channels")
    if "backward" in out:
        Bz, L, H, P, N, G = 1, 2048, 24, 64, 128, 1
        hs = 2
        d = inputs.ssd_inputs(Bz, L, hs, P, N, G, io_dtype="bf16", seed=0)
        dy = inputs.round_to(np.random.default_rng(1).standard_normal(d["x"].shape), "bf16")
        per, reps = _timed(lambda: oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"],
                                                      threads=thr), seconds)
        out["backward"]["oracle"] = rec(Bz * L / (per * H / hs), "tokens/s",
                                        f"{hs} of {H} heads (one B/C group, so one host thread), all {L} tokens, "
                                        f"{reps} repetition(s), scaled to all heads")


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
    sample = f"first {Ls} of {w['seqlen']} tokens per step, all {w['nheads']} heads, float64"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(el / K * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": args.workload or HEADLINE, "batch": w["batch"], "seqlen": w["seqlen"],
                   "nheads": w["nheads"], "headdim": w["headdim"], "dstate": w["dstate"], "ngroups": w["ngroups"],
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--chunk", type=int, default=0, help="force a chunk size (default: best of 64/128/256)")
    ap.add_argument("--workload", default=None, help="reference arm: workload name (default: the headline)")
    ap.add_argument("--ref-budget-s", type=float, default=60.0, help="reference arm: total oracle seconds")
    ap.add_argument("--skip-extra", action="store_true", help="skip the decode and Mamba-1 lines")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3  # at least three warm-up steps
    if args.impl == "reference":
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
