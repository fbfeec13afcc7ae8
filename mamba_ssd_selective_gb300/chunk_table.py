"""Measures the fastest SSD prefill chunk size per shape on this GPU.

`python -m mamba_ssd_selective_gb300.chunk_table` times ssd_scan_chunked
(bf16, P = 64, N = 128, one B/C group) at chunk sizes 64, 128 and 256 over a
grid of batch, sequence length and head count, each shape in a CUDA graph of
steps whose inputs rotate past the L2 cache, and prints the measurements as
JSON plus the C table that ssd_best_chunk() (csrc/chunk_policy.cu) is built
from. Timing only: the inputs are random device tensors.

The pages pick chunk sizes by measuring a static sweep and keeping the best
per regime (the static-oracle and learned-table policies of "COREY ...",
section 5.2); this is that table for the tensor-core path on GB300.
"""
from __future__ import annotations

import argparse
import json
import math

import torch

from . import binding

CHUNKS = (64, 128, 256)
BATCHES = (1, 2, 4, 8)
LENGTHS = (512, 1024, 2048, 4096, 8192)
HEADS = (24, 48, 80)
P, N = 64, 128


def time_shape(Bz: int, L: int, H: int, reps: int = 3) -> dict:
    dev, bf = torch.device("cuda"), torch.bfloat16
    g = torch.Generator(device=dev).manual_seed(0)
    per = Bz * L * (2 * H * P + H + 2 * N) * 2
    nsets = max(2, math.ceil(3 * 129e6 / per))
    ws_max = max(binding.ssd_workspace_size(Bz, L, H, P, N, 1, bf, q) for q in CHUNKS)
    A = -torch.exp(torch.rand(H, generator=g, device=dev) * math.log(16.0))
    Dv = torch.rand(H, generator=g, device=dev) + 0.5
    sets = []
    for _ in range(nsets):
        s = dict(x=torch.randn(Bz, L, H, P, generator=g, device=dev).to(bf),
                 dt=torch.nn.functional.softplus(torch.randn(Bz, L, H, generator=g, device=dev) * 0.5 - 4).to(bf),
                 B=torch.randn(Bz, L, 1, N, generator=g, device=dev).to(bf),
                 C=torch.randn(Bz, L, 1, N, generator=g, device=dev).to(bf))
        s["y"] = torch.empty_like(s["x"])
        s["f"] = torch.empty(Bz, H, P, N, device=dev)
        s["ws"] = torch.empty(ws_max, dtype=torch.uint8, device=dev)
        sets.append(s)
    out = {}
    for q in CHUNKS:
        def step(s):
            binding.ssd_scan_chunked(s["x"], s["dt"], A, s["B"], s["C"], Dv, None, chunk_size=q, y=s["y"],
                                     final_state=s["f"], workspace=s["ws"])
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
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        out[q] = e0.elapsed_time(e1) * 1e3 / (reps * steps)
        del graph
    del sets
    torch.cuda.empty_cache()
    return out


def c_table(rows: list) -> str:
    lines = ["// {batch, seqlen, nheads, best chunk}: measured by mamba_ssd_selective_gb300.chunk_table",
             "const ChunkEntry kChunkTable[] = {"]
    for r in rows:
        lines.append(f"    {{{r['batch']}, {r['seqlen']}, {r['nheads']}, {r['best']}}},")
    lines.append("};")
    return "\n".join(lines)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--out", default=None, help="also write the JSON here")
    args = ap.parse_args()
    binding.load()
    rows = []
    for H in HEADS:
        for Bz in BATCHES:
            for L in LENGTHS:
                us = time_shape(Bz, L, H)
                best = min(us, key=us.get)
                rows.append({"batch": Bz, "seqlen": L, "nheads": H, "best": best,
                             "us": {str(q): round(v, 2) for q, v in us.items()}})
                print(json.dumps(rows[-1]), flush=True)
    if args.out:
        with open(args.out, "w") as f:
            json.dump(rows, f, indent=1)
    print(c_table(rows))


if __name__ == "__main__":
    main()
