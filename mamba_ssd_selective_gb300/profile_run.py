"""Runs workloads of the library eagerly, a few calls each, for profiler
launch lists (ncu) of their kernels; timing-free and output-free.

    python -m mamba_ssd_selective_gb300.profile_run [--calls K] [names...]

Names: decode_layer (B64 H80 P64 N128, width-4 conv, norm over all channels),
mamba1_softplus (B1 L4096 D1024 N16 with delta_softplus: time segments),
backward (SSD backward, B1 L2048 H24 P64 N128), mamba1 (B8 L2048 D5120 N16),
prefill (B1 L4096 H24 P64 N128, chunk 128). Inputs are the seeded synthetic
workloads of `inputs`.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import binding, inputs


def _t(a, dtype=torch.float32):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def decode_layer(calls):
    Bz, H, P, N, G, W = 64, 80, 64, 128, 1, 4
    prm = inputs.decode_layer_params(Bz, H, P, N, G, W, seed=0)
    li = inputs.decode_layer_step_inputs(0, Bz, H, P, N, G, io_dtype="bf16", seed=0)
    bf = torch.bfloat16
    xBC, dt, z = _t(li["xBC"], bf), _t(li["dt"], bf), _t(li["z"], bf)
    consts = (_t(prm["conv_w"]), _t(prm["conv_b"]))
    A, D, nw = _t(prm["A"]), _t(prm["D"]), _t(prm["norm_w"])
    cst, sst = _t(prm["conv_state"]), _t(prm["ssm_state"])
    for _ in range(calls):
        binding.decode_layer_step(xBC, cst, *consts, dt, A, D, sst, z, nw, norm_group=H * P)


def mamba1_softplus(calls):
    w = inputs.WORKLOADS["mamba1_B1_L4096_D1024_softplus"]
    d = inputs.diag_option_inputs(w["batch"], w["seqlen"], w["dim"], w["dstate"], io_dtype="bf16", seed=0,
                                  bias=False, z=False)
    bf = torch.bfloat16
    args = (_t(d["x"], bf), _t(d["dt"], bf), _t(d["A"]), _t(d["B"], bf), _t(d["C"], bf), _t(d["D"]))
    for _ in range(calls):
        binding.selective_scan_diag(*args, None, chunk_size=w["chunk"], delta_softplus=True)


def mamba1(calls):
    w = inputs.WORKLOADS["mamba1_B8_L2048_D5120"]
    d = inputs.diag_inputs(w["batch"], w["seqlen"], w["dim"], w["dstate"], io_dtype="bf16", seed=0)
    bf = torch.bfloat16
    args = (_t(d["x"], bf), _t(d["dt"], bf), _t(d["A"]), _t(d["B"], bf), _t(d["C"], bf), _t(d["D"]))
    for _ in range(calls):
        binding.selective_scan_diag(*args, None, chunk_size=w["chunk"])


def backward(calls):
    d = inputs.ssd_inputs(1, 2048, 24, 64, 128, 1, io_dtype="bf16", seed=0)
    dy = inputs.round_to(np.random.default_rng(1).standard_normal(d["x"].shape), "bf16")
    bf = torch.bfloat16
    args = (_t(d["x"], bf), _t(d["dt"], bf), _t(d["A"]), _t(d["B"], bf), _t(d["C"], bf), _t(dy, bf), _t(d["D"]))
    for _ in range(calls):
        binding.ssd_scan_chunked_bwd(*args)


def prefill(calls):
    w = inputs.WORKLOADS["ssd_m2_130m_L4096"]
    d = inputs.ssd_inputs(w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                          io_dtype="bf16", seed=0)
    bf = torch.bfloat16
    args = (_t(d["x"], bf), _t(d["dt"], bf), _t(d["A"]), _t(d["B"], bf), _t(d["C"], bf), _t(d["D"]))
    for _ in range(calls):
        binding.ssd_scan_chunked(*args, None, chunk_size=128)


RUNS = {"decode_layer": decode_layer, "mamba1_softplus": mamba1_softplus, "backward": backward, "mamba1": mamba1,
        "prefill": prefill}


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("names", nargs="*", default=["decode_layer", "mamba1_softplus", "backward"])
    ap.add_argument("--calls", type=int, default=2)
    args = ap.parse_args()
    binding.load()
    for name in args.names:
        RUNS[name](args.calls)
        torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
