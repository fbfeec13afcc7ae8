"""Seeded synthetic inputs for the SSD selective scan, its decode step and the
Mamba-1 diagonal scan.

This module draws random tensors only. It holds none of the scan's arithmetic:
no decay, no recurrence, no contraction. Both the CUDA path (through the tests
and ``bench.py``) and the float64 CPU oracle take their inputs from here, so
that each side sees exactly the same values.

Value distributions (the workloads of the Mamba-2 SSD pages, "Compiler-First
State Space Duality ..." and the COREY Mamba-1 benchmarks):

* ``x ~ N(0, 1)``; ``B, C ~ N(0, 1)``.
* ``dt``: per head (per channel for Mamba-1) a target step ``dt0`` is drawn
  log-uniform in ``[1e-3, 1e-1]``; its softplus inverse is the bias ``b``; per
  token ``dt = softplus(eps + b)`` with ``eps ~ N(0, 0.5)`` (0.5 read as a
  standard deviation).
* ``A_h = -exp(U(log 1, log 16))`` per head; Mamba-1 uses ``A[d, n] = -(n+1)``.
* ``D ~ U(0.5, 1.5)`` per head (per channel for Mamba-1).
* decode state ``~ N(0, 0.1)`` (0.1 read as a standard deviation).

Every tensor comes from its own PCG64 stream keyed by ``(seed, stream id)``,
so a tensor does not depend on which others were drawn. Values are generated
in float64 and rounded once to the I/O dtype (``"bf16"`` or ``"f32"``); the
arrays returned are float64 and hold exactly the rounded values, which is
what the oracle consumes. ``A``, ``D`` and states are always float32 values.
"""
from __future__ import annotations

import numpy as np

# stream ids, fixed forever: changing one changes every seeded workload
_S_X, _S_DT_NOISE, _S_DT0, _S_A, _S_B, _S_C, _S_D, _S_STATE = 1, 2, 3, 4, 5, 6, 7, 8
_S_Z = 9
_S_CONV_W, _S_CONV_B, _S_NORM_W, _S_CONV_STATE = 10, 11, 12, 13
_S_LAYER_BASE = 100000  # decode-layer step s uses streams _S_LAYER_BASE + 4*s + k
_S_DECODE_BASE = 1000  # decode step s uses streams _S_DECODE_BASE + 8*s + k


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def round_to(a: np.ndarray, io_dtype: str) -> np.ndarray:
    """Round float64 values to the I/O dtype and widen back exactly to float64.

    bf16 rounding is round-to-nearest-even of the float32 bit pattern
    (float64 -> float32 -> bfloat16); NaN/Inf never occur in these inputs.
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    if io_dtype == "f32":
        return f.astype(np.float64)
    if io_dtype != "bf16":
        raise ValueError(f"io_dtype must be 'f32' or 'bf16', got {io_dtype!r}")
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, z)


def _dt_bias(rng: np.random.Generator, n: int, dt_min=1e-3, dt_max=1e-1) -> np.ndarray:
    """Bias whose softplus is a log-uniform target step in [dt_min, dt_max]."""
    dt0 = np.exp(rng.uniform(np.log(dt_min), np.log(dt_max), size=n))
    return dt0 + np.log(-np.expm1(-dt0))  # softplus^{-1}(dt0)


def _dt(seed: int, shape, nchan: int, noise_stream: int, io_dtype: str) -> np.ndarray:
    bias = _dt_bias(_rng(seed, _S_DT0), nchan)
    eps = _rng(seed, noise_stream).normal(0.0, 0.5, size=shape)
    return round_to(_softplus(eps + bias), io_dtype)


def ssd_inputs(batch: int, seqlen: int, nheads: int, headdim: int, dstate: int,
               ngroups: int = 1, io_dtype: str = "bf16", seed: int = 0,
               init_state: bool = False) -> dict:
    """Inputs of one SSD prefill: x[B,L,H,P], dt[B,L,H], A[H], B/C[B,L,G,N],
    D[H], init_state[B,H,P,N] (or None)."""
    Bsz, L, H, P, N, G = batch, seqlen, nheads, headdim, dstate, ngroups
    out = {
        "x": round_to(_rng(seed, _S_X).standard_normal((Bsz, L, H, P)), io_dtype),
        "dt": _dt(seed, (Bsz, L, H), H, _S_DT_NOISE, io_dtype),
        "A": round_to(-np.exp(_rng(seed, _S_A).uniform(np.log(1.0), np.log(16.0), size=H)), "f32"),
        "B": round_to(_rng(seed, _S_B).standard_normal((Bsz, L, G, N)), io_dtype),
        "C": round_to(_rng(seed, _S_C).standard_normal((Bsz, L, G, N)), io_dtype),
        "D": round_to(_rng(seed, _S_D).uniform(0.5, 1.5, size=H), "f32"),
        "init_state": None,
    }
    if init_state:
        out["init_state"] = round_to(_rng(seed, _S_STATE).normal(0.0, 0.1, size=(Bsz, H, P, N)), "f32")
    return out


def decode_state(batch: int, nheads: int, headdim: int, dstate: int, seed: int = 0) -> np.ndarray:
    """Initial decode state [B,H,P,N], float32 values ~ N(0, 0.1)."""
    return round_to(_rng(seed, _S_STATE).normal(0.0, 0.1, size=(batch, nheads, headdim, dstate)), "f32")


def decode_params(nheads: int, seed: int = 0) -> dict:
    """Per-head constants of the decode workload: A[H], D[H]."""
    return {
        "A": round_to(-np.exp(_rng(seed, _S_A).uniform(np.log(1.0), np.log(16.0), size=nheads)), "f32"),
        "D": round_to(_rng(seed, _S_D).uniform(0.5, 1.5, size=nheads), "f32"),
    }


def decode_step_inputs(step: int, batch: int, nheads: int, headdim: int, dstate: int,
                       ngroups: int = 1, io_dtype: str = "bf16", seed: int = 0) -> dict:
    """Per-token inputs of decode step ``step``: x[B,H,P], dt[B,H], B/C[B,G,N]."""
    base = _S_DECODE_BASE + 8 * int(step)
    return {
        "x": round_to(_rng(seed, base + 0).standard_normal((batch, nheads, headdim)), io_dtype),
        "dt": _dt(seed, (batch, nheads), nheads, base + 1, io_dtype),
        "B": round_to(_rng(seed, base + 2).standard_normal((batch, ngroups, dstate)), io_dtype),
        "C": round_to(_rng(seed, base + 3).standard_normal((batch, ngroups, dstate)), io_dtype),
    }


def diag_inputs(batch: int, seqlen: int, dim: int, dstate: int, io_dtype: str = "bf16",
                seed: int = 0, init_state: bool = False, random_A: bool = False) -> dict:
    """Inputs of one Mamba-1 diagonal scan: x/dt[B,L,D], A[D,N] = -(n+1)
    (or, with random_A, -exp(U(ln 1, ln 16)) drawn per (channel, state)),
    B/C[B,L,N], D[D], init_state[B,D,N] (or None)."""
    Bsz, L, Dm, N = batch, seqlen, dim, dstate
    if random_A:
        A = -np.exp(_rng(seed, _S_A).uniform(0.0, np.log(16.0), size=(Dm, N)))
    else:
        A = -np.broadcast_to(np.arange(1, N + 1, dtype=np.float64), (Dm, N)).copy()
    out = {
        "x": round_to(_rng(seed, _S_X).standard_normal((Bsz, L, Dm)), io_dtype),
        "dt": _dt(seed, (Bsz, L, Dm), Dm, _S_DT_NOISE, io_dtype),
        "A": round_to(A, "f32"),
        "B": round_to(_rng(seed, _S_B).standard_normal((Bsz, L, N)), io_dtype),
        "C": round_to(_rng(seed, _S_C).standard_normal((Bsz, L, N)), io_dtype),
        "D": round_to(_rng(seed, _S_D).uniform(0.5, 1.5, size=Dm), "f32"),
        "init_state": None,
    }
    if init_state:
        out["init_state"] = round_to(_rng(seed, _S_STATE).normal(0.0, 0.1, size=(Bsz, Dm, N)), "f32")
    return out


def diag_option_inputs(batch: int, seqlen: int, dim: int, dstate: int, io_dtype: str = "bf16",
                       seed: int = 0, init_state: bool = False, bias: bool = True, z: bool = True,
                       random_A: bool = False) -> dict:
    """Inputs of a Mamba-1 scan run with delta_softplus: "dt" holds the raw
    pre-activation step. With bias, dt = eps and delta_bias[D] (float32) is
    the per-channel softplus^{-1} of a log-uniform target step in [1e-3, 1e-1];
    without, dt = eps + bias rounded to the I/O dtype. eps ~ N(0, 0.5), so
    softplus(dt + delta_bias) has the distribution of the other workloads'
    steps. With z, a gate z[B,L,D] ~ N(0, 1)."""
    out = diag_inputs(batch, seqlen, dim, dstate, io_dtype=io_dtype, seed=seed, init_state=init_state,
                      random_A=random_A)
    b = _dt_bias(_rng(seed, _S_DT0), dim)
    eps = _rng(seed, _S_DT_NOISE).normal(0.0, 0.5, size=(batch, seqlen, dim))
    if bias:
        out["dt"] = round_to(eps, io_dtype)
        out["delta_bias"] = round_to(b, "f32")
    else:
        out["dt"] = round_to(eps + b, io_dtype)
        out["delta_bias"] = None
    out["z"] = round_to(_rng(seed, _S_Z).standard_normal((batch, seqlen, dim)), io_dtype) if z else None
    return out


def decode_layer_params(batch: int, nheads: int, headdim: int, dstate: int, ngroups: int, width: int = 4,
                        seed: int = 0, conv_state: bool = True) -> dict:
    """Constants and initial states of a decode layer body: conv_w[Cc,W] ~
    U(-1/sqrt(W), 1/sqrt(W)), conv_b[Cc] ~ U(-0.1, 0.1), norm_w[H*P] ~
    U(0.5, 1.5), A/D as the decode workload, conv window[B,Cc,W] ~ N(0, 1)
    (or zeros), SSM state[B,H,P,N] ~ N(0, 0.1); Cc = H*P + 2*G*N."""
    Cc = nheads * headdim + 2 * ngroups * dstate
    r = 1.0 / np.sqrt(width)
    out = dict(decode_params(nheads, seed))
    out.update(
        conv_w=round_to(_rng(seed, _S_CONV_W).uniform(-r, r, size=(Cc, width)), "f32"),
        conv_b=round_to(_rng(seed, _S_CONV_B).uniform(-0.1, 0.1, size=Cc), "f32"),
        norm_w=round_to(_rng(seed, _S_NORM_W).uniform(0.5, 1.5, size=nheads * headdim), "f32"),
        conv_state=(round_to(_rng(seed, _S_CONV_STATE).standard_normal((batch, Cc, width)), "f32") if conv_state
                    else np.zeros((batch, Cc, width))),
        ssm_state=decode_state(batch, nheads, headdim, dstate, seed),
    )
    return out


def decode_layer_step_inputs(step: int, batch: int, nheads: int, headdim: int, dstate: int, ngroups: int,
                             io_dtype: str = "bf16", seed: int = 0) -> dict:
    """Per-token inputs of decode-layer step ``step``: xBC[B, H*P + 2*G*N] ~
    N(0, 1), dt[B,H] as the decode workload, gate z[B, H*P] ~ N(0, 1)."""
    base = _S_LAYER_BASE + 4 * int(step)
    Cc = nheads * headdim + 2 * ngroups * dstate
    return {
        "xBC": round_to(_rng(seed, base + 0).standard_normal((batch, Cc)), io_dtype),
        "dt": _dt(seed, (batch, nheads), nheads, base + 1, io_dtype),
        "z": round_to(_rng(seed, base + 2).standard_normal((batch, nheads * headdim)), io_dtype),
    }


# The benchmark workloads, named by what they are.
WORKLOADS = {
    "ssd_tiny_f32": dict(kind="ssd", batch=1, seqlen=256, nheads=4, headdim=64, dstate=16,
                         ngroups=1, io_dtype="f32", chunk=64),
    "ssd_m2_130m_L4096": dict(kind="ssd", batch=1, seqlen=4096, nheads=24, headdim=64,
                              dstate=128, ngroups=1, io_dtype="bf16", chunk=256),
    "ssd_m2_2p7b_L1024": dict(kind="ssd", batch=1, seqlen=1024, nheads=80, headdim=64,
                              dstate=128, ngroups=1, io_dtype="bf16", chunk=256),
    "ssd_m2_2p7b_L4096": dict(kind="ssd", batch=1, seqlen=4096, nheads=80, headdim=64,
                              dstate=128, ngroups=1, io_dtype="bf16", chunk=256),
    "ssd_m2_2p7b_L8192": dict(kind="ssd", batch=1, seqlen=8192, nheads=80, headdim=64,
                              dstate=128, ngroups=1, io_dtype="bf16", chunk=256),
    "ssd_m2_2p7b_B8_L2048": dict(kind="ssd", batch=8, seqlen=2048, nheads=80, headdim=64,
                                 dstate=128, ngroups=1, io_dtype="bf16", chunk=256),
    "decode_B64_H80": dict(kind="decode", batch=64, nheads=80, headdim=64, dstate=128,
                           ngroups=1, io_dtype="bf16", steps=1000),
    "mamba1_B8_L2048_D5120": dict(kind="diag", batch=8, seqlen=2048, dim=5120, dstate=16,
                                  io_dtype="bf16", chunk=2048),
    # decode layer body (conv step + silu, SSD decode step, gated RMS norm) as
    # one captured graph of 1000 steps: the decode workload's shape with a
    # width-4 conv, and the layer of the fused-decode sketch (d_inner 8192,
    # 128 heads, 8 groups, conv_dim 10240, norm over all of d_inner)
    "decode_layer_B64_H80": dict(kind="decode_layer", batch=64, nheads=80, headdim=64, dstate=128, ngroups=1,
                                 width=4, norm_group=5120, io_dtype="bf16", steps=1000),
    "decode_layer_B1_H128_G8": dict(kind="decode_layer", batch=1, nheads=128, headdim=64, dstate=128, ngroups=8,
                                    width=4, norm_group=8192, io_dtype="bf16", steps=1000),
    # selective_scan_fn as timed with delta_softplus set: batch 1, dim 1024,
    # length 4096, d_state 16 (the pages ran fp16; bf16 here, same bytes)
    "mamba1_B1_L4096_D1024_softplus": dict(kind="diag", batch=1, seqlen=4096, dim=1024, dstate=16,
                                           io_dtype="bf16", chunk=2048, delta_softplus=True),
}
