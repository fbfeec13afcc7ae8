"""Seeded random shapes through every compute path, against the oracle.

Shapes are drawn from a fixed-seed generator (so a failure reproduces): the
prefill with the tensor-core head size (P 64, N 128) at random batch, length
(including very short and ragged), head and group counts and chunk size; the
CUDA-core prefill at other head sizes; the Mamba-1 scan with and without the
options and time segments; the decode step.
"""
import numpy as np
import pytest
import torch

import oracle
from mamba_ssd_selective_gb300 import inputs
from tests.helpers import IO_TORCH, check, check_bf16, dev

pytestmark = pytest.mark.gpu


def _prefill_shapes():
    rng = np.random.default_rng(2024)
    out = []
    for _ in range(10):
        G = int(rng.choice([1, 1, 2, 3]))
        H = G * int(rng.integers(1, 7))
        L = int(rng.choice([1, 5, 63, 64, 65, 127, 129, 300, 777, 1500]))
        out.append((int(rng.integers(1, 3)), L, H, 64, 128, G, int(rng.choice([64, 128, 256]))))
    return out


@pytest.mark.parametrize("shape", _prefill_shapes())
def test_random_prefill_tensor_core(ssd, shape):
    Bz, L, H, P, N, G, q = shape
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=L + H, init_state=True)
    yr, hr = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    t = torch.bfloat16
    y, h = ssd.ssd_scan_chunked(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                dev(d["D"]), dev(d["init_state"]), chunk_size=q)
    torch.cuda.synchronize()
    check_bf16(y, yr, f"{shape} y")
    check_bf16(h, hr, f"{shape} final_state")


def _simt_shapes():
    rng = np.random.default_rng(7)
    out = []
    for _ in range(8):
        G = int(rng.choice([1, 2]))
        out.append((int(rng.integers(1, 3)), int(rng.integers(1, 400)), G * int(rng.integers(1, 4)),
                    int(rng.choice([8, 16, 32, 48, 64])), int(rng.choice([4, 16, 32, 64])), G,
                    str(rng.choice(["f32", "bf16"])), int(rng.choice([64, 128, 256]))))
    return out


@pytest.mark.parametrize("shape", _simt_shapes())
def test_random_prefill_cuda_cores(ssd, shape):
    Bz, L, H, P, N, G, io, q = shape
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype=io, seed=L * 3 + P, init_state=True)
    yr, hr = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    t = IO_TORCH[io]
    y, h = ssd.ssd_scan_chunked(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                dev(d["D"]), dev(d["init_state"]), chunk_size=q)
    torch.cuda.synchronize()
    check(io, y, yr, f"{shape} y")
    check(io, h, hr, f"{shape} final_state")


def _diag_shapes():
    rng = np.random.default_rng(11)
    out = []
    for _ in range(10):
        out.append((int(rng.integers(1, 3)), int(rng.choice([1, 31, 100, 129, 500, 2100])),
                    int(rng.choice([8, 24, 64, 72, 136, 200, 264])), int(rng.choice([4, 8, 16, 24, 32])),
                    str(rng.choice(["f32", "bf16"])), bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("shape", _diag_shapes())
def test_random_diag(ssd, shape):
    Bz, L, Dm, N, io, opts = shape
    if opts:
        d = inputs.diag_option_inputs(Bz, L, Dm, N, io_dtype=io, seed=L + Dm, init_state=True, random_A=True)
    else:
        d = inputs.diag_inputs(Bz, L, Dm, N, io_dtype=io, seed=L + Dm, init_state=True, random_A=True)
        d.update(z=None, delta_bias=None)
    yr, hr = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], z=d["z"],
                             delta_bias=d["delta_bias"], delta_softplus=opts)
    t = IO_TORCH[io]
    y, h = ssd.selective_scan_diag(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                   dev(d["D"]), dev(d["init_state"]), chunk_size=96,
                                   z=dev(d["z"], t) if d["z"] is not None else None,
                                   delta_bias=dev(d["delta_bias"]) if d["delta_bias"] is not None else None,
                                   delta_softplus=opts)
    torch.cuda.synchronize()
    check(io, y, yr, f"{shape} y")
    check(io, h, hr, f"{shape} final_state")


def _decode_shapes():
    rng = np.random.default_rng(13)
    out = []
    for _ in range(8):
        G = int(rng.choice([1, 2, 4]))
        out.append((int(rng.choice([1, 3, 20])), G * int(rng.integers(1, 9)), int(rng.choice([16, 32, 64])),
                    int(rng.choice([16, 64, 128, 130])), G, str(rng.choice(["f32", "bf16"]))))
    return out


@pytest.mark.parametrize("shape", _decode_shapes())
def test_random_decode(ssd, shape):
    Bz, H, P, N, G, io = shape
    st0 = inputs.decode_state(Bz, H, P, N, seed=H)
    prm = inputs.decode_params(H, seed=H)
    t = IO_TORCH[io]
    st = dev(st0)
    ref = st0.copy()
    for k in range(3):
        di = inputs.decode_step_inputs(k, Bz, H, P, N, G, io_dtype=io, seed=H)
        y = ssd.ssd_decode_step(st, dev(di["x"], t), dev(di["dt"], t), dev(prm["A"]), dev(di["B"], t),
                                dev(di["C"], t), dev(prm["D"]))
        torch.cuda.synchronize()
        yr, ref = oracle.ssd_decode(ref, di["x"], di["dt"], prm["A"], di["B"], di["C"], prm["D"])
        check(io, y, yr, f"{shape} y step {k}")
    check(io, st, ref, f"{shape} state")
