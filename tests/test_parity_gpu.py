"""Parity of the CUDA kernels with the float64 oracle, through the C ABI.

Small cases compare every element; the full-size workloads compare every
element where the oracle finishes in seconds and sampled heads / channels
otherwise. Tolerances are in tests/helpers.py.
"""
import numpy as np
import pytest
import torch

import oracle
from mamba_ssd_selective_gb300 import inputs
from tests.helpers import IO_TORCH, check, check_bf16, dev, head_slice, host

pytestmark = pytest.mark.gpu


def run_scan(ssd, d, io, chunk, simt=False, init=True, D=True, want_final=True):
    t = IO_TORCH[io]
    y, hT = ssd.ssd_scan_chunked(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                 dev(d["D"]) if D else None, dev(d["init_state"]) if init else None,
                                 chunk_size=chunk, simt=simt, want_final_state=want_final)
    torch.cuda.synchronize()
    return y, hT


def ref_scan(d, init=True, D=True):
    return oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"] if D else None,
                          d["init_state"] if init else None)


# ----------------------------------------------------------------- prefill

@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_prefill_tiny_f32_workload(ssd, chunk):
    """B1 L256 H4 P64 N16 G1, float32, zero initial state (chunk 64 is the workload's own)."""
    w = inputs.WORKLOADS["ssd_tiny_f32"]
    d = inputs.ssd_inputs(w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                          io_dtype="f32", seed=0)
    yr, hr = ref_scan(d, init=False)
    y, h = run_scan(ssd, d, "f32", chunk, init=False)
    check("f32", y, yr, "y")
    check("f32", h, hr, "final_state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("shape", [(2, 333, 4, 48, 20, 2), (1, 300, 2, 64, 128, 1), (3, 129, 6, 80, 70, 3)])
def test_prefill_ragged_groups_init(ssd, io, chunk, shape):
    """Ragged L (not a multiple of the chunk), P/N not multiples of 64, groups, init state and D."""
    Bz, L, H, P, N, G = shape
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype=io, seed=7, init_state=True)
    yr, hr = ref_scan(d)
    y, h = run_scan(ssd, d, io, chunk)
    check(io, y, yr, "y")
    check(io, h, hr, "final_state")


@pytest.mark.parametrize("shape", [(1, 4096, 21, 64, 128, 3), (2, 8192, 8, 64, 128, 1), (1, 4096, 15, 64, 128, 1),
                                   (1, 2048, 42, 64, 128, 1), (1, 1024, 39, 64, 128, 1), (2, 2048, 12, 64, 128, 3)])
def test_prefill_tensor_core_head_groups(ssd, shape):
    """Tensor-core path at shapes whose chunk-state cost model picks head groups
    of 7, 8, 5, 6 and 3 heads (MMA chains of 4 + 3, 4 + 4, 4 + 1, 4 + 2 and 3)
    and several B/C groups; every element against the oracle, with an initial
    state."""
    Bz, L, H, P, N, G = shape
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=11, init_state=True)
    yr, hr = ref_scan(d)
    y, h = run_scan(ssd, d, "bf16", 128)
    check("bf16", y, yr, "y")
    check("bf16", h, hr, "final_state")


@pytest.mark.parametrize("shape", [(1, 512, 24, 64, 128, 1), (2, 777, 8, 64, 128, 2)])
def test_prefill_policy_chunk(ssd, shape):
    """chunk_size=None takes the static policy's chunk; every element against
    the oracle."""
    Bz, L, H, P, N, G = shape
    assert ssd.ssd_best_chunk(Bz, L, H, P, N, G, torch.bfloat16) in (64, 128, 256)
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=19, init_state=True)
    yr, hr = ref_scan(d)
    y, h = run_scan(ssd, d, "bf16", None)
    check("bf16", y, yr, "y")
    check("bf16", h, hr, "final_state")


@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_prefill_m2_130m_workload_full(ssd, chunk, simt):
    """B1 L4096 H24 P64 N128 G1, bf16 inputs / fp32 state: every element of y and the state."""
    w = inputs.WORKLOADS["ssd_m2_130m_L4096"]
    d = inputs.ssd_inputs(w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                          io_dtype="bf16", seed=0)
    yr, hr = _cached_ref("m2_130m", d)
    y, h = run_scan(ssd, d, "bf16", chunk, simt=simt, init=False)
    check("bf16", y, yr, "y")
    check("bf16", h, hr, "final_state")


_REF_CACHE = {}


def _cached_ref(key, d, init=False):
    if key not in _REF_CACHE:
        _REF_CACHE[key] = ref_scan(d, init=init)
    return _REF_CACHE[key]


@pytest.mark.slow
@pytest.mark.parametrize("name", ["ssd_m2_2p7b_L1024", "ssd_m2_2p7b_L4096", "ssd_m2_2p7b_L8192",
                                  "ssd_m2_2p7b_B8_L2048"])
def test_prefill_m2_2p7b_workloads_sampled_heads(ssd, name):
    """H80 P64 N128 workloads at full size on the GPU; the oracle checks sampled heads
    (all batches, all tokens, y and final state), for each chunk size."""
    w = inputs.WORKLOADS[name]
    d = inputs.ssd_inputs(w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"],
                          io_dtype="bf16", seed=0)
    heads = [0, 37, 79]
    refs = {h: ref_scan(head_slice(d, h), init=False) for h in heads}
    for chunk in (64, 128, 256):
        y, hT = run_scan(ssd, d, "bf16", chunk, init=False)
        for h in heads:
            yr, hr = refs[h]
            check_bf16(y[:, :, h:h + 1], yr, f"{name} chunk {chunk} head {h} y")
            check_bf16(hT[:, h:h + 1], hr, f"{name} chunk {chunk} head {h} state")
        del y, hT


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_prefill_edge_lengths(ssd, io):
    """L = 0 (state passes through), 1, shorter than a chunk, one past a chunk."""
    for L in (0, 1, 5, 65, 257):
        d = inputs.ssd_inputs(2, L, 2, 64, 128, 1, io_dtype=io, seed=L, init_state=True)
        yr, hr = ref_scan(d)
        for chunk in (64, 256):
            y, h = run_scan(ssd, d, io, chunk)
            if L:
                check(io, y, yr, f"L={L} y")
            check(io, h, hr, f"L={L} state")
    # L = 0 without an initial state gives a zero final state
    d = inputs.ssd_inputs(1, 0, 2, 64, 16, 1, io_dtype=io, seed=1)
    _, h = run_scan(ssd, d, io, 64, init=False)
    assert float(h.abs().max()) == 0.0


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_prefill_optional_outputs_and_aliasing(ssd, io):
    """D = NULL, final_state = NULL, and final_state aliasing init_state."""
    t = IO_TORCH[io]
    d = inputs.ssd_inputs(1, 200, 4, 64, 128, 1, io_dtype=io, seed=3, init_state=True)
    yr, hr = ref_scan(d, D=False)
    y, h = run_scan(ssd, d, io, 128, D=False, want_final=False)
    assert h is None
    check(io, y, yr, "y without D")
    st = dev(d["init_state"])
    y2, h2 = ssd.ssd_scan_chunked(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                  None, st, chunk_size=128, final_state=st)
    torch.cuda.synchronize()
    assert h2.data_ptr() == st.data_ptr()
    check(io, st, hr, "state updated in place")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_prefill_deterministic_and_batched_equals_solo(ssd, io):
    d = inputs.ssd_inputs(3, 300, 4, 64, 128, 1, io_dtype=io, seed=5, init_state=True)
    y1, h1 = run_scan(ssd, d, io, 128)
    y2, h2 = run_scan(ssd, d, io, 128)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)
    for b in range(3):
        db = {k: (v[b:b + 1] if (v is not None and k not in ("A", "D")) else v) for k, v in d.items()}
        yb, hb = run_scan(ssd, db, io, 128)
        assert torch.equal(yb[0], y1[b]) and torch.equal(hb[0], h1[b])


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_prefill_split_resume_and_decode_continuation(ssd, io):
    """scan(L1) then scan(L2 | state) == scan(L1 + L2); prefill(L) then one decode
    step == prefill(L + 1)."""
    t = IO_TORCH[io]
    d = inputs.ssd_inputs(2, 301, 4, 64, 128, 1, io_dtype=io, seed=9, init_state=True)
    yf, hf = run_scan(ssd, d, io, 128)
    cut = 170
    a = {k: (v[:, :cut] if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    b = {k: (v[:, cut:] if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    y1, h1 = run_scan(ssd, a, io, 128)
    b["init_state"] = host(h1)
    y2, h2 = run_scan(ssd, b, io, 128)
    check(io, host(torch.cat([y1, y2], 1)), host(yf), "split y")
    check(io, host(h2), host(hf), "split state")
    # prefill(L-1) + decode == prefill(L)
    p = {k: (v[:, :300] if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    _, hp = run_scan(ssd, p, io, 128)
    yd = ssd.ssd_decode_step(hp, dev(d["x"][:, 300], t), dev(d["dt"][:, 300], t), dev(d["A"]),
                             dev(d["B"][:, 300], t), dev(d["C"][:, 300], t), dev(d["D"]))
    torch.cuda.synchronize()
    check(io, host(yd), host(yf[:, 300]), "decode after prefill y")
    check(io, host(hp), host(hf), "decode after prefill state")


def test_prefill_chunk_size_independent_within_tolerance(ssd):
    d = inputs.ssd_inputs(1, 1000, 4, 64, 128, 1, io_dtype="bf16", seed=2, init_state=True)
    y64, h64 = run_scan(ssd, d, "bf16", 64)
    for q in (128, 256):
        yq, hq = run_scan(ssd, d, "bf16", q)
        check_bf16(yq, host(y64), f"chunk {q} vs 64 y")
        check_bf16(hq, host(h64), f"chunk {q} vs 64 state")


# ------------------------------------------------------------------ decode

def _decode_inputs(step, Bz, H, P, N, G, io):
    return inputs.decode_step_inputs(step, Bz, H, P, N, G, io_dtype=io, seed=0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(4, 80, 64, 128, 1), (3, 6, 10, 30, 2), (2, 4, 64, 256, 4),
                                   (16, 80, 64, 128, 2), (20, 64, 48, 128, 4)])
def test_decode_steps_every_element(ssd, io, shape):
    """Ten in-place steps, every y and state element. The last two shapes have
    at least eight (b, h) per SM, where the launch takes four-warp CTAs, one
    per (b, h), eight resident per SM (P = 48: 12 rows per warp)."""
    Bz, H, P, N, G = shape
    t = IO_TORCH[io]
    st_ref = inputs.decode_state(Bz, H, P, N, seed=0)
    prm = inputs.decode_params(H, seed=0)
    st = dev(st_ref)
    A, D = dev(prm["A"]), dev(prm["D"])
    for s in range(10):
        di = _decode_inputs(s, Bz, H, P, N, G, io)
        y = ssd.ssd_decode_step(st, dev(di["x"], t), dev(di["dt"], t), A, dev(di["B"], t), dev(di["C"], t), D)
        yr, st_ref = oracle.ssd_decode(st_ref, di["x"], di["dt"], prm["A"], di["B"], di["C"], prm["D"])
        torch.cuda.synchronize()
        check(io, y, yr, f"step {s} y")
    check(io, st, st_ref, "state after 10 steps")


@pytest.mark.slow
def test_decode_workload_1000_steps_sampled(ssd):
    """B64 H80 P64 N128, fp32 state ~N(0,0.1), bf16 per-step inputs, 1000 in-place
    steps. The oracle replays sampled (b, h) rows as one 1000-token sequence
    (decode == prefill of the same tokens, pinned on the oracle) and checks y
    at steps 1, 10, 100, 1000 and the state after step 1000."""
    w = inputs.WORKLOADS["decode_B64_H80"]
    Bz, H, P, N, G, steps = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["steps"]
    t = torch.bfloat16
    st0 = inputs.decode_state(Bz, H, P, N, seed=0)
    prm = inputs.decode_params(H, seed=0)
    st = dev(st0)
    A, D = dev(prm["A"]), dev(prm["D"])
    samples = [(0, 0), (17, 41), (63, 79), (32, 5)]
    seq = {k: [] for k in ("x", "dt", "B", "C")}
    ys = {}
    for s in range(steps):
        di = _decode_inputs(s, Bz, H, P, N, G, "bf16")
        y = ssd.ssd_decode_step(st, dev(di["x"], t), dev(di["dt"], t), A, dev(di["B"], t), dev(di["C"], t), D)
        if s + 1 in (1, 10, 100, 1000):
            ys[s + 1] = host(y)
        for k in seq:
            seq[k].append(di[k])
    torch.cuda.synchronize()
    stg = host(st)
    for (b, h) in samples:
        g = h // (H // G)
        x = np.stack([a[b, h] for a in seq["x"]])[None, :, None, :]
        dt = np.array([a[b, h] for a in seq["dt"]])[None, :, None]
        Bm = np.stack([a[b, g] for a in seq["B"]])[None, :, None, :]
        Cm = np.stack([a[b, g] for a in seq["C"]])[None, :, None, :]
        yr, hr = oracle.ssd_seq(x, dt, prm["A"][h:h + 1], Bm, Cm, prm["D"][h:h + 1], st0[b:b + 1, h:h + 1])
        for s, yg in ys.items():
            check_bf16(yg[b, h], yr[0, s - 1, 0], f"(b,h)=({b},{h}) y at step {s}")
        check_bf16(stg[b, h], hr[0, 0], f"(b,h)=({b},{h}) state after {steps} steps")


# ------------------------------------------------------------------ Mamba-1

def run_diag(ssd, d, io, chunk, init=True):
    t = IO_TORCH[io]
    y, h = ssd.selective_scan_diag(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                   dev(d["D"]), dev(d["init_state"]) if init else None, chunk_size=chunk)
    torch.cuda.synchronize()
    return y, h


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 300, 256, 16), (1, 65, 200, 16), (2, 100, 136, 8), (1, 50, 72, 24),
                                   (1, 77, 130, 5), (2, 64, 100, 40)])
def test_diag_every_element(ssd, io, shape):
    Bz, L, Dm, N = shape
    d = inputs.diag_inputs(Bz, L, Dm, N, io_dtype=io, seed=4, init_state=True, random_A=True)
    yr, hr = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    y, h = run_diag(ssd, d, io, 64)
    check(io, y, yr, "y")
    check(io, h, hr, "final_state")


@pytest.mark.parametrize("dim", [300, 320])
def test_diag_chunk_size_bitwise_independent(ssd, dim):
    d = inputs.diag_inputs(2, 1000, dim, 16, io_dtype="bf16", seed=6, init_state=True)
    y0, h0 = run_diag(ssd, d, "bf16", 32)
    for c in (96, 256, 512, 1024, 2048):
        y, h = run_diag(ssd, d, "bf16", c)
        assert torch.equal(y, y0) and torch.equal(h, h0), f"chunk {c}"


@pytest.mark.slow
def test_diag_mamba1_workload_sampled(ssd):
    """B8 L2048 D5120 N16, A = -(1..16): full size on the GPU; the oracle checks
    sampled channels of every batch (all tokens, y and final state)."""
    w = inputs.WORKLOADS["mamba1_B8_L2048_D5120"]
    d = inputs.diag_inputs(w["batch"], w["seqlen"], w["dim"], w["dstate"], io_dtype="bf16", seed=0)
    chans = np.array([0, 1, 127, 128, 2049, 4000, 5119])
    ds = dict(x=d["x"][:, :, chans], dt=d["dt"][:, :, chans], A=d["A"][chans], B=d["B"], C=d["C"], D=d["D"][chans])
    yr, hr = oracle.diag_seq(ds["x"], ds["dt"], ds["A"], ds["B"], ds["C"], ds["D"])
    for chunk in (256, 2048):
        y, h = run_diag(ssd, d, "bf16", chunk, init=False)
        yh, hh = host(y)[:, :, chans], host(h)[:, chans]
        for i, c in enumerate(chans):
            check_bf16(yh[:, :, i], yr[:, :, i], f"channel {c} y")
            check_bf16(hh[:, i], hr[:, i], f"channel {c} state")


def run_diag_opts(ssd, d, io, chunk, softplus=True, init=True):
    t = IO_TORCH[io]
    y, h = ssd.selective_scan_diag(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                   dev(d["D"]), dev(d["init_state"]) if init else None, chunk_size=chunk,
                                   z=dev(d["z"], t) if d["z"] is not None else None,
                                   delta_bias=dev(d["delta_bias"]) if d["delta_bias"] is not None else None,
                                   delta_softplus=softplus)
    torch.cuda.synchronize()
    return y, h


DIAG_OPTS = {"softplus_bias_z": (True, True, True), "softplus_bias": (True, True, False),
             "z_only": (False, False, True), "bias_only": (False, True, False)}


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", sorted(DIAG_OPTS))
@pytest.mark.parametrize("shape", [(2, 300, 256, 16), (2, 100, 136, 8), (1, 50, 72, 24), (1, 77, 130, 5)])
def test_diag_options_every_element(ssd, io, opts, shape):
    softplus, bias, z = DIAG_OPTS[opts]
    Bz, L, Dm, N = shape
    d = inputs.diag_option_inputs(Bz, L, Dm, N, io_dtype=io, seed=14, init_state=True, bias=bias, z=z,
                                  random_A=True)
    if not softplus:   # feed steps that are valid without the softplus
        d["dt"] = inputs.round_to(np.abs(d["dt"]) * 0.05, io)
        if d["delta_bias"] is not None:
            d["delta_bias"] = np.abs(d["delta_bias"]) * 0.01
    yr, hr = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], z=d["z"],
                             delta_bias=d["delta_bias"], delta_softplus=softplus)
    y, h = run_diag_opts(ssd, d, io, 64, softplus=softplus)
    check(io, y, yr, "y")
    check(io, h, hr, "final_state")


@pytest.mark.parametrize("dim", [300, 320])
def test_diag_options_chunk_size_bitwise_independent(ssd, dim):
    d = inputs.diag_option_inputs(2, 1000, dim, 16, io_dtype="bf16", seed=16, init_state=True)
    y0, h0 = run_diag_opts(ssd, d, "bf16", 32)
    for c in (96, 256, 1024, 2048):
        y, h = run_diag_opts(ssd, d, "bf16", c)
        assert torch.equal(y, y0) and torch.equal(h, h0), f"chunk {c}"


@pytest.mark.slow
def test_diag_softplus_workload_sampled(ssd):
    """B1 L4096 D1024 N16 with delta_softplus (the raw step carries its bias):
    full size on the GPU, sampled channels through the oracle."""
    w = inputs.WORKLOADS["mamba1_B1_L4096_D1024_softplus"]
    d = inputs.diag_option_inputs(w["batch"], w["seqlen"], w["dim"], w["dstate"], io_dtype="bf16", seed=0,
                                  bias=False, z=False)
    chans = np.array([0, 5, 127, 128, 513, 1023])
    yr, hr = oracle.diag_seq(d["x"][:, :, chans], d["dt"][:, :, chans], d["A"][chans], d["B"], d["C"],
                             d["D"][chans], delta_softplus=True)
    for chunk in (256, 2048):
        y, h = run_diag_opts(ssd, d, "bf16", chunk, init=False)
        yh, hh = host(y)[:, :, chans], host(h)[:, chans]
        for i, c in enumerate(chans):
            check_bf16(yh[:, :, i], yr[:, :, i], f"channel {c} y")
            check_bf16(hh[:, i], hr[:, i], f"channel {c} state")


@pytest.mark.parametrize("opts", ["none", "softplus_bias_z"])
@pytest.mark.parametrize("shape", [(1, 1000, 64, 16), (2, 777, 136, 8), (1, 513, 72, 24), (1, 4096, 1024, 16)])
def test_diag_time_segmented_scan(ssd, opts, shape):
    """Small batch x dim, long sequence: the scan is cut into time segments
    (ragged last segment); every element against the oracle, and within bf16
    rounding of the one-pass scan of the same inputs."""
    Bz, L, Dm, N = shape
    assert ssd.selective_scan_diag_workspace_size(Bz, L, Dm, N, torch.bfloat16) > 0
    if opts == "none":
        d = inputs.diag_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=17, init_state=True, random_A=True)
        d.update(z=None, delta_bias=None)
        softplus = False
    else:
        d = inputs.diag_option_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=17, init_state=True, random_A=True)
        softplus = True
    yr, hr = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], z=d["z"],
                             delta_bias=d["delta_bias"], delta_softplus=softplus)
    y, h = run_diag_opts(ssd, d, "bf16", 64, softplus=softplus)
    check_bf16(y, yr, "y")
    check_bf16(h, hr, "final_state")
    t = torch.bfloat16
    y1, h1 = ssd.selective_scan_diag(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                     dev(d["D"]), dev(d["init_state"]), chunk_size=64,
                                     z=dev(d["z"], t) if d["z"] is not None else None,
                                     delta_bias=dev(d["delta_bias"]) if d["delta_bias"] is not None else None,
                                     delta_softplus=softplus, segmented=False)
    check_bf16(y, host(y1), "segmented vs one-pass y")
    np.testing.assert_allclose(host(h), host(h1), rtol=1e-4, atol=1e-5)


def test_diag_segmented_chunk_size_bitwise_independent(ssd):
    d = inputs.diag_option_inputs(1, 3000, 128, 16, io_dtype="bf16", seed=18, init_state=True)
    assert ssd.selective_scan_diag_workspace_size(1, 3000, 128, 16, torch.bfloat16) > 0
    y0, h0 = run_diag_opts(ssd, d, "bf16", 32)
    for c in (96, 256, 1024, 2048):
        y, h = run_diag_opts(ssd, d, "bf16", c)
        assert torch.equal(y, y0) and torch.equal(h, h0), f"chunk {c}"


# ---------------------------------------------------------------- backward

def _bwd_case(shape, io, seed):
    Bz, L, H, P, N, G = shape
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype=io, seed=seed, init_state=True)
    rng = np.random.default_rng(seed + 1000)
    dy = inputs.round_to(rng.standard_normal(d["x"].shape), io)
    dfin = inputs.round_to(rng.normal(0.0, 0.1, size=d["init_state"].shape), "f32")
    return d, dy, dfin


def _check_grads(g, ref, tol, what=""):
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        if k not in g or k not in ref:
            continue
        got, want = host(g[k]), ref[k]
        scale = float(np.max(np.abs(want))) if want.size else 0.0
        err = float(np.max(np.abs(got - want))) if want.size else 0.0
        assert err <= tol * scale + 1e-30, f"{what} {k}: max|err| = {err:.3e} > {tol} * max|ref| = {tol * scale:.3e}"


@pytest.mark.parametrize("io,tol", [("f32", 1e-4), ("bf16", 2e-2)])
@pytest.mark.parametrize("shape", [(1, 256, 4, 64, 16, 1), (2, 200, 4, 32, 64, 2), (1, 130, 3, 64, 128, 1),
                                   (2, 77, 6, 16, 32, 3), (1, 150, 2, 18, 10, 1), (2, 70, 2, 30, 64, 2)])
def test_backward_every_element(ssd, io, tol, shape):
    """Every gradient (dx, ddt, dA, dB, dC, dD, dinit) against the float64
    reverse-mode oracle; ragged last chunks, several B/C groups, and head
    sizes that are not multiples of 4 (element-wise loads and stores)."""
    d, dy, dfin = _bwd_case(shape, io, 21)
    ref = oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"], d["init_state"], dfin)
    t = IO_TORCH[io]
    g = ssd.ssd_scan_chunked_bwd(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                 dev(dy, t), dev(d["D"]), dev(d["init_state"]), dev(dfin))
    torch.cuda.synchronize()
    _check_grads(g, ref, tol, f"{io} {shape}")


@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("shape", [(1, 128, 2, 64, 128, 1), (2, 300, 4, 64, 128, 2), (1, 1000, 6, 64, 128, 3),
                                   (3, 129, 2, 64, 128, 1), (1, 300, 3, 64, 128, 1), (2, 257, 6, 64, 128, 6)])
def test_backward_tensor_core_shapes(ssd, shape, simt):
    """bf16, P 64, N 128: the per-chunk gradients on the tensor cores (chunks
    of 128 tokens) and, forced, on the CUDA cores (chunks of 64): every
    gradient against the float64 oracle within the bf16 bound; one full chunk,
    ragged last chunks (300 = 2 x 128 + 44, 129 = 128 + 1, 257 = 2 x 128 + 1),
    several B/C groups, eight chunks; an even number of heads per group (the
    gradient kernel sums pairs of heads) and an odd one (3, and 1 with six
    groups: one part per head)."""
    d, dy, dfin = _bwd_case(shape, "bf16", 31)
    ref = oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"], d["init_state"], dfin)
    t = torch.bfloat16
    g = ssd.ssd_scan_chunked_bwd(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                 dev(dy, t), dev(d["D"]), dev(d["init_state"]), dev(dfin), simt=simt)
    torch.cuda.synchronize()
    _check_grads(g, ref, 2e-2, f"bf16 {shape} simt={simt}")
    worst = {}
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        want = ref[k]
        worst[k] = float(np.max(np.abs(host(g[k]) - want)) / max(float(np.max(np.abs(want))), 1e-30))
    print(f"backward {shape} simt={simt}: " + ", ".join(f"{k} {v:.1e}" for k, v in worst.items()))


@pytest.mark.parametrize("shape,optionals", [((1, 2048, 24, 64, 128, 1), False), ((4, 2048, 80, 64, 128, 1), True),
                                             ((2, 4096, 48, 64, 128, 8), True)])
def test_backward_full_size_every_element(ssd, shape, optionals):
    """The sizes the bench times, on the tensor-core path: the 130M-shaped
    layer at L 2048 with the bench's own inputs (no initial state, no final
    cotangent), and the 2.7B-shaped layer at B4 L2048 with both; and eight
    B/C groups of six heads at B2 L4096; every element of every gradient
    against the float64 oracle within the bf16 bound (the oracle runs on the
    host's threads: a few seconds)."""
    Bz, L, H, P, N, G = shape
    if optionals:
        d, dy, dfin = _bwd_case(shape, "bf16", 41)
    else:
        d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=0)
        dy = inputs.round_to(np.random.default_rng(1).standard_normal(d["x"].shape), "bf16")
        d["init_state"], dfin = None, None
    ref = oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"], d["init_state"], dfin)
    t = torch.bfloat16
    g = ssd.ssd_scan_chunked_bwd(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                                 dev(dy, t), dev(d["D"]), None if d["init_state"] is None else dev(d["init_state"]),
                                 None if dfin is None else dev(dfin))
    torch.cuda.synchronize()
    if not optionals:
        ref = {k: v for k, v in ref.items() if k != "dinit"}
    _check_grads(g, ref, 2e-2, f"bf16 {shape}")
    worst = {k: float(np.max(np.abs(host(g[k]) - ref[k])) / max(float(np.max(np.abs(ref[k]))), 1e-30))
             for k in ("dx", "ddt", "dA", "dB", "dC", "dD")}
    print(f"backward {shape}: " + ", ".join(f"{k} {v:.1e}" for k, v in worst.items()))


def test_backward_deterministic_and_without_optionals(ssd):
    """Two runs give the same bits; with no D, no initial state and no final
    cotangent the gradients still match the oracle."""
    d, dy, _ = _bwd_case((1, 300, 4, 64, 128, 1), "bf16", 23)
    t = torch.bfloat16
    args = (dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t), dev(dy, t))
    g1 = ssd.ssd_scan_chunked_bwd(*args)
    g2 = ssd.ssd_scan_chunked_bwd(*args)
    torch.cuda.synchronize()
    for k in g1:
        if g1[k] is not None:
            assert torch.equal(g1[k], g2[k]), k
    ref = oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy)
    ref["dD"] = None
    _check_grads({k: v for k, v in g1.items() if k != "dD"}, {k: v for k, v in ref.items() if k != "dD"}, 2e-2)


# ------------------------------------------------- decode-layer neighbours

@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("shape", [(3, 77), (2, 5376)])
def test_conv1d_step_every_element(ssd, io, width, shape):
    """Six steps on one window: every output element against the oracle, and
    the window (copies of inputs, no arithmetic) bit-exact."""
    Bz, C = shape
    rng = np.random.default_rng(50 + width)
    t = IO_TORCH[io]
    w = inputs.round_to(rng.uniform(-0.5, 0.5, size=(C, width)), "f32")
    bias = inputs.round_to(rng.uniform(-0.1, 0.1, size=C), "f32") if width != 3 else None
    st0 = inputs.round_to(rng.standard_normal((Bz, C, width)), "f32")
    ref_st = st0.copy()
    g_st = dev(st0)
    for step in range(6):
        x = inputs.round_to(rng.standard_normal((Bz, C)), io)
        silu = step % 2 == 0
        ref = oracle.conv1d_step(ref_st, x, w, bias, silu=silu)
        out = ssd.conv1d_step(dev(x, t), g_st, dev(w), dev(bias), silu=silu)
        torch.cuda.synchronize()
        check(io, out, ref, f"step {step} out")
        np.testing.assert_array_equal(host(g_st), ref_st)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("gate", [True, False])
@pytest.mark.parametrize("shape", [(3, 512, 512), (3, 512, 128), (64, 5120, 5120), (2, 8192, 1024), (1, 96, 32)])
def test_gated_rmsnorm_every_element(ssd, io, gate, shape):
    Bz, D, grp = shape
    rng = np.random.default_rng(60)
    t = IO_TORCH[io]
    y = inputs.round_to(rng.standard_normal((Bz, D)), io)
    z = inputs.round_to(rng.standard_normal((Bz, D)), io) if gate else None
    w = inputs.round_to(rng.uniform(0.5, 1.5, size=D), "f32")
    ref = oracle.gated_rmsnorm(y, z, w, grp, eps=1e-5)
    out = ssd.gated_rmsnorm(dev(y, t), dev(z, t), dev(w), grp, eps=1e-5)
    torch.cuda.synchronize()
    check(io, out, ref, "out")


def _layer_case(Bz, H, P, N, G, W, io, steps, seed=7):
    prm = inputs.decode_layer_params(Bz, H, P, N, G, W, seed=seed)
    st = [inputs.decode_layer_step_inputs(k, Bz, H, P, N, G, io_dtype=io, seed=seed) for k in range(steps)]
    return prm, st


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 4, 64, 128, 2, 4, 128), (3, 6, 32, 16, 3, 3, 96), (1, 128, 64, 128, 8, 4, 8192),
                                   (2, 8, 64, 128, 1, 4, 64), (16, 80, 64, 128, 1, 4, 5120)])
def test_decode_layer_steps_match_oracle(ssd, io, shape):
    """Eight layer steps (conv + silu, SSD decode step, gated norm): every
    output element each step and both states at the end, against the oracle."""
    Bz, H, P, N, G, W, grp = shape
    t = IO_TORCH[io]
    prm, steps = _layer_case(Bz, H, P, N, G, W, io, 8)
    cst, sst = prm["conv_state"].copy(), prm["ssm_state"].copy()
    g_cst, g_sst = dev(prm["conv_state"]), dev(prm["ssm_state"])
    for k, s_ in enumerate(steps):
        ref = oracle.decode_layer_step(cst, sst, s_["xBC"], prm["conv_w"], prm["conv_b"], s_["dt"], prm["A"],
                                       prm["D"], s_["z"], prm["norm_w"], H, P, N, G, group=grp, eps=1e-5)
        out = ssd.decode_layer_step(dev(s_["xBC"], t), g_cst, dev(prm["conv_w"]), dev(prm["conv_b"]),
                                    dev(s_["dt"], t), dev(prm["A"]), dev(prm["D"]), g_sst, dev(s_["z"], t),
                                    dev(prm["norm_w"]), norm_group=grp, eps=1e-5)
        torch.cuda.synchronize()
        check(io, out, ref, f"step {k} out")
    np.testing.assert_array_equal(host(g_cst), cst)
    check(io, g_sst, sst, "ssm_state after 8 steps")


def test_decode_graph_equals_eager_steps(ssd):
    """A 16-step loop captured by the library as one CUDA graph gives the
    same bits as 16 eager layer steps; a second launch continues the states."""
    Bz, H, P, N, G, W, K = 4, 8, 64, 128, 1, 4, 16
    t = torch.bfloat16
    prm, steps = _layer_case(Bz, H, P, N, G, W, "bf16", K, seed=9)
    xBC = dev(np.stack([s_["xBC"] for s_ in steps]), t)
    dt = dev(np.stack([s_["dt"] for s_ in steps]), t)
    z = dev(np.stack([s_["z"] for s_ in steps]), t)
    consts = [dev(prm["conv_w"]), dev(prm["conv_b"])]
    A, Dv, nw = dev(prm["A"]), dev(prm["D"]), dev(prm["norm_w"])
    e_cst, e_sst = dev(prm["conv_state"]), dev(prm["ssm_state"])
    g_cst, g_sst = dev(prm["conv_state"]), dev(prm["ssm_state"])
    graph = ssd.DecodeGraph(xBC, g_cst, *consts, dt, A, Dv, g_sst, z, nw, norm_group=P)
    try:
        for rep in range(2):
            eager = torch.stack([ssd.decode_layer_step(xBC[k], e_cst, *consts, dt[k], A, Dv, e_sst, z[k], nw,
                                                       norm_group=P) for k in range(K)])
            out = graph.launch()
            torch.cuda.synchronize()
            assert torch.equal(out, eager), f"launch {rep}: outputs differ"
            assert torch.equal(g_cst, e_cst) and torch.equal(g_sst, e_sst), f"launch {rep}: states differ"
    finally:
        graph.close()


# ------------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives(ssd):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert ssd.ssd_workspace_status(ws) == ssd.SSD_OK
    ssd.ssd_selftest_bounded_wait(ws, 1000)
    assert ssd.ssd_workspace_status(ws) == ssd.SSD_ERR_TIMEOUT
    # the context is still usable
    d = inputs.ssd_inputs(1, 64, 2, 64, 16, 1, io_dtype="f32", seed=1)
    yr, hr = ref_scan(d, init=False)
    y, h = run_scan(ssd, d, "f32", 64, init=False)
    check("f32", y, yr, "y after timeout self-test")


def test_workspace_status_ok_after_tensor_core_scan(ssd):
    d = inputs.ssd_inputs(1, 512, 4, 64, 128, 1, io_dtype="bf16", seed=1)
    t = torch.bfloat16
    ws = torch.empty(ssd.ssd_workspace_size(1, 512, 4, 64, 128, 1, t, 128), dtype=torch.uint8, device="cuda")
    ssd.ssd_scan_chunked(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t),
                         dev(d["D"]), None, chunk_size=128, workspace=ws)
    assert ssd.ssd_workspace_status(ws) == ssd.SSD_OK


@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_tensor_core_scan_repeated_no_timeouts(ssd, chunk):
    """Hundreds of back-to-back tensor-core scans of the 130M-shaped layer: no
    bounded wait may expire (a lost barrier phase would), and every repetition
    gives the same bits."""
    w = inputs.WORKLOADS["ssd_m2_130m_L4096"]
    Bz, L, H, P, N, G = w["batch"], w["seqlen"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype="bf16", seed=3)
    t = torch.bfloat16
    args = [dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t), dev(d["D"]), None]
    ws = torch.empty(ssd.ssd_workspace_size(Bz, L, H, P, N, G, t, chunk), dtype=torch.uint8, device="cuda")
    y0, h0 = ssd.ssd_scan_chunked(*args, chunk_size=chunk, workspace=ws)
    assert ssd.ssd_workspace_status(ws) == ssd.SSD_OK
    y, h = torch.empty_like(y0), torch.empty_like(h0)
    for rep in range(150):
        ssd.ssd_scan_chunked(*args, chunk_size=chunk, y=y, final_state=h, workspace=ws)
        assert ssd.ssd_workspace_status(ws) == ssd.SSD_OK, f"bounded wait expired in repetition {rep}"
    assert torch.equal(y, y0) and torch.equal(h, h0)


@pytest.mark.parametrize("case", ["tensor_core", "simt", "no_tokens"])
def test_scan_clears_a_stale_timeout_status(ssd, case):
    """The status word reports the latest call only: a TIMEOUT left in the
    workspace by an earlier call is cleared by the next scan."""
    L = 0 if case == "no_tokens" else 256
    io = torch.bfloat16 if case != "simt" else torch.float32
    d = inputs.ssd_inputs(1, max(L, 1), 4, 64, 128, 1, io_dtype="bf16" if io == torch.bfloat16 else "f32", seed=2)
    x, dt = dev(d["x"], io)[:, :L].contiguous(), dev(d["dt"], io)[:, :L].contiguous()
    Bm, Cm = dev(d["B"], io)[:, :L].contiguous(), dev(d["C"], io)[:, :L].contiguous()
    ws = torch.empty(max(256, ssd.ssd_workspace_size(1, L, 4, 64, 128, 1, io, 128)), dtype=torch.uint8, device="cuda")
    ssd.ssd_selftest_bounded_wait(ws, 1000)
    assert ssd.ssd_workspace_status(ws) == ssd.SSD_ERR_TIMEOUT
    ssd.ssd_scan_chunked(x, dt, dev(d["A"]), Bm, Cm, dev(d["D"]), None, chunk_size=128, workspace=ws,
                         simt=(case == "simt"))
    assert ssd.ssd_workspace_status(ws) == ssd.SSD_OK
