"""Pins of the float64 oracle against facts fixed outside the oracle itself.

The pages print no worked numeric example of the scan, so each oracle function
is pinned by: an independent quadratic (masked attention) form, closed forms
(A = 0, L = 1, dt = 0, memoryless decay), a library IIR filter
(scipy.signal.lfilter), brute-force expansions with explicit products of the
per-token decays, a hand-worked example in tests/golden, and the invariants of
the recurrence (carried-state continuation, split/resume, decode after
prefill, superposition, batched == solo, Mamba-2 == Mamba-1 with tied decays).
Each check is chosen so that a plausible slip in the oracle -- a dropped D or
dt term, a wrong sign of A, y read from the pre-update state, P and N swapped,
a wrong group index -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from mamba_ssd_selective_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(B=2, L=37, H=4, P=3, N=5, G=2, seed=3, init=True, io="f32"):
    d = inputs.ssd_inputs(B, L, H, P, N, G, io_dtype=io, seed=seed, init_state=init)
    # make the two groups clearly different and the decay non-trivial
    return d


def test_quadratic_form_matches_recurrence():
    d = _small()
    y1, h1 = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    y2, h2 = oracle.ssd_quadratic(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    np.testing.assert_allclose(y1, y2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h1, h2, rtol=1e-11, atol=1e-12)


def test_quadratic_form_detects_group_swap():
    # the check above must be able to fail: swapping the groups of B changes y
    d = _small()
    y1, _ = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    y2, _ = oracle.ssd_quadratic(d["x"], d["dt"], d["A"], d["B"][:, :, ::-1].copy(), d["C"], d["D"],
                                 d["init_state"])
    assert np.max(np.abs(y1 - y2)) > 1e-3


def test_A_zero_closed_form():
    """A = 0: no decay, the state is a plain running sum h_t = h0 + sum_{s<=t} dt_s x_s B_s^T."""
    d = _small()
    A0 = np.zeros_like(d["A"])
    y, hT = oracle.ssd_seq(d["x"], d["dt"], A0, d["B"], d["C"], d["D"], d["init_state"])
    B_, L, H, P = d["x"].shape
    G = d["B"].shape[2]
    for b in range(B_):
        for h in range(H):
            g = h // (H // G)
            inc = (d["dt"][b, :, h, None, None] * d["x"][b, :, h, :, None]
                   * d["B"][b, :, g, None, :])                     # [L, P, N]
            hs = d["init_state"][b, h][None] + np.cumsum(inc, axis=0)
            ref_y = np.einsum("tn,tpn->tp", d["C"][b, :, g], hs) + d["D"][h] * d["x"][b, :, h]
            np.testing.assert_allclose(y[b, :, h], ref_y, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(hT[b, h], hs[-1], rtol=1e-12, atol=1e-12)


def test_single_token_closed_form():
    """L = 1, zero initial state: y = dt (C.B) x + D x and h = dt x B^T."""
    d = inputs.ssd_inputs(3, 1, 4, 6, 5, 2, io_dtype="f32", seed=11)
    y, hT = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    for b in range(3):
        for h in range(4):
            g = h // 2
            cb = float(np.dot(d["C"][b, 0, g], d["B"][b, 0, g]))
            dtv = d["dt"][b, 0, h]
            np.testing.assert_allclose(y[b, 0, h], dtv * cb * d["x"][b, 0, h] + d["D"][h] * d["x"][b, 0, h],
                                       rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(hT[b, h], dtv * np.outer(d["x"][b, 0, h], d["B"][b, 0, g]),
                                       rtol=1e-13, atol=1e-14)


def test_memoryless_under_strong_decay():
    """dt*A << -50: earlier tokens are forgotten, y_t = dt_t (C_t.B_t) x_t + D x_t."""
    d = inputs.ssd_inputs(1, 20, 2, 3, 4, 1, io_dtype="f32", seed=5)
    dt = np.full_like(d["dt"], 1.0)
    A = np.full_like(d["A"], -200.0)
    y, _ = oracle.ssd_seq(d["x"], dt, A, d["B"], d["C"], d["D"])
    cb = np.einsum("ltn,ltn->lt", d["C"][:, :, 0], d["B"][:, :, 0])  # [B, L]
    ref = cb[:, :, None, None] * d["x"] + d["D"][None, None, :, None] * d["x"]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_dt_zero_keeps_state():
    """dt = 0: the state is left unchanged and y_t = C_t . h0 + D x_t."""
    d = _small()
    dt0 = np.zeros_like(d["dt"])
    y, hT = oracle.ssd_seq(d["x"], dt0, d["A"], d["B"], d["C"], d["D"], d["init_state"])
    np.testing.assert_array_equal(hT, d["init_state"])
    B_, L, H, P = d["x"].shape
    for h in range(H):
        g = h // (H // 2)
        ref = np.einsum("btn,bpn->btp", d["C"][:, :, g], d["init_state"][:, h]) + d["D"][h] * d["x"][:, :, h]
        np.testing.assert_allclose(y[:, :, h], ref, rtol=1e-12, atol=1e-12)


def test_lfilter_constant_dt():
    """With dt constant per head, every state entry (p, n) is a first-order IIR
    filter of the input u_t = dt x_t[p] B_t[n] with pole exp(dt A):
    scipy.signal.lfilter([1], [1, -alpha], u, zi=[alpha h0])."""
    signal = pytest.importorskip("scipy.signal")
    d = inputs.ssd_inputs(1, 50, 3, 4, 6, 1, io_dtype="f32", seed=21, init_state=True)
    dtc = np.array([0.05, 0.2, 0.7])
    dt = np.broadcast_to(dtc, d["dt"].shape).copy()
    y, hT = oracle.ssd_seq(d["x"], dt, d["A"], d["B"], d["C"], d["D"], d["init_state"])
    for h in range(3):
        alpha = math.exp(dtc[h] * d["A"][h])
        hs = np.zeros((50, 4, 6))
        for p in range(4):
            for n in range(6):
                u = dtc[h] * d["x"][0, :, h, p] * d["B"][0, :, 0, n]
                hs[:, p, n], _ = signal.lfilter([1.0], [1.0, -alpha], u, zi=[alpha * d["init_state"][0, h, p, n]])
        ref_y = np.einsum("tn,tpn->tp", d["C"][0, :, 0], hs) + d["D"][h] * d["x"][0, :, h]
        np.testing.assert_allclose(y[0, :, h], ref_y, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hT[0, h], hs[-1], rtol=1e-11, atol=1e-12)


def _brute_force_y(x, dt, A, Bm, Cm, D, h0):
    """Explicit expansion with products of per-token decays (no sums of exponents):
    y_t[p] = sum_n C_t[n] (prod_{k<=t} alpha_k h0[p,n]
             + sum_{s<=t} prod_{s<k<=t} alpha_k dt_s x_s[p] B_s[n]) + D x_t[p]."""
    L, P = x.shape
    N = Bm.shape[1]
    alpha = [math.exp(dt[k] * A) for k in range(L)]
    y = np.zeros((L, P))
    for t in range(L):
        for p in range(P):
            acc = 0.0
            for n in range(N):
                decay_all = 1.0
                for k in range(t + 1):
                    decay_all *= alpha[k]
                hv = decay_all * h0[p][n]
                for s in range(t + 1):
                    dec = 1.0
                    for k in range(s + 1, t + 1):
                        dec *= alpha[k]
                    hv += dec * dt[s] * x[s][p] * Bm[s][n]
                acc += Cm[t][n] * hv
            y[t][p] = acc + D * x[t][p]
    return y


def test_brute_force_tiny():
    d = inputs.ssd_inputs(1, 4, 1, 2, 2, 1, io_dtype="f32", seed=8, init_state=True)
    y, _ = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    ref = _brute_force_y(d["x"][0, :, 0], d["dt"][0, :, 0], d["A"][0], d["B"][0, :, 0], d["C"][0, :, 0],
                         d["D"][0], d["init_state"][0, 0])
    np.testing.assert_allclose(y[0, :, 0], ref, rtol=1e-13, atol=1e-14)


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_ssd.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    x = np.array(inp["x"], dtype=np.float64).reshape(1, -1, 1, 1)
    L = x.shape[1]
    dt = np.array(inp["dt"]).reshape(1, L, 1)
    Bm = np.array(inp["B"]).reshape(1, L, 1, 1)
    Cm = np.array(inp["C"]).reshape(1, L, 1, 1)
    y, hT = oracle.ssd_seq(x, dt, [inp["A"]], Bm, Cm, [inp["D"]])
    np.testing.assert_allclose(y.reshape(-1), g["expected"]["y"], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(hT.reshape(-1), g["expected"]["final_state"], rtol=1e-15, atol=1e-15)


def test_carried_state_chunk_by_chunk_equals_full_run():
    d = _small(L=64)
    yf, hf = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    for Q in (1, 7, 16, 64):
        h = d["init_state"]
        ys = []
        for s in range(0, 64, Q):
            sl = slice(s, s + Q)
            yc, h = oracle.ssd_seq(d["x"][:, sl], d["dt"][:, sl], d["A"], d["B"][:, sl], d["C"][:, sl],
                                   d["D"], h)
            ys.append(yc)
        np.testing.assert_allclose(np.concatenate(ys, axis=1), yf, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h, hf, rtol=1e-12, atol=1e-13)


def test_split_and_resume_anywhere():
    d = _small(L=41)
    yf, hf = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    for cut in (0, 1, 13, 40, 41):
        a, b = slice(0, cut), slice(cut, None)
        y1, h1 = oracle.ssd_seq(d["x"][:, a], d["dt"][:, a], d["A"], d["B"][:, a], d["C"][:, a], d["D"],
                                d["init_state"])
        y2, h2 = oracle.ssd_seq(d["x"][:, b], d["dt"][:, b], d["A"], d["B"][:, b], d["C"][:, b], d["D"], h1)
        np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), yf, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h2, hf, rtol=1e-12, atol=1e-13)


def test_decode_after_prefill_equals_longer_prefill():
    d = _small(L=30)
    yf, hf = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    y1, h1 = oracle.ssd_seq(d["x"][:, :29], d["dt"][:, :29], d["A"], d["B"][:, :29], d["C"][:, :29], d["D"],
                            d["init_state"])
    yd, hd = oracle.ssd_decode(h1, d["x"][:, 29], d["dt"][:, 29], d["A"], d["B"][:, 29], d["C"][:, 29], d["D"])
    np.testing.assert_allclose(yd, yf[:, 29], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hd, hf, rtol=1e-12, atol=1e-13)
    # the input state is not modified by the wrapper
    y1b, h1b = oracle.ssd_seq(d["x"][:, :29], d["dt"][:, :29], d["A"], d["B"][:, :29], d["C"][:, :29], d["D"],
                              d["init_state"])
    np.testing.assert_array_equal(h1, h1b)


def test_superposition_in_x_and_h0():
    """Linear in (x, h0) for fixed dt, B, C: y(x, h0) = y(x, 0) + y(0, h0) (D applies to x)."""
    d = _small()
    y, h = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    ya, ha = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None)
    yb, hb = oracle.ssd_seq(np.zeros_like(d["x"]), d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    np.testing.assert_allclose(y, ya + yb, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h, ha + hb, rtol=1e-11, atol=1e-12)


def test_batched_equals_solo_bitwise():
    d = _small(B=3)
    y, h = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    for b in range(3):
        s = slice(b, b + 1)
        ys, hs = oracle.ssd_seq(d["x"][s], d["dt"][s], d["A"], d["B"][s], d["C"][s], d["D"], d["init_state"][s])
        np.testing.assert_array_equal(ys, y[s])
        np.testing.assert_array_equal(hs, h[s])


def test_thread_count_does_not_change_result():
    d = _small(B=3)
    r1 = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], threads=1)
    r2 = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], threads=5)
    np.testing.assert_array_equal(r1[0], r2[0])
    np.testing.assert_array_equal(r1[1], r2[1])


# ---------------------------------------------------------------- Mamba-1 diag

def test_mamba2_equals_mamba1_with_tied_decay():
    """SSD head h with headdim P is P Mamba-1 channels sharing dt_h and A[d, n] = A_h."""
    d = inputs.ssd_inputs(2, 33, 3, 4, 5, 1, io_dtype="f32", seed=4, init_state=True)
    Bz, L, H, P = d["x"].shape
    N = 5
    y, h = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    xd = d["x"].reshape(Bz, L, H * P)
    dtd = np.repeat(d["dt"], P, axis=2)
    Ad = np.repeat(np.repeat(d["A"][:, None], P, axis=0), N, axis=1)
    Dd = np.repeat(d["D"], P)
    yd, hd = oracle.diag_seq(xd, dtd, Ad, d["B"][:, :, 0], d["C"][:, :, 0], Dd,
                             d["init_state"].reshape(Bz, H * P, N))
    np.testing.assert_allclose(yd.reshape(y.shape), y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hd.reshape(h.shape), h, rtol=1e-12, atol=1e-13)


def test_diag_lfilter_constant_dt():
    signal = pytest.importorskip("scipy.signal")
    d = inputs.diag_inputs(1, 40, 3, 4, io_dtype="f32", seed=9, init_state=True)
    dtc = np.array([0.01, 0.1, 0.5])
    dt = np.broadcast_to(dtc, d["dt"].shape).copy()
    A = d["A"] * np.array([1.0, 0.3, 2.0])[:, None]   # distinct per-channel, per-state poles
    y, hT = oracle.diag_seq(d["x"], dt, A, d["B"], d["C"], d["D"], d["init_state"])
    for ch in range(3):
        hs = np.zeros((40, 4))
        for n in range(4):
            alpha = math.exp(dtc[ch] * A[ch, n])
            u = dtc[ch] * d["x"][0, :, ch] * d["B"][0, :, n]
            hs[:, n], _ = signal.lfilter([1.0], [1.0, -alpha], u, zi=[alpha * d["init_state"][0, ch, n]])
        ref = np.einsum("tn,tn->t", d["C"][0], hs) + d["D"][ch] * d["x"][0, :, ch]
        np.testing.assert_allclose(y[0, :, ch], ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hT[0, ch], hs[-1], rtol=1e-11, atol=1e-12)


def test_diag_single_token_and_dt_zero():
    d = inputs.diag_inputs(2, 1, 5, 3, io_dtype="f32", seed=2)
    y, h = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    ref = (d["dt"][:, 0] * d["x"][:, 0] * np.einsum("bn,bn->b", d["C"][:, 0], d["B"][:, 0])[:, None]
           + d["D"][None] * d["x"][:, 0])
    np.testing.assert_allclose(y[:, 0], ref, rtol=1e-13, atol=1e-14)
    d2 = inputs.diag_inputs(1, 9, 4, 3, io_dtype="f32", seed=2, init_state=True)
    y2, h2 = oracle.diag_seq(d2["x"], np.zeros_like(d2["dt"]), d2["A"], d2["B"], d2["C"], d2["D"],
                             d2["init_state"])
    np.testing.assert_array_equal(h2, d2["init_state"])
    ref2 = np.einsum("btn,bdn->btd", d2["C"], d2["init_state"]) + d2["D"][None, None] * d2["x"]
    np.testing.assert_allclose(y2, ref2, rtol=1e-12, atol=1e-13)


def _diag_opt_inputs(seed, L=30, Dm=5, N=4):
    d = inputs.diag_inputs(2, L, Dm, N, io_dtype="f32", seed=seed, init_state=True)
    rng = np.random.default_rng(seed + 100)
    raw = rng.normal(-2.0, 1.5, size=d["dt"].shape)      # pre-activation steps, mostly negative
    bias = rng.uniform(-3.0, 1.0, size=Dm)
    z = rng.normal(0.0, 2.0, size=d["x"].shape)
    return d, raw, bias, z


def test_diag_delta_bias_and_softplus_reduce_to_transformed_dt():
    """delta_bias then softplus equals the plain scan fed softplus(dt + bias),
    with softplus taken from numpy (logaddexp(0, v) = log(1 + e^v))."""
    d, raw, bias, _ = _diag_opt_inputs(21)
    base = (d["A"], d["B"], d["C"], d["D"])
    for sp in (False, True):
        for b in (None, bias):
            v = raw + (0.0 if b is None else b[None, None, :])
            want = np.logaddexp(0.0, v) if sp else v
            y1, h1 = oracle.diag_seq(d["x"], raw, *base, d["init_state"], delta_bias=b, delta_softplus=sp)
            y2, h2 = oracle.diag_seq(d["x"], want, *base, d["init_state"])
            np.testing.assert_allclose(y1, y2, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(h1, h2, rtol=1e-13, atol=1e-14)


def test_diag_softplus_of_large_steps():
    """softplus(v) -> v for large v and -> e^v for very negative v: the scan
    with softplus matches the plain scan fed v (or e^v) there."""
    d = inputs.diag_inputs(1, 12, 3, 4, io_dtype="f32", seed=5, init_state=True)
    big = np.full(d["dt"].shape, 40.0)
    y1, h1 = oracle.diag_seq(d["x"], big, d["A"] * 1e-3, d["B"], d["C"], d["D"], d["init_state"], delta_softplus=True)
    y2, h2 = oracle.diag_seq(d["x"], big, d["A"] * 1e-3, d["B"], d["C"], d["D"], d["init_state"])
    np.testing.assert_allclose(y1, y2, rtol=1e-13, atol=1e-14)
    tiny = np.full(d["dt"].shape, -30.0)
    y3, h3 = oracle.diag_seq(d["x"], tiny, d["A"], d["B"], d["C"], d["D"], d["init_state"], delta_softplus=True)
    y4, h4 = oracle.diag_seq(d["x"], np.exp(tiny), d["A"], d["B"], d["C"], d["D"], d["init_state"])
    np.testing.assert_allclose(y3, y4, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(h3, h4, rtol=1e-12, atol=1e-14)


def test_diag_z_gate_is_silu_of_z():
    """The gate multiplies the finished output (D term included) by
    z * sigmoid(z), sigmoid from scipy; the state is not gated."""
    special = pytest.importorskip("scipy.special")
    d, raw, bias, z = _diag_opt_inputs(33)
    args = (d["x"], raw, d["A"], d["B"], d["C"], d["D"], d["init_state"])
    yg, hg = oracle.diag_seq(*args, z=z, delta_bias=bias, delta_softplus=True)
    y0, h0 = oracle.diag_seq(*args, delta_bias=bias, delta_softplus=True)
    np.testing.assert_allclose(yg, y0 * z * special.expit(z), rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(hg, h0)


def test_diag_options_single_token_closed_form():
    """L = 1, zero state: out = (s x (C.B) + D x) * z * sigmoid(z) with
    s = softplus(dt + bias), written out by hand."""
    d, raw, bias, z = _diag_opt_inputs(8, L=1, Dm=4, N=3)
    y, h = oracle.diag_seq(d["x"], raw, d["A"], d["B"], d["C"], d["D"], z=z, delta_bias=bias, delta_softplus=True)
    for b in range(2):
        cb = sum(d["C"][b, 0, n] * d["B"][b, 0, n] for n in range(3))
        for ch in range(4):
            s_ = math.log1p(math.exp(raw[b, 0, ch] + bias[ch]))
            xv, zv = d["x"][b, 0, ch], z[b, 0, ch]
            ref = (s_ * xv * cb + d["D"][ch] * xv) * zv / (1.0 + math.exp(-zv))
            assert abs(y[b, 0, ch] - ref) <= 1e-13 * max(1.0, abs(ref))
            for n in range(3):
                assert abs(h[b, ch, n] - s_ * xv * d["B"][b, 0, n]) <= 1e-14 * max(1.0, abs(h[b, ch, n]))


def test_conv_step_sequence_is_numpy_convolve():
    """T causal conv steps from a zero window equal the causal convolution of
    the input sequence with the reversed taps (numpy.convolve), plus bias;
    silu on top equals v * sigmoid(v) with scipy's sigmoid."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(40)
    Bz, C, W, T = 2, 5, 4, 23
    xs = rng.standard_normal((T, Bz, C))
    w = rng.standard_normal((C, W))
    bias = rng.standard_normal(C)
    for silu in (False, True):
        st = np.zeros((Bz, C, W))
        outs = np.stack([oracle.conv1d_step(st, xs[t], w, bias, silu=silu) for t in range(T)])
        for b in range(Bz):
            for c in range(C):
                ref = np.convolve(xs[:, b, c], w[c, ::-1])[:T] + bias[c]
                if silu:
                    ref = ref * special.expit(ref)
                np.testing.assert_allclose(outs[:, b, c], ref, rtol=1e-13, atol=1e-14)
        # the window keeps the last W inputs, oldest first
        np.testing.assert_array_equal(st, np.moveaxis(xs[T - W:], 0, -1))


def test_conv_step_continues_from_its_window():
    """A window filled by earlier steps makes the next outputs those of the
    unsplit sequence (numpy.convolve over the concatenation)."""
    rng = np.random.default_rng(41)
    C, W, T0, T1 = 3, 3, 7, 9
    xs = rng.standard_normal((T0 + T1, 1, C))
    w = rng.standard_normal((C, W))
    st = np.zeros((1, C, W))
    for t in range(T0):
        oracle.conv1d_step(st, xs[t], w, None, silu=False)
    outs = np.stack([oracle.conv1d_step(st, xs[T0 + t], w, None, silu=False) for t in range(T1)])
    for c in range(C):
        ref = np.convolve(xs[:, 0, c], w[c, ::-1])[T0:T0 + T1]
        np.testing.assert_allclose(outs[:, 0, c], ref, rtol=1e-13, atol=1e-14)


def test_gated_rmsnorm_invariants():
    """With unit weights and eps = 0 every group of the output has RMS 1; the
    output is invariant to scaling y; groups are independent; a gate of +40
    (silu(40) = 40 to 1e-17) is no gate at all; a zero gate gives zero."""
    rng = np.random.default_rng(42)
    Bz, D, grp = 3, 24, 8
    y = rng.standard_normal((Bz, D))
    z = rng.standard_normal((Bz, D))
    one = np.ones(D)
    out = oracle.gated_rmsnorm(y, z, one, grp, eps=0.0)
    rms = np.sqrt((out.reshape(Bz, D // grp, grp) ** 2).mean(-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.gated_rmsnorm(7.5 * y, z, one, grp, eps=0.0), out, rtol=1e-13, atol=1e-14)
    part = oracle.gated_rmsnorm(y[:, 8:16], z[:, 8:16], one[8:16], grp, eps=0.0)
    np.testing.assert_allclose(part, out[:, 8:16], rtol=1e-13, atol=1e-14)
    w = rng.standard_normal(D)
    np.testing.assert_allclose(oracle.gated_rmsnorm(y, np.full((Bz, D), 40.0), w, grp, eps=1e-5),
                               oracle.gated_rmsnorm(40.0 * y, None, w, grp, eps=1e-5), rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(oracle.gated_rmsnorm(y, np.zeros((Bz, D)), w, grp, eps=1e-5), 0.0)


def test_gated_rmsnorm_gate_ratio_and_eps():
    """y = 1 everywhere: outputs are proportional to silu(z) = z * sigmoid(z)
    (scipy's sigmoid); and eps enters as sqrt(mean(g^2) + eps)."""
    special = pytest.importorskip("scipy.special")
    z = np.array([[0.7, -1.3, 2.2, 0.1]])
    out = oracle.gated_rmsnorm(np.ones((1, 4)), z, np.ones(4), eps=0.0)
    s_ = z * special.expit(z)
    np.testing.assert_allclose(out / out[0, 0], s_ / s_[0, 0], rtol=1e-13)
    # one channel: out = y / sqrt(y^2 + eps)
    for yv, eps in ((0.3, 0.5), (2.0, 1e-5)):
        o = oracle.gated_rmsnorm(np.array([[yv]]), None, np.ones(1), eps=eps)
        assert abs(o[0, 0] - yv / math.sqrt(yv * yv + eps)) <= 1e-15


def test_decode_layer_matches_conv_then_prefill_then_norm():
    """T decode-layer steps from zero states equal the whole-sequence
    pipeline built from other pinned pieces: numpy's causal convolution of
    xBC with silu, the SSD prefill oracle on the split x | B | C, and the
    gated norm of each token."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(43)
    Bz, H, P, N, G, W, T = 2, 4, 3, 5, 2, 4, 11
    Cc = H * P + 2 * G * N
    xBC = rng.standard_normal((T, Bz, Cc))
    cw, cb = rng.standard_normal((Cc, W)) * 0.5, rng.standard_normal(Cc) * 0.1
    dt = np.exp(rng.uniform(np.log(1e-2), np.log(0.3), size=(T, Bz, H)))
    A = -np.exp(rng.uniform(0, np.log(8), size=H))
    Dv = rng.uniform(0.5, 1.5, size=H)
    z = rng.standard_normal((T, Bz, H * P))
    nw = rng.uniform(0.5, 1.5, size=H * P)
    cst, sst = np.zeros((Bz, Cc, W)), np.zeros((Bz, H, P, N))
    outs = np.stack([oracle.decode_layer_step(cst, sst, xBC[t], cw, cb, dt[t], A, Dv, z[t], nw, H, P, N, G,
                                              group=P * 2, eps=1e-5) for t in range(T)])
    conv = np.empty_like(xBC)
    for b in range(Bz):
        for c in range(Cc):
            v = np.convolve(xBC[:, b, c], cw[c, ::-1])[:T] + cb[c]
            conv[:, b, c] = v * special.expit(v)
    x = np.moveaxis(conv[:, :, :H * P], 0, 1).reshape(Bz, T, H, P)
    Bm = np.moveaxis(conv[:, :, H * P:H * P + G * N], 0, 1).reshape(Bz, T, G, N)
    Cm = np.moveaxis(conv[:, :, H * P + G * N:], 0, 1).reshape(Bz, T, G, N)
    y, hT = oracle.ssd_seq(x, np.moveaxis(dt, 0, 1), A, Bm, Cm, Dv)
    for t in range(T):
        ref = oracle.gated_rmsnorm(y[:, t].reshape(Bz, H * P), z[t], nw, P * 2, eps=1e-5)
        np.testing.assert_allclose(outs[t], ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sst, hT, rtol=1e-11, atol=1e-13)


def _fd_case(L, seed):
    d = inputs.ssd_inputs(2, L, 4, 3, 5, 2, io_dtype="f32", seed=seed, init_state=True)
    rng = np.random.default_rng(seed + 7)
    dy = rng.standard_normal(d["x"].shape)
    dfin = rng.standard_normal(d["init_state"].shape)
    return d, dy, dfin


def _objective(d, dy, dfin, **over):
    a = {k: over.get(k, d[k]) for k in ("x", "dt", "A", "B", "C", "D", "init_state")}
    y, hT = oracle.ssd_seq(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["init_state"])
    return float(np.sum(dy * y) + np.sum(dfin * hT))


@pytest.mark.parametrize("L,sample", [(9, None), (70, 40)])
def test_backward_matches_central_differences(L, sample):
    """Every gradient of L = <dy, y> + <dfinal, h_T> against central finite
    differences of the forward oracle (step 1e-6 in float64: truncation
    ~1e-12, rounding ~1e-10), at a length that stays inside one 64-token
    checkpoint and one that crosses it; two B/C groups of two heads."""
    d, dy, dfin = _fd_case(L, 30 + L)
    g = oracle.ssd_seq_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"], d["init_state"], dfin)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init_state": "dinit"}
    rng = np.random.default_rng(L)
    eps = 1e-6
    for k, gk in names.items():
        base = np.array(d[k], dtype=np.float64)
        flat = np.arange(base.size) if sample is None else rng.choice(base.size, min(sample, base.size), False)
        for i in flat:
            plus, minus = base.copy(), base.copy()
            plus.flat[i] += eps
            minus.flat[i] -= eps
            fd = (_objective(d, dy, dfin, **{k: plus}) - _objective(d, dy, dfin, **{k: minus})) / (2 * eps)
            got = g[gk].flat[i]
            assert abs(got - fd) <= 1e-6 * max(1.0, abs(fd)), f"{gk}[{i}]: {got} vs finite difference {fd}"


def test_backward_linearity_in_cotangents():
    """Gradients are linear in (dy, dfinal): the sum of the gradients for two
    cotangents is the gradient for their sum; a zero cotangent gives zeros."""
    d, dy, dfin = _fd_case(20, 5)
    args = (d["x"], d["dt"], d["A"], d["B"], d["C"])
    g1 = oracle.ssd_seq_bwd(*args, dy, d["D"], d["init_state"], None)
    g2 = oracle.ssd_seq_bwd(*args, np.zeros_like(dy), d["D"], d["init_state"], dfin)
    g12 = oracle.ssd_seq_bwd(*args, dy, d["D"], d["init_state"], dfin)
    for k in g12:
        np.testing.assert_allclose(g1[k] + g2[k], g12[k], rtol=1e-12, atol=1e-12)
    g0 = oracle.ssd_seq_bwd(*args, np.zeros_like(dy), d["D"], d["init_state"], None)
    for k in g0:
        assert not np.any(g0[k]), k


def test_diag_split_resume():
    d = inputs.diag_inputs(2, 50, 6, 4, io_dtype="f32", seed=12, init_state=True)
    yf, hf = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    y1, h1 = oracle.diag_seq(d["x"][:, :17], d["dt"][:, :17], d["A"], d["B"][:, :17], d["C"][:, :17], d["D"],
                             d["init_state"])
    y2, h2 = oracle.diag_seq(d["x"][:, 17:], d["dt"][:, 17:], d["A"], d["B"][:, 17:], d["C"][:, 17:], d["D"], h1)
    np.testing.assert_allclose(np.concatenate([y1, y2], 1), yf, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h2, hf, rtol=1e-12, atol=1e-13)


def test_empty_sequence_returns_initial_state():
    d = _small(L=0)
    y, h = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    assert y.shape[1] == 0
    np.testing.assert_array_equal(h, d["init_state"])
