"""Float64 CPU oracle for the SSD selective scan, its decode step and the
Mamba-1 diagonal scan.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it; the product path never does. It shares
no code with the CUDA library (``mamba_ssd_selective_gb300``) and imports
nothing from it.

Two independent formulations live here:

* ``ssd_oracle.c`` -- the token-by-token recurrence (the plain definition),
  compiled with gcc and called through ctypes: :func:`ssd_seq`,
  :func:`ssd_decode`, :func:`diag_seq`.
* ``quadratic.py`` -- the masked "attention" (quadratic) form of the same SSD
  scan, numpy float64, for tiny inputs: :func:`ssd_quadratic`.

Every function is pinned by ``tests/test_oracle_pins.py`` against closed forms,
a library IIR filter, brute-force expansions and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .quadratic import ssd_quadratic  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libssd_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math, no reassociation)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, dp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_ssd_seq.argtypes = [i64] * 6 + [dp] * 9 + [ci]
        lib.oracle_ssd_decode.argtypes = [i64] * 5 + [dp] * 8 + [ci]
        lib.oracle_diag_seq.argtypes = [i64] * 4 + [dp] * 9 + [ci]
        lib.oracle_diag_seq_ex.argtypes = [i64] * 4 + [dp] * 8 + [ci] + [dp] * 3 + [ci]
        lib.oracle_conv1d_step.argtypes = [i64] * 3 + [dp] * 4 + [ci, dp]
        lib.oracle_ssd_seq_bwd.argtypes = [i64] * 6 + [dp] * 16 + [ci]
        lib.oracle_gated_rmsnorm.argtypes = [i64] * 3 + [dp] * 3 + [ctypes.c_double, dp]
        for f in (lib.oracle_ssd_seq, lib.oracle_ssd_decode, lib.oracle_diag_seq, lib.oracle_diag_seq_ex,
                  lib.oracle_conv1d_step, lib.oracle_gated_rmsnorm, lib.oracle_ssd_seq_bwd):
            f.restype = ci
        _lib = lib
    return _lib


def _f64(a, shape=None, name="array"):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def ssd_seq(x, dt, A, B, C, D=None, init_state=None, threads=None):
    """Token-by-token SSD recurrence in float64.

    x[B,L,H,P], dt[B,L,H], A[H], B/C[B,L,G,N], D[H] or None,
    init_state[B,H,P,N] or None. Returns (y[B,L,H,P], final_state[B,H,P,N]).
    """
    x = _f64(x)
    Bsz, L, H, P = x.shape
    G, N = np.shape(B)[2], np.shape(B)[3]
    dt = _f64(dt, (Bsz, L, H), "dt")
    A = _f64(A, (H,), "A")
    Bm = _f64(B, (Bsz, L, G, N), "B")
    Cm = _f64(C, (Bsz, L, G, N), "C")
    D = _f64(D, (H,), "D")
    h0 = _f64(init_state, (Bsz, H, P, N), "init_state")
    y = np.empty((Bsz, L, H, P))
    hT = np.empty((Bsz, H, P, N))
    rc = _load().oracle_ssd_seq(Bsz, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                _ptr(D), _ptr(h0), _ptr(y), _ptr(hT), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_ssd_seq: invalid sizes")
    return y, hT


def ssd_decode(state, x, dt, A, B, C, D=None, threads=None):
    """One decode token in float64. state[B,H,P,N] is NOT modified: the new
    state is returned. x[B,H,P], dt[B,H], B/C[B,G,N]. Returns (y[B,H,P], state')."""
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    Bsz, H, P, N = st.shape
    G = np.shape(B)[1]
    x = _f64(x, (Bsz, H, P), "x")
    dt = _f64(dt, (Bsz, H), "dt")
    A = _f64(A, (H,), "A")
    Bm = _f64(B, (Bsz, G, N), "B")
    Cm = _f64(C, (Bsz, G, N), "C")
    D = _f64(D, (H,), "D")
    y = np.empty((Bsz, H, P))
    rc = _load().oracle_ssd_decode(Bsz, H, P, N, G, _ptr(st), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm),
                                   _ptr(Cm), _ptr(D), _ptr(y), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_ssd_decode: invalid sizes")
    return y, st


def diag_seq(x, dt, A, B, C, D=None, init_state=None, threads=None, z=None, delta_bias=None,
             delta_softplus=False):
    """Mamba-1 diagonal recurrence in float64.

    x/dt[B,L,Dm], A[Dm,N], B/C[B,L,N], D[Dm] or None, init_state[B,Dm,N] or
    None. Options of selective_scan_fn: delta_bias[Dm] is added to dt, then
    with delta_softplus the step is softplus of the sum; z[B,L,Dm] gates the
    output by silu(z). Returns (y[B,L,Dm], final_state[B,Dm,N]).
    """
    x = _f64(x)
    Bsz, L, Dm = x.shape
    N = np.shape(A)[1]
    dt = _f64(dt, (Bsz, L, Dm), "dt")
    A = _f64(A, (Dm, N), "A")
    Bm = _f64(B, (Bsz, L, N), "B")
    Cm = _f64(C, (Bsz, L, N), "C")
    D = _f64(D, (Dm,), "D")
    z = _f64(z, (Bsz, L, Dm), "z")
    db = _f64(delta_bias, (Dm,), "delta_bias")
    h0 = _f64(init_state, (Bsz, Dm, N), "init_state")
    y = np.empty((Bsz, L, Dm))
    hT = np.empty((Bsz, Dm, N))
    rc = _load().oracle_diag_seq_ex(Bsz, L, Dm, N, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                    _ptr(z), _ptr(db), int(bool(delta_softplus)), _ptr(h0), _ptr(y), _ptr(hT),
                                    threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_diag_seq: invalid sizes")
    return y, hT


def conv1d_step(state, x, w, bias=None, silu=True):
    """One causal depthwise convolution step in float64.

    state[B,C,W] (the last W inputs, oldest first) is updated in place (it
    must be a float64 C-contiguous array); x[B,C], w[C,W], bias[C] or None.
    Returns out[B,C] = act(sum_k w[c,k] * window[k] + bias[c]).
    """
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64 and state.flags.c_contiguous):
        raise TypeError("state must be a C-contiguous float64 array (updated in place)")
    Bsz, C, W = state.shape
    x = _f64(x, (Bsz, C), "x")
    w = _f64(w, (C, W), "w")
    bias = _f64(bias, (C,), "bias")
    out = np.empty((Bsz, C))
    if _load().oracle_conv1d_step(Bsz, C, W, _ptr(state), _ptr(x), _ptr(w), _ptr(bias), int(bool(silu)),
                                  _ptr(out)) != 0:
        raise ValueError("oracle_conv1d_step: invalid sizes")
    return out


def gated_rmsnorm(y, z, w, group=None, eps=1e-5):
    """Gated RMS norm in float64: g = y * silu(z) (z None: g = y), then per
    group of `group` channels (default: all) g / sqrt(mean(g^2) + eps) * w."""
    y = _f64(y)
    Bsz, D = y.shape
    z = _f64(z, (Bsz, D), "z")
    w = _f64(w, (D,), "w")
    group = D if group is None else int(group)
    out = np.empty((Bsz, D))
    if _load().oracle_gated_rmsnorm(Bsz, D, group, _ptr(y), _ptr(z), _ptr(w), float(eps), _ptr(out)) != 0:
        raise ValueError("oracle_gated_rmsnorm: invalid sizes")
    return out


def decode_layer_step(conv_state, ssm_state, xBC, conv_w, conv_b, dt, A, D, z, norm_w, nheads, headdim, dstate,
                      ngroups, group=None, eps=1e-5):
    """One token of the Mamba-2 decode layer body in float64, states updated
    in place: xBC <- silu(causal conv step of xBC); x, B, C = split(xBC)
    (H*P, G*N, G*N channels); y = SSD decode step; out = gated RMS norm of y
    with gate z. conv_state[B,Cc,W], ssm_state[B,H,P,N] float64 arrays."""
    Bsz = xBC.shape[0]
    H, P, N, G = nheads, headdim, dstate, ngroups
    xc = conv1d_step(conv_state, xBC, conv_w, conv_b, silu=True)
    x = xc[:, :H * P].reshape(Bsz, H, P)
    Bm = xc[:, H * P:H * P + G * N].reshape(Bsz, G, N)
    Cm = xc[:, H * P + G * N:].reshape(Bsz, G, N)
    y, st = ssd_decode(ssm_state, x, dt, A, Bm, Cm, D)
    ssm_state[...] = st
    return gated_rmsnorm(y.reshape(Bsz, H * P), z, norm_w, group, eps)


def ssd_seq_bwd(x, dt, A, B, C, dy, D=None, init_state=None, dfinal=None, threads=None):
    """Gradients of the SSD scan in float64 by reverse-mode differentiation of
    the token loop, for output cotangent dy[B,L,H,P] and final-state cotangent
    dfinal[B,H,P,N] (None: 0). Returns dict dx, ddt, dA, dB, dC, dD, dinit."""
    x = _f64(x)
    Bsz, L, H, P = x.shape
    G, N = np.shape(B)[2], np.shape(B)[3]
    dt = _f64(dt, (Bsz, L, H), "dt")
    A = _f64(A, (H,), "A")
    Bm = _f64(B, (Bsz, L, G, N), "B")
    Cm = _f64(C, (Bsz, L, G, N), "C")
    D = _f64(D, (H,), "D")
    h0 = _f64(init_state, (Bsz, H, P, N), "init_state")
    dy = _f64(dy, (Bsz, L, H, P), "dy")
    dfinal = _f64(dfinal, (Bsz, H, P, N), "dfinal")
    out = dict(dx=np.empty((Bsz, L, H, P)), ddt=np.empty((Bsz, L, H)), dA=np.empty(H),
               dB=np.empty((Bsz, L, G, N)), dC=np.empty((Bsz, L, G, N)), dD=np.empty(H),
               dinit=np.empty((Bsz, H, P, N)))
    rc = _load().oracle_ssd_seq_bwd(Bsz, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                    _ptr(h0), _ptr(dy), _ptr(dfinal), _ptr(out["dx"]), _ptr(out["ddt"]),
                                    _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                                    _ptr(out["dinit"]), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_ssd_seq_bwd: invalid sizes")
    return out
