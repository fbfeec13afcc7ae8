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
        for f in (lib.oracle_ssd_seq, lib.oracle_ssd_decode, lib.oracle_diag_seq, lib.oracle_diag_seq_ex):
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
