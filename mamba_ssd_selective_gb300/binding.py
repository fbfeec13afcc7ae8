"""Thin Python binding of libssdscan.so (C ABI in include/ssd_scan.h).

Argument marshalling only: checks that torch tensors have the documented
shapes, dtypes, device and layout (the C ABI receives raw pointers and cannot),
allocates outputs and the workspace with torch when the caller passes none,
and forwards pointers plus the current CUDA stream. Every step of the scan
runs in the library's CUDA kernels; there is no fallback. If the library has
not been built, or does not load, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_TIMEOUT, SSD_ERR_BOUNDS = 0, 1, 2, 3, 4, 5
SSD_F32, SSD_BF16 = 0, 1
SSD_FLAG_SIMT = 1
SSD_FLAG_FUSED = 2
SSD_FLAG_STAGED = 4
PATH_NAMES = {0: "simt", 1: "staged", 2: "fused"}
_PATH_FLAGS = {None: 0, "auto": 0, "simt": SSD_FLAG_SIMT, "fused": SSD_FLAG_FUSED, "staged": SSD_FLAG_STAGED}

_STATUS_NAMES = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_CUDA",
                 4: "SSD_ERR_TIMEOUT", 5: "SSD_ERR_BOUNDS"}


class SsdError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class ssd_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    """The library this process loads: the bounds-checked debug build when the
    environment sets SSD_DEBUG_BOUNDS_LIB=1, else the release build."""
    return _build.DBG_LIB_PATH if os.environ.get("SSD_DEBUG_BOUNDS_LIB") == "1" else _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Loads libssdscan.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m mamba_ssd_selective_gb300.build` (or __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
            dp = ctypes.POINTER(ssd_dims)
            lib.ssd_workspace_size.argtypes = [dp, ctypes.c_int]
            lib.ssd_workspace_size.restype = sz
            lib.ssd_best_chunk.argtypes = [dp]
            lib.ssd_best_chunk.restype = ctypes.c_int
            lib.ssd_scan_path.argtypes = [dp, ctypes.c_int]
            lib.ssd_scan_path.restype = ctypes.c_int
            lib.ssd_scan_chunked_bwd_workspace_size.argtypes = [dp]
            lib.ssd_scan_chunked_bwd_workspace_size.restype = sz
            lib.ssd_scan_chunked_bwd.argtypes = [dp] + [vp] * 17 + [sz, vp]
            lib.ssd_scan_chunked_bwd.restype = ctypes.c_int
            f32 = ctypes.c_float
            lib.ssd_conv1d_step.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, i32, vp, vp]
            lib.ssd_gated_rmsnorm.argtypes = [i64, i64, i64, i32, vp, vp, vp, f32, vp, vp]
            lib.ssd_decode_layer_workspace_size.argtypes = [dp]
            lib.ssd_decode_layer_workspace_size.restype = sz
            lib.ssd_decode_layer_step.argtypes = [dp, i64] + [vp] * 10 + [i64, f32, vp, vp, sz, vp]
            lib.ssd_decode_graph_create.argtypes = [dp, i64, i32] + [vp] * 10 + [i64, f32, vp, vp, sz,
                                                                                 ctypes.POINTER(vp)]
            lib.ssd_decode_graph_launch.argtypes = [vp, vp]
            lib.ssd_decode_graph_destroy.argtypes = [vp]
            for f in (lib.ssd_conv1d_step, lib.ssd_gated_rmsnorm, lib.ssd_decode_layer_step,
                      lib.ssd_decode_graph_create, lib.ssd_decode_graph_launch, lib.ssd_decode_graph_destroy):
                f.restype = ctypes.c_int
            lib.ssd_scan_chunked.argtypes = [dp] + [vp] * 7 + [ctypes.c_int, vp, vp, vp, sz, vp]
            lib.ssd_scan_chunked_noalloc.argtypes = [dp] + [vp] * 7 + [ctypes.c_int, vp, vp, vp]
            lib.ssd_scan_chunked_noalloc.restype = ctypes.c_int
            lib.ssd_scan_chunked_noalloc_status.argtypes = [vp, ctypes.POINTER(vp)]
            lib.ssd_scan_chunked_noalloc_status.restype = ctypes.c_int
            lib.ssd_decode_step.argtypes = [dp] + [vp] * 9
            lib.selective_scan_diag.argtypes = [i64, i64, i64, i64, i32] + [vp] * 7 + [ctypes.c_int, vp, vp, vp]
            lib.selective_scan_diag_ex.argtypes = ([i64, i64, i64, i64, i32] + [vp] * 8 + [i32, vp, ctypes.c_int]
                                                   + [vp] * 3 + [sz, vp])
            lib.selective_scan_diag_workspace_size.argtypes = [i64, i64, i64, i64, i32]
            lib.selective_scan_diag_workspace_size.restype = sz
            lib.ssd_workspace_status.argtypes = [vp, vp]
            lib.ssd_selftest_bounded_wait.argtypes = [vp, ctypes.c_int, vp]
            lib.ssd_debug_bounds_status.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int64),
                                                    ctypes.c_int]
            lib.ssd_debug_bounds_status.restype = ctypes.c_int
            lib.ssd_record_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
            lib.ssd_record_stage_events.restype = ctypes.c_int
            lib.ssd_last_error.argtypes = []
            lib.ssd_last_error.restype = ctypes.c_char_p
            for f in (lib.ssd_scan_chunked, lib.ssd_decode_step, lib.selective_scan_diag, lib.selective_scan_diag_ex,
                      lib.ssd_workspace_status,
                      lib.ssd_selftest_bounded_wait):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != SSD_OK:
        raise SsdError(status, load().ssd_last_error().decode())


def _io_code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return SSD_F32
    if dtype == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"io dtype must be float32 or bfloat16, got {dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected dtype {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(Bsz, L, H, P, N, G, io, flags=0) -> ssd_dims:
    return ssd_dims(Bsz, L, H, P, N, G, io, flags)


def ssd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups, io_dtype, chunk_size) -> int:
    d = _dims(batch, seqlen, nheads, headdim, dstate, ngroups, _io_code(io_dtype))
    return int(load().ssd_workspace_size(ctypes.byref(d), int(chunk_size)))


def ssd_best_chunk(batch, seqlen, nheads, headdim, dstate, ngroups, io_dtype) -> int:
    """Chunk size of the library's static policy for these sizes (0: invalid)."""
    d = _dims(batch, seqlen, nheads, headdim, dstate, ngroups, _io_code(io_dtype))
    return int(load().ssd_best_chunk(ctypes.byref(d)))


def ssd_scan_path(batch, seqlen, nheads, headdim, dstate, ngroups, io_dtype, chunk_size, path=None) -> str:
    """Name of the kernel path ("simt", "staged", "fused") ssd_scan_chunked
    takes for these sizes on the current device."""
    d = _dims(batch, seqlen, nheads, headdim, dstate, ngroups, _io_code(io_dtype), _PATH_FLAGS[path])
    code = int(load().ssd_scan_path(ctypes.byref(d), int(chunk_size)))
    if code < 0:
        raise SsdError(SSD_ERR_INVALID_ARG, "invalid sizes, chunk size or path for ssd_scan_path")
    return PATH_NAMES[code]


def ssd_scan_chunked(x, dt, A, B, C, D=None, init_state=None, chunk_size=None, y=None, final_state=None,
                     workspace=None, stream=None, simt=False, want_final_state=True, path=None):
    """Chunked SSD prefill. x[B,L,H,P], dt[B,L,H], B/C[B,L,G,N] (float32 or
    bfloat16), A[H], D[H], init_state[B,H,P,N] (float32). chunk_size None takes
    the library's static policy (ssd_best_chunk). `path` forces a kernel path
    for bf16 inputs: "fused" (single pass, chunk 128), "staged" (three
    tensor-core kernels), "simt" (CUDA cores); None lets the library choose.
    Returns (y, final_state)."""
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [B,L,H,P] and B, C [B,L,G,N]")
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev, io = x.device, x.dtype
    _need(x, "x", (Bsz, L, H, P), io, dev)
    _need(dt, "dt", (Bsz, L, H), io, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(B, "B", (Bsz, L, G, N), io, dev)
    _need(C, "C", (Bsz, L, G, N), io, dev)
    _need(D, "D", (H,), torch.float32, dev)
    _need(init_state, "init_state", (Bsz, H, P, N), torch.float32, dev)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", (Bsz, L, H, P), io, dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((Bsz, H, P, N), dtype=torch.float32, device=dev)
    _need(final_state, "final_state", (Bsz, H, P, N), torch.float32, dev)
    if path not in _PATH_FLAGS:
        raise ValueError(f"path must be one of {sorted(k for k in _PATH_FLAGS if k)} or None, got {path!r}")
    d = _dims(Bsz, L, H, P, N, G, _io_code(io), SSD_FLAG_SIMT if simt else _PATH_FLAGS[path])
    lib = load()
    if chunk_size is None:
        chunk_size = int(lib.ssd_best_chunk(ctypes.byref(d))) or 128
    ws_bytes = int(lib.ssd_workspace_size(ctypes.byref(d), int(chunk_size)))
    if ws_bytes == 0:
        _check(lib.ssd_scan_chunked(ctypes.byref(d), None, None, None, None, None, None, None, int(chunk_size),
                                    None, None, None, 0, None))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    elif workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace too small: {workspace.numel() * workspace.element_size()} < {ws_bytes}")
    _check(lib.ssd_scan_chunked(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(init_state), int(chunk_size), _ptr(y), _ptr(final_state), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream, dev)))
    return y, final_state


def ssd_scan_chunked_bwd(x, dt, A, B, C, dy, D=None, init_state=None, dfinal_state=None, workspace=None,
                         stream=None, want_dinit=True, simt=False):
    """Gradients of <dy, y> + <dfinal_state, final_state> for ssd_scan_chunked's
    inputs. Returns a dict of float32 tensors dx, ddt, dA, dB, dC, dD (None when
    D is None) and dinit (None unless want_dinit). simt=True keeps the
    per-chunk gradients on the CUDA cores where the tensor cores would take them."""
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [B,L,H,P] and B, C [B,L,G,N]")
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev, io = x.device, x.dtype
    _need(x, "x", (Bsz, L, H, P), io, dev)
    _need(dt, "dt", (Bsz, L, H), io, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(B, "B", (Bsz, L, G, N), io, dev)
    _need(C, "C", (Bsz, L, G, N), io, dev)
    _need(D, "D", (H,), torch.float32, dev)
    _need(init_state, "init_state", (Bsz, H, P, N), torch.float32, dev)
    _need(dy, "dy", (Bsz, L, H, P), io, dev)
    _need(dfinal_state, "dfinal_state", (Bsz, H, P, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty((Bsz, L, H, P), **f32), ddt=torch.empty((Bsz, L, H), **f32), dA=torch.empty(H, **f32),
             dB=torch.empty((Bsz, L, G, N), **f32), dC=torch.empty((Bsz, L, G, N), **f32),
             dD=torch.empty(H, **f32) if D is not None else None,
             dinit=torch.empty((Bsz, H, P, N), **f32) if want_dinit else None)
    d = _dims(Bsz, L, H, P, N, G, _io_code(io), SSD_FLAG_SIMT if simt else 0)
    lib = load()
    need = int(lib.ssd_scan_chunked_bwd_workspace_size(ctypes.byref(d)))
    if need == 0:
        _check(lib.ssd_scan_chunked_bwd(ctypes.byref(d), *[None] * 17, 0, None))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    _check(lib.ssd_scan_chunked_bwd(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                    _ptr(init_state), _ptr(dy), _ptr(dfinal_state), _ptr(g["dx"]), _ptr(g["ddt"]),
                                    _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dinit"]),
                                    _ptr(workspace), workspace.numel(), _stream(stream, dev)))
    return g


def ssd_scan_chunked_noalloc(x, dt, A, B, C, D=None, init_state=None, chunk_size=256, y=None, final_state=None,
                             stream=None, simt=False):
    """ssd_scan_chunked without a workspace argument: the per-chunk states go to
    the library's built-in 64 MiB device scratch, so the C call allocates
    nothing (for callers that cannot allocate where they run the scan, such as
    plug-ins whose framework owns all device memory). Such callers pass `y`
    and `final_state`; this wrapper allocates them only when they are None.
    The scan runs on x's device, which must be the current CUDA device: the
    library looks the scratch up on the current device. Returns (y, final_state)."""
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [B,L,H,P] and B, C [B,L,G,N]")
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev, io = x.device, x.dtype
    if dev.type != "cuda" or dev.index != torch.cuda.current_device():
        raise ValueError(f"ssd_scan_chunked_noalloc: x is on {dev}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}; the built-in scratch is per device")
    _need(dt, "dt", (Bsz, L, H), io, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(B, "B", (Bsz, L, G, N), io, dev)
    _need(C, "C", (Bsz, L, G, N), io, dev)
    _need(D, "D", (H,), torch.float32, dev)
    _need(init_state, "init_state", (Bsz, H, P, N), torch.float32, dev)
    _need(x, "x", (Bsz, L, H, P), io, dev)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None:
        final_state = torch.empty((Bsz, H, P, N), dtype=torch.float32, device=dev)
    _need(y, "y", (Bsz, L, H, P), io, dev)
    _need(final_state, "final_state", (Bsz, H, P, N), torch.float32, dev)
    d = _dims(Bsz, L, H, P, N, G, _io_code(io), SSD_FLAG_SIMT if simt else 0)
    _check(load().ssd_scan_chunked_noalloc(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                           _ptr(init_state), int(chunk_size), _ptr(y), _ptr(final_state),
                                           _stream(stream, dev)))
    return y, final_state


def ssd_scan_chunked_noalloc_status(stream=None):
    """Status code of the latest ssd_scan_chunked_noalloc call on the current
    device (waits for `stream`): SSD_OK or SSD_ERR_TIMEOUT. Also returns the
    built-in scratch's device address, as (status, address)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    addr = ctypes.c_void_p()
    rc = load().ssd_scan_chunked_noalloc_status(_stream(stream, dev), ctypes.byref(addr))
    return int(rc), addr.value


def ssd_decode_step(state, x, dt, A, B, C, D=None, y=None, stream=None):
    """One decode token; `state` [B,H,P,N] float32 is updated in place. Returns y[B,H,P]."""
    Bsz, H, P, N = state.shape
    G = B.shape[1]
    dev, io = x.device, x.dtype
    _need(state, "state", (Bsz, H, P, N), torch.float32, dev)
    _need(x, "x", (Bsz, H, P), io, dev)
    _need(dt, "dt", (Bsz, H), io, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(B, "B", (Bsz, G, N), io, dev)
    _need(C, "C", (Bsz, G, N), io, dev)
    _need(D, "D", (H,), torch.float32, dev)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", (Bsz, H, P), io, dev)
    d = _dims(Bsz, 1, H, P, N, G, _io_code(io))
    _check(load().ssd_decode_step(ctypes.byref(d), _ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                  _ptr(D), _ptr(y), _stream(stream, dev)))
    return y


def selective_scan_diag_workspace_size(batch, seqlen, dim, dstate, io_dtype) -> int:
    """Bytes of scratch selective_scan_diag needs for its time-segmented scan
    of this shape (0: one pass per sequence)."""
    return int(load().selective_scan_diag_workspace_size(batch, seqlen, dim, dstate, _io_code(io_dtype)))


def selective_scan_diag(x, dt, A, B, C, D=None, init_state=None, chunk_size=2048, y=None, final_state=None,
                        stream=None, want_final_state=True, z=None, delta_bias=None, delta_softplus=False,
                        workspace=None, segmented=True):
    """Mamba-1 diagonal scan. x/dt[B,L,D], A[D,N], B/C[B,L,N], D[D],
    init_state[B,D,N]; options of selective_scan_fn: z[B,L,D] (output gate
    silu(z)), delta_bias[D] and delta_softplus (dt <- softplus(dt + bias)).
    With segmented (default) the scratch of the time-segmented scan is taken
    from `workspace` (uint8, at least selective_scan_diag_workspace_size
    bytes) or allocated here; segmented=False runs one pass per sequence.
    Returns (y, final_state)."""
    Bsz, L, Dm = x.shape
    N = A.shape[1]
    dev, io = x.device, x.dtype
    _need(x, "x", (Bsz, L, Dm), io, dev)
    _need(dt, "dt", (Bsz, L, Dm), io, dev)
    _need(A, "A", (Dm, N), torch.float32, dev)
    _need(B, "B", (Bsz, L, N), io, dev)
    _need(C, "C", (Bsz, L, N), io, dev)
    _need(D, "D", (Dm,), torch.float32, dev)
    _need(z, "z", (Bsz, L, Dm), io, dev)
    _need(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _need(init_state, "init_state", (Bsz, Dm, N), torch.float32, dev)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", (Bsz, L, Dm), io, dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((Bsz, Dm, N), dtype=torch.float32, device=dev)
    _need(final_state, "final_state", (Bsz, Dm, N), torch.float32, dev)
    ws_bytes = 0
    if segmented:
        need = selective_scan_diag_workspace_size(Bsz, L, Dm, N, io) if Bsz > 0 and L > 0 else 0
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if workspace is not None:
            _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
            ws_bytes = workspace.numel()
    else:
        workspace = None
    _check(load().selective_scan_diag_ex(Bsz, L, Dm, N, _io_code(io), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                         _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
                                         _ptr(init_state), int(chunk_size), _ptr(y), _ptr(final_state),
                                         _ptr(workspace), ws_bytes, _stream(stream, dev)))
    return y, final_state


def ssd_workspace_status(workspace, stream=None) -> int:
    """Waits for the stream and returns the status word of a workspace (0 = OK)."""
    return int(load().ssd_workspace_status(_ptr(workspace), _stream(stream, workspace.device)))


def ssd_record_stage_events(events) -> None:
    """Arms per-stage timing of the next ssd_scan_chunked call on this thread.
    `events`: 4 torch.cuda.Event(enable_timing=True) that have been recorded
    once (so that the CUDA events exist), or None to cancel."""
    if events is None:
        _check(load().ssd_record_stage_events(None, 0))
        return
    arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(int(e.cuda_event)) for e in events])
    _check(load().ssd_record_stage_events(arr, len(events)))


def ssd_debug_bounds_status(clear=True):
    """(status, site, index) of the bounds checks of a debug build (see
    ssd_debug_bounds_status in ssd_scan.h); waits for the device."""
    site, index = ctypes.c_int(0), ctypes.c_int64(-1)
    rc = int(load().ssd_debug_bounds_status(ctypes.byref(site), ctypes.byref(index), 1 if clear else 0))
    return rc, site.value, index.value


def ssd_selftest_bounded_wait(workspace, spin_limit, stream=None) -> None:
    _check(load().ssd_selftest_bounded_wait(_ptr(workspace), int(spin_limit), _stream(stream, workspace.device)))


# ------------------------------------------------------- decode-layer pieces

def conv1d_step(x, conv_state, weight, bias=None, silu=True, out=None, stream=None):
    """Causal depthwise convolution step: x[B,C] shifts into the window
    conv_state[B,C,W] (float32, in place); returns act(weight . window + bias)."""
    Bsz, C = x.shape
    W = conv_state.shape[2]
    dev, io = x.device, x.dtype
    _need(conv_state, "conv_state", (Bsz, C, W), torch.float32, dev)
    _need(weight, "weight", (C, W), torch.float32, dev)
    _need(bias, "bias", (C,), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", (Bsz, C), io, dev)
    _check(load().ssd_conv1d_step(Bsz, C, W, _io_code(io), _ptr(x), _ptr(conv_state), _ptr(weight), _ptr(bias),
                                  1 if silu else 0, _ptr(out), _stream(stream, dev)))
    return out


def gated_rmsnorm(y, z, weight, group=None, eps=1e-5, out=None, stream=None):
    """out = g / sqrt(mean over each group of g^2 + eps) * weight, g = y * silu(z)."""
    Bsz, D = y.shape
    dev, io = y.device, y.dtype
    _need(z, "z", (Bsz, D), io, dev)
    _need(weight, "weight", (D,), torch.float32, dev)
    if out is None:
        out = torch.empty_like(y)
    _need(out, "out", (Bsz, D), io, dev)
    _check(load().ssd_gated_rmsnorm(Bsz, D, D if group is None else int(group), _io_code(io), _ptr(y), _ptr(z),
                                    _ptr(weight), float(eps), _ptr(out), _stream(stream, dev)))
    return out


def _layer_args(xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z, norm_weight, norm_group, out,
                workspace, steps=None):
    lead = () if steps is None else (steps,)
    Bsz, H, P, N = ssm_state.shape
    Cc = xBC.shape[-1]
    W = conv_state.shape[2]
    G = (Cc - H * P) // (2 * N)
    if G < 1 or H * P + 2 * G * N != Cc:
        raise ValueError(f"xBC has {Cc} channels; expected H*P + 2*G*N for some G")
    dev, io = xBC.device, xBC.dtype
    _need(xBC, "xBC", lead + (Bsz, Cc), io, dev)
    _need(conv_state, "conv_state", (Bsz, Cc, W), torch.float32, dev)
    _need(conv_weight, "conv_weight", (Cc, W), torch.float32, dev)
    _need(conv_bias, "conv_bias", (Cc,), torch.float32, dev)
    _need(dt, "dt", lead + (Bsz, H), io, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(D, "D", (H,), torch.float32, dev)
    _need(ssm_state, "ssm_state", (Bsz, H, P, N), torch.float32, dev)
    _need(z, "z", lead + (Bsz, H * P), io, dev)
    _need(norm_weight, "norm_weight", (H * P,), torch.float32, dev)
    if out is None:
        out = torch.empty(lead + (Bsz, H * P), dtype=io, device=dev)
    _need(out, "out", lead + (Bsz, H * P), io, dev)
    d = _dims(Bsz, 1, H, P, N, G, _io_code(io))
    need = int(load().ssd_decode_layer_workspace_size(ctypes.byref(d)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8, dev)
    group = H * P if norm_group is None else int(norm_group)
    return d, W, group, out, workspace


def decode_layer_step(xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z, norm_weight,
                      norm_group=None, eps=1e-5, out=None, workspace=None, stream=None):
    """One token of the decode layer body (conv step + silu, SSD decode step,
    gated RMS norm), states updated in place. xBC[B, H*P + 2*G*N], conv_state
    [B, Cc, W], ssm_state[B,H,P,N] float32, dt[B,H], z[B, H*P]. Returns out[B, H*P]."""
    d, W, group, out, workspace = _layer_args(xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z,
                                              norm_weight, norm_group, out, workspace)
    _check(load().ssd_decode_layer_step(ctypes.byref(d), W, _ptr(xBC), _ptr(conv_state), _ptr(conv_weight),
                                        _ptr(conv_bias), _ptr(dt), _ptr(A), _ptr(D), _ptr(ssm_state), _ptr(z),
                                        _ptr(norm_weight), group, float(eps), _ptr(out), _ptr(workspace),
                                        workspace.numel(), _stream(stream, xBC.device)))
    return out


class DecodeGraph:
    """`steps` decode-layer steps captured once as a CUDA graph by the library
    (ssd_decode_graph_create) and replayed with one launch. xBC[steps,B,Cc],
    dt[steps,B,H], z[steps,B,H*P] and out[steps,B,H*P] hold the per-step
    inputs and outputs; every tensor must outlive the graph."""

    def __init__(self, xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z, norm_weight,
                 norm_group=None, eps=1e-5, out=None, workspace=None):
        steps = xBC.shape[0]
        d, W, group, out, workspace = _layer_args(xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z,
                                                  norm_weight, norm_group, out, workspace, steps=steps)
        self.out, self._keep = out, (xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z,
                                     norm_weight, workspace)
        h = ctypes.c_void_p()
        _check(load().ssd_decode_graph_create(ctypes.byref(d), W, steps, _ptr(xBC), _ptr(conv_state),
                                              _ptr(conv_weight), _ptr(conv_bias), _ptr(dt), _ptr(A), _ptr(D),
                                              _ptr(ssm_state), _ptr(z), _ptr(norm_weight), group, float(eps),
                                              _ptr(out), _ptr(workspace), workspace.numel(), ctypes.byref(h)))
        self._h = h
        self.device = xBC.device

    def launch(self, stream=None):
        _check(load().ssd_decode_graph_launch(self._h, _stream(stream, self.device)))
        return self.out

    def close(self):
        if self._h:
            _check(load().ssd_decode_graph_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
