"""Host-side checks of the C ABI (no GPU needed).

The library must build, load, and export every function include/ssd_scan.h
declares; argument validation must reject bad calls before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from mamba_ssd_selective_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from mamba_ssd_selective_gb300 import binding
    nvbuild.build()
    return binding.load()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?(?:size_t|ssd_status|char|void|int)\s*\*?\s*(\w+)\s*\(", text, re.M):
            names.append(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ("ssd_scan_chunked", "ssd_decode_step", "selective_scan_diag", "ssd_workspace_size",
                 "ssd_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libssdscan.so does not export {name}"


def test_library_links_no_libcuda_and_no_oracle():
    # the CUDA runtime is static and the driver API is fetched at run time, so the
    # library loads on a machine without a GPU driver; it never links the oracle
    nvbuild.build()
    import subprocess
    out = subprocess.run(["readelf", "-d", nvbuild.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out
    assert "oracle" not in out


def _dims(binding, **kw):
    base = dict(batch=1, seqlen=256, nheads=4, headdim=64, dstate=16, ngroups=1, io_dtype=0, flags=0)
    base.update(kw)
    return binding.ssd_dims(**base)


def test_workspace_size(lib):
    from mamba_ssd_selective_gb300 import binding
    d = _dims(binding, batch=2, seqlen=1000, nheads=3, headdim=64, dstate=128, io_dtype=1)
    ws = lib.ssd_workspace_size(ctypes.byref(d), 128)
    nc = (1000 + 127) // 128
    n_state = 2 * nc * 3 * 64 * 128
    assert ws >= 256 + n_state * 4 + n_state * 2 + 2 * 3 * nc * 4
    assert ws % 256 == 0
    assert lib.ssd_workspace_size(ctypes.byref(d), 100) == 0          # bad chunk size
    assert lib.ssd_workspace_size(None, 128) == 0                      # no dims
    bad = _dims(binding, nheads=3, ngroups=2)
    assert lib.ssd_workspace_size(ctypes.byref(bad), 64) == 0          # H % G != 0


def _scan(lib, d, chunk=64, x=0x1000, ws=0x100000, ws_bytes=1 << 30):
    vp = ctypes.c_void_p
    return lib.ssd_scan_chunked(ctypes.byref(d) if d is not None else None, vp(x), vp(0x1000), vp(0x1000),
                                vp(0x1000), vp(0x1000), None, None, chunk, vp(0x1000), None,
                                vp(ws) if ws else None, ws_bytes, None)


def test_validation_rejects_before_any_cuda_call(lib):
    from mamba_ssd_selective_gb300 import binding
    E = binding.SSD_ERR_INVALID_ARG
    d = _dims(binding)
    assert _scan(lib, None) == E
    assert b"dims" in lib.ssd_last_error()
    assert _scan(lib, d, chunk=100) == E
    assert b"chunk_size" in lib.ssd_last_error()
    assert _scan(lib, d, x=0) == E                                     # NULL x
    assert _scan(lib, d, x=0x1008) == E                                # misaligned x
    assert b"aligned" in lib.ssd_last_error()
    assert _scan(lib, d, ws=0) == E                                    # NULL workspace
    assert _scan(lib, d, ws=0x100010) == E                             # workspace not 256-aligned
    assert _scan(lib, d, ws_bytes=16) == E                             # workspace too small
    assert b"too small" in lib.ssd_last_error()
    assert _scan(lib, _dims(binding, nheads=6, ngroups=4)) == E
    assert _scan(lib, _dims(binding, io_dtype=7)) == E
    assert _scan(lib, _dims(binding, flags=8)) == E
    assert _scan(lib, _dims(binding, flags=binding.SSD_FLAG_FUSED | binding.SSD_FLAG_SIMT)) == E
    assert _scan(lib, _dims(binding, flags=binding.SSD_FLAG_FUSED | binding.SSD_FLAG_STAGED)) == E
    assert b"SSD_FLAG_FUSED" in lib.ssd_last_error()
    assert _scan(lib, _dims(binding, headdim=0)) == E
    assert _scan(lib, _dims(binding, seqlen=-1)) == E
    assert _scan(lib, _dims(binding, nheads=70000)) == binding.SSD_ERR_UNSUPPORTED
    # an empty batch is a valid no-op and touches nothing
    assert _scan(lib, _dims(binding, batch=0), x=0, ws=0) == binding.SSD_OK


def test_decode_and_diag_validation(lib):
    from mamba_ssd_selective_gb300 import binding
    vp = ctypes.c_void_p
    d = _dims(binding)
    E = binding.SSD_ERR_INVALID_ARG
    assert lib.ssd_decode_step(ctypes.byref(d), None, *[vp(0x1000)] * 5, None, vp(0x1000), None) == E
    assert lib.ssd_decode_step(ctypes.byref(d), vp(0x1004), *[vp(0x1000)] * 5, None, vp(0x1000), None) == E
    assert lib.ssd_decode_step(ctypes.byref(_dims(binding, batch=0)), *[None] * 9) == binding.SSD_OK
    args = [vp(0x1000)] * 5 + [None, None]
    assert lib.selective_scan_diag(1, 64, 128, 16, 1, *args, 48, vp(0x1000), None, None) == E   # chunk % 32
    assert lib.selective_scan_diag(1, 64, 128, 65, 1, *args, 64, vp(0x1000), None, None) == \
        binding.SSD_ERR_UNSUPPORTED
    assert lib.selective_scan_diag(1, 64, 0, 16, 1, *args, 64, vp(0x1000), None, None) == E
    assert lib.selective_scan_diag(1, 64, 128, 16, 3, *args, 64, vp(0x1000), None, None) == E
    assert lib.selective_scan_diag(0, 64, 128, 16, 1, *[None] * 7, 64, None, None, None) == binding.SSD_OK
    assert lib.ssd_selftest_bounded_wait(None, 10, None) == E
    assert lib.ssd_selftest_bounded_wait(vp(0x1000), 0, None) == E


def test_backward_validation_and_workspace_size(lib):
    from mamba_ssd_selective_gb300 import binding
    vp = ctypes.c_void_p
    d = _dims(binding, batch=2, seqlen=200, nheads=4, headdim=64, dstate=128, io_dtype=1)
    ws = lib.ssd_scan_chunked_bwd_workspace_size(ctypes.byref(d))
    nc = (200 + 63) // 64
    assert ws >= 2 * (2 * nc * 4 * 64 * 128 * 4) + 2 * (2 * 200 * 4 * 128 * 4) and ws % 256 == 0
    assert lib.ssd_scan_chunked_bwd_workspace_size(ctypes.byref(_dims(binding, headdim=128))) == 0   # P > 64
    assert lib.ssd_scan_chunked_bwd_workspace_size(ctypes.byref(_dims(binding, dstate=256))) == 0    # N > 128
    assert lib.ssd_scan_chunked_bwd_workspace_size(None) == 0
    ptr = [vp(0x1000)] * 16

    def bwd(dims, ptrs=ptr, ws_ptr=vp(0x100000), ws_bytes=1 << 40):
        return lib.ssd_scan_chunked_bwd(ctypes.byref(dims) if dims is not None else None, *ptrs, ws_ptr, ws_bytes, None)
    assert bwd(None) == binding.SSD_ERR_INVALID_ARG
    assert bwd(_dims(binding, headdim=128)) == binding.SSD_ERR_UNSUPPORTED
    assert bwd(d, ws_bytes=16) == binding.SSD_ERR_INVALID_ARG
    assert b"too small" in lib.ssd_last_error()
    assert bwd(d, ws_ptr=vp(0x100010)) == binding.SSD_ERR_INVALID_ARG                          # not 256-aligned
    bad = list(ptr)
    bad[7] = vp(0x1008)                                                                        # dy misaligned
    assert bwd(d, bad) == binding.SSD_ERR_INVALID_ARG
    bad = list(ptr)
    bad[9] = None                                                                              # dx missing
    assert bwd(d, bad) == binding.SSD_ERR_INVALID_ARG


def test_scan_path_query(lib):
    from mamba_ssd_selective_gb300 import binding
    r = ctypes.byref
    assert lib.ssd_scan_path(None, 128) == -1
    assert lib.ssd_scan_path(r(_dims(binding)), 100) == -1
    assert lib.ssd_scan_path(r(_dims(binding, nheads=6, ngroups=4)), 128) == -1
    # float32 inputs and the SIMT flag always take the CUDA-core path
    assert lib.ssd_scan_path(r(_dims(binding, io_dtype=binding.SSD_F32)), 128) == 0
    assert lib.ssd_scan_path(r(_dims(binding, io_dtype=binding.SSD_BF16, flags=binding.SSD_FLAG_SIMT)), 128) == 0


def test_best_chunk_policy(lib):
    from mamba_ssd_selective_gb300 import binding
    pick = lambda **kw: lib.ssd_best_chunk(ctypes.byref(_dims(binding, **kw)))
    bf = dict(headdim=64, dstate=128, io_dtype=1)
    assert pick(batch=1, seqlen=4096, nheads=24, **bf) == 128     # 130M-shaped layer
    for L in (1024, 4096, 8192):
        assert pick(batch=1, seqlen=L, nheads=80, **bf) == 128    # 2.7B-shaped layers
    assert pick(batch=8, seqlen=2048, nheads=80, **bf) == 128
    assert pick(batch=1, seqlen=512, nheads=24, **bf) == 64       # the one grid point where 64 won
    for b, L, h in ((3, 700, 30), (16, 65536, 128), (1, 1, 1), (5, 3000, 64)):   # off the grid
        assert pick(batch=b, seqlen=L, nheads=h, **bf) in (64, 128, 256)
    assert pick(batch=1, seqlen=4096, nheads=4, headdim=64, dstate=16, io_dtype=0) == 128   # CUDA-core shapes
    assert lib.ssd_best_chunk(None) == 0
    assert pick(batch=1, seqlen=4096, nheads=6, ngroups=4) == 0  # H % G != 0
    assert pick(batch=0) == 0
    assert binding.ssd_best_chunk(1, 4096, 24, 64, 128, 1, __import__("torch").bfloat16) == 128


def test_diag_ex_validation_and_workspace_size(lib):
    from mamba_ssd_selective_gb300 import binding
    vp = ctypes.c_void_p
    E = binding.SSD_ERR_INVALID_ARG
    # time segments only where one pass per sequence leaves the GPU idle
    ws = lib.selective_scan_diag_workspace_size(1, 4096, 1024, 16, 1)
    assert ws > 0 and ws >= 1024 * 16 * 4 * 2
    assert lib.selective_scan_diag_workspace_size(8, 2048, 5120, 16, 1) == 0    # enough channels already
    assert lib.selective_scan_diag_workspace_size(1, 4096, 1024, 16, 0) == 0    # float32 path: one pass
    assert lib.selective_scan_diag_workspace_size(1, 100, 1024, 16, 1) == 0     # too short to split
    assert lib.selective_scan_diag_workspace_size(1, 4096, 1024, 65, 1) == 0    # invalid dstate
    assert lib.selective_scan_diag_workspace_size(0, 4096, 1024, 16, 1) == 0

    def ex(softplus=0, z=None, bias=None, ws_ptr=None, ws_bytes=0, y=0x1000):
        return lib.selective_scan_diag_ex(1, 4096, 1024, 16, 1, *[vp(0x1000)] * 5, None, z, bias, softplus, None,
                                          64, vp(y) if y else None, None, ws_ptr, ws_bytes, None)
    assert ex(softplus=2) == E
    assert b"delta_softplus" in lib.ssd_last_error()
    assert ex(z=vp(0x1008)) == E                                    # misaligned z
    assert ex(bias=vp(0x1004)) == E                                 # misaligned delta_bias
    assert ex(ws_ptr=vp(0x100010), ws_bytes=1 << 30) == E           # workspace not 256-aligned
    assert ex(ws_ptr=vp(0x100000), ws_bytes=16) == E                # workspace too small
    assert b"too small" in lib.ssd_last_error()
    assert ex(y=0) == E                                             # NULL y


def test_binding_checks_shapes_on_cpu_tensors():
    import torch
    from mamba_ssd_selective_gb300 import binding
    x = torch.zeros(1, 8, 2, 4)
    with pytest.raises((ValueError, TypeError)):
        binding.ssd_scan_chunked(x, torch.zeros(1, 8, 3), torch.zeros(2), torch.zeros(1, 8, 1, 4),
                                 torch.zeros(1, 8, 1, 4), chunk_size=64)


def test_tensor_core_probe_compiles(tmp_path):
    """The tensor-core probe of the GPU tests builds against the library's
    inline-PTX helpers (nvcc cross-compiles for sm_103a without a GPU), so a
    helper it needs cannot disappear unnoticed before a GPU run."""
    import subprocess
    try:
        nvcc = nvbuild.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not installed")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc", "tc_probe.cu")
    cmd = [nvcc] + nvbuild.ARCH + ["-O0", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", nvbuild.CSRC,
                                   "-I", nvbuild.INCLUDE, src, "-o", str(tmp_path / "libtcprobe.so")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]


def test_debug_bounds_status_in_a_release_build(lib):
    """The release library runs no bounds checks and says so, without a CUDA call."""
    from mamba_ssd_selective_gb300 import binding
    site, index = ctypes.c_int(7), ctypes.c_int64(7)
    assert lib.ssd_debug_bounds_status(ctypes.byref(site), ctypes.byref(index), 0) == binding.SSD_ERR_UNSUPPORTED
    assert b"SSD_DEBUG_BOUNDS" in lib.ssd_last_error()


def test_debug_bounds_translation_units_compile(tmp_path):
    """Every translation unit with bounds predicates compiles with -DSSD_DEBUG_BOUNDS (nvcc, sm_103a)."""
    from mamba_ssd_selective_gb300 import build
    import subprocess
    for src in ("decode.cu", "diag.cu", "chunked_fused.cu", "chunked_simt.cu", "ssd_api.cu"):
        cmd = [build.nvcc()] + build._flags(False, True) + ["-c", os.path.join(build.CSRC, src), "-o",
                                                            str(tmp_path / (src + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
