"""Builds libssdscan.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel to an object file under
``_build/`` and linked into ``lib/libssdscan.so`` (CUDA runtime linked
statically, no libcuda link: the TMA tensor-map encoder is fetched from the
driver at run time). Objects are rebuilt only when a source or header is
newer. Run ``python -m mamba_ssd_selective_gb300.build [-v]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libssdscan.so")
# debug build: bounds predicates in the kernels (-DSSD_DEBUG_BOUNDS), separate objects and library
DBG_BUILD_DIR = os.path.join(PKG, "_build_dbg")
DBG_LIB_PATH = os.path.join(LIB_DIR, "libssdscan_dbg.so")

SOURCES = ["ssd_api.cu", "decode.cu", "chunked_simt.cu", "chunked_tc.cu", "chunked_fused.cu", "diag.cu", "noalloc.cu", "chunk_policy.cu", "decode_layer.cu", "chunked_bwd.cu", "chunked_bwd_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssdscan.so")
    return p


def _flags(verbose: bool, debug_bounds: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if debug_bounds:
        f += ["-DSSD_DEBUG_BOUNDS"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _deps():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, sources) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _compile(src: str, verbose: bool, debug_bounds: bool = False) -> str:
    obj = os.path.join(DBG_BUILD_DIR if debug_bounds else BUILD_DIR,
                       os.path.splitext(os.path.basename(src))[0] + ".o")
    if not _stale(obj, [src] + _deps()) and not verbose:
        return obj
    tmp = obj + f".tmp{os.getpid()}"
    cmd = [nvcc()] + _flags(verbose, debug_bounds) + ["-c", src, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(tmp, obj)
    return obj


def build(verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compiles and links libssdscan.so (with debug_bounds, the checked
    libssdscan_dbg.so); returns its path."""
    bdir, lib = (DBG_BUILD_DIR, DBG_LIB_PATH) if debug_bounds else (BUILD_DIR, LIB_PATH)
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug_bounds), srcs))
    if _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
