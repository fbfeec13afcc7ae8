"""The tensor-core building blocks against a plain matrix product.

Compiles tests/csrc/tc_probe.cu (one tcgen05 MMA tile per operand layout the
tensor-core SSD kernels use: K-major and MN-major SW128 operands, written by
threads or loaded by TMA, and an A operand held in tensor memory) and compares each result with torch's float32
matmul of the same bf16 values.
"""
import ctypes
import os
import subprocess

import pytest
import torch

from mamba_ssd_selective_gb300 import build as nvbuild

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(tmp_path_factory, cuda_device):
    out = str(tmp_path_factory.mktemp("probe") / "libtcprobe.so")
    cmd = [nvbuild.nvcc()] + nvbuild.ARCH + ["-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                                             "-I", nvbuild.CSRC, "-I", nvbuild.INCLUDE,
                                             os.path.join(HERE, "csrc", "tc_probe.cu"), "-o", out]
    subprocess.run(cmd, check=True)
    lib = ctypes.CDLL(out)
    lib.tc_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.tc_probe.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("N,K", [(64, 64), (64, 128), (128, 128), (64, 256), (128, 256)])
def test_tcgen05_tile(probe, variant, N, K):
    g = torch.Generator().manual_seed(variant * 1000 + N + K)
    a_mn = variant in (2, 4)
    b_mn = variant in (1, 2, 4)
    Am = torch.randn(128, K, generator=g).to(torch.bfloat16)          # logical A [M][K]
    Bn = torch.randn(N, K, generator=g).to(torch.bfloat16)            # logical B^T [N][K]
    A_store = (Am.t() if a_mn else Am).contiguous().cuda()
    B_store = (Bn.t() if b_mn else Bn).contiguous().cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe(variant, A_store.data_ptr(), B_store.data_ptr(), D.data_ptr(), N, K, status.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "bounded wait gave up"
    ref = Am.float() @ Bn.float().t()
    torch.testing.assert_close(D.cpu(), ref, rtol=1e-4, atol=1e-3)
