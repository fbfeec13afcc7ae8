"""Exponential (SFU) and packed-FMA throughput on this GPU, measured by a small
CUDA probe (tests/probes/xu_fma_rates.cu) built with nvcc and run as a child
process. It is evidence for the Mamba-1 scan's design (one ex2 and about one
packed FMA per state element, both pipes near the same rate), not a parity
test: it checks that the probe ran and that both rates are positive."""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_xu_and_fma_rates():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "xu_fma_rates")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                        os.path.join(HERE, "probes", "xu_fma_rates.cu")], check=True, capture_output=True, timeout=300)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(out.stdout)
    assert out.returncode == 0, out.stdout + out.stderr
    rates = {}
    for m in re.finditer(r"warps/SM\s+(\d+) mode (\d) .*?: [\d.]+ ms, ([\d.]+) chain steps", out.stdout):
        rates[(int(m.group(1)), int(m.group(2)))] = float(m.group(3))
    assert len(rates) == 12 and all(v > 0 for v in rates.values()), out.stdout
