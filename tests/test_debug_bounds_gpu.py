"""The bounds-checked debug build (SSD_DEBUG_BOUNDS) on valid inputs: every
checked kernel -- decode step, Mamba-1 scan (one pass and time-segmented),
state pass of the three-kernel prefill, single-pass prefill -- gives the
oracle's results and no bounds check fires (a check never traps: a failure
is recorded and reported by ssd_debug_bounds_status).

The debug library is built here and loaded in a child process
(SSD_DEBUG_BOUNDS_LIB=1), so that this process keeps the release library.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

CHILD = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
import oracle
from mamba_ssd_selective_gb300 import binding, inputs
from tests.helpers import check, dev, host
lib = binding.load()
assert binding.lib_path().endswith("libssdscan_dbg.so")
bf = torch.bfloat16
out = {}
rc, site, index = binding.ssd_debug_bounds_status(clear=True)
out["fresh"] = rc
# decode steps (4-warp and 8-warp launch shapes)
for (Bz, H, P, N, G) in [(2, 8, 64, 128, 1), (16, 80, 64, 128, 2)]:
    st0 = inputs.decode_state(Bz, H, P, N, seed=1)
    prm = inputs.decode_params(H, seed=1)
    st = dev(st0)
    for s in range(3):
        di = inputs.decode_step_inputs(s, Bz, H, P, N, G, io_dtype="bf16", seed=1)
        y = binding.ssd_decode_step(st, dev(di["x"], bf), dev(di["dt"], bf), dev(prm["A"]), dev(di["B"], bf),
                                    dev(di["C"], bf), dev(prm["D"]))
        yr, st0 = oracle.ssd_decode(st0, di["x"], di["dt"], prm["A"], di["B"], di["C"], prm["D"])
        check("bf16", y, yr, "decode y")
    check("bf16", st, st0, "decode state")
# Mamba-1: one pass per sequence, and the time-segmented scan
for (Bz, L, Dm, N, sp) in [(2, 300, 256, 16, False), (1, 4096, 256, 16, True)]:
    d = inputs.diag_option_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=2, bias=False, z=False) if sp else \
        inputs.diag_inputs(Bz, L, Dm, N, io_dtype="bf16", seed=2, init_state=True)
    y, h = binding.selective_scan_diag(dev(d["x"], bf), dev(d["dt"], bf), dev(d["A"]), dev(d["B"], bf),
                                       dev(d["C"], bf), dev(d["D"]), dev(d.get("init_state")), chunk_size=256,
                                       delta_softplus=sp)
    yr, hr = oracle.diag_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d.get("init_state"),
                             delta_softplus=sp)
    check("bf16", y, yr, "mamba1 y")
    check("bf16", h, hr, "mamba1 state")
# prefill through the three-kernel path and the single pass
for path in ("staged", "fused"):
    d = inputs.ssd_inputs(2, 1000, 8, 64, 128, 2, io_dtype="bf16", seed=3, init_state=True)
    y, h = binding.ssd_scan_chunked(dev(d["x"], bf), dev(d["dt"], bf), dev(d["A"]), dev(d["B"], bf),
                                    dev(d["C"], bf), dev(d["D"]), dev(d["init_state"]), chunk_size=128, path=path)
    yr, hr = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
    check("bf16", y, yr, path + " y")
    check("bf16", h, hr, path + " state")
rc, site, index = binding.ssd_debug_bounds_status(clear=True)
out.update(rc=rc, site=site, index=index)
print(json.dumps(out))
'''


def test_debug_bounds_build_runs_clean(cuda_device):
    from mamba_ssd_selective_gb300 import build
    path = build.build(debug_bounds=True)
    assert os.path.exists(path)
    env = dict(os.environ, SSD_DEBUG_BOUNDS_LIB="1")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], capture_output=True, text=True,
                       env=env, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["fresh"] == 0
    assert res["rc"] == 0 and res["site"] == 0, res
