"""The allocation-free prefill entry point against the regular one and the oracle.

ssd_scan_chunked_noalloc is for callers that cannot allocate device memory
where they run the scan (for example a plug-in whose host framework owns all
device memory, or a latency-critical loop that cannot take the device-wide
synchronisation an allocation brings). It keeps the per-chunk states in the
library's built-in device scratch instead of a caller workspace. It must give
the results of ssd_scan_chunked with a workspace, and match the float64
oracle within the parity tolerances, on two calls in a row -- the second one
runs while the scratch still holds the first call's states -- and the second
call must not change the device's free memory. A bounded wait that gives up
must be visible through ssd_scan_chunked_noalloc_status, and the next call
must clear it.

This file is collected last on purpose, and its tests also pass alone in a
fresh process.
"""
import ctypes

import pytest
import torch

import oracle
from mamba_ssd_selective_gb300 import inputs
from tests.helpers import IO_TORCH, check, dev, host

pytestmark = pytest.mark.gpu

# two calls in a row with different sizes and values
CASES = [(1, 1000, 4, 64, 128, 1, 7), (2, 777, 6, 64, 128, 2, 8)]


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(io, cuda_device):
    from mamba_ssd_selective_gb300 import binding
    binding.load()
    t = IO_TORCH[io]
    free_after = []
    for (Bz, L, H, P, N, G, seed) in CASES:
        d = inputs.ssd_inputs(Bz, L, H, P, N, G, io_dtype=io, seed=seed, init_state=True)
        args = [dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t), dev(d["C"], t), dev(d["D"]),
                dev(d["init_state"])]
        y_ref, h_ref = binding.ssd_scan_chunked(*args, chunk_size=128)
        y = torch.empty_like(y_ref)
        h = torch.empty_like(h_ref)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        binding.ssd_scan_chunked_noalloc(*args, chunk_size=128, y=y, final_state=h)
        torch.cuda.synchronize()
        free_after.append((free_before, torch.cuda.mem_get_info()[0]))
        what = f"(B{Bz} L{L} H{H} G{G})"
        check(io, host(y), host(y_ref), f"noalloc y vs workspace entry point {what}")
        check(io, host(h), host(h_ref), f"noalloc final state vs workspace entry point {what}")
        yo, ho = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"])
        check(io, host(y), yo, f"noalloc y vs oracle {what}")
        check(io, host(h), ho, f"noalloc final state vs oracle {what}")
        status, _ = binding.ssd_scan_chunked_noalloc_status()
        assert status == binding.SSD_OK
    # the second call finds its scratch already set up and allocates nothing
    assert free_after[1][0] == free_after[1][1]


def test_noalloc_status_reports_a_timeout_and_the_next_call_clears_it(cuda_device):
    """A bounded wait that gives up on the built-in scratch's status word is
    reported by ssd_scan_chunked_noalloc_status; the next no-alloc scan starts
    from a clear status and reports SSD_OK."""
    from mamba_ssd_selective_gb300 import binding
    lib = binding.load()
    status, addr = binding.ssd_scan_chunked_noalloc_status()
    assert addr and addr % 256 == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ssd_selftest_bounded_wait(ctypes.c_void_p(addr), 1000, stream) == binding.SSD_OK
    status, _ = binding.ssd_scan_chunked_noalloc_status()
    assert status == binding.SSD_ERR_TIMEOUT
    d = inputs.ssd_inputs(1, 300, 4, 64, 128, 1, io_dtype="bf16", seed=9)
    t = torch.bfloat16
    y, h = binding.ssd_scan_chunked_noalloc(dev(d["x"], t), dev(d["dt"], t), dev(d["A"]), dev(d["B"], t),
                                            dev(d["C"], t), dev(d["D"]), None, chunk_size=128)
    status, _ = binding.ssd_scan_chunked_noalloc_status()
    assert status == binding.SSD_OK
    yo, ho = oracle.ssd_seq(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    check("bf16", host(y), yo, "noalloc y after a recorded timeout")
    check("bf16", host(h), ho, "noalloc final state after a recorded timeout")


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    """B1 L4096 H24 P64 N128 at chunk 64 needs about 75 MB of per-chunk states,
    more than the 64 MiB scratch: rejected before any launch."""
    from mamba_ssd_selective_gb300 import binding
    lib = binding.load()
    d = binding.ssd_dims(1, 4096, 24, 64, 128, 1, binding.SSD_BF16, 0)
    assert lib.ssd_workspace_size(ctypes.byref(d), 64) > 64 << 20
    vp = ctypes.c_void_p
    rc = lib.ssd_scan_chunked_noalloc(ctypes.byref(d), *[vp(0x1000)] * 5, None, None, 64, vp(0x1000), None, None)
    assert rc == binding.SSD_ERR_UNSUPPORTED
    assert b"scratch" in lib.ssd_last_error()
