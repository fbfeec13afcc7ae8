"""Shared helpers of the GPU parity tests: moving seeded inputs to the device
and the parity tolerances.

Tolerances (written here once, used by every parity test):
* float32 path: element-wise |gpu - ref| <= 1e-4 + 1e-5 |ref| on y and on the
  final state -- the element-wise parity tolerances (relative 1e-5, absolute
  1e-4) of "Compiler-First State Space Duality ...", Table 6, read as allclose.
* bf16-input path (fp32 state and accumulation, bf16 tensor-core operands):
  max |gpu - ref| <= 2e-2 * max |ref|, separately for y and for the final state.
"""
import numpy as np
import torch

F32_ATOL, F32_RTOL = 1e-4, 1e-5
BF16_REL_MAX = 2e-2

IO_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def dev(a, dtype=torch.float32, device="cuda"):
    """float64 numpy array holding values exact in `dtype` -> device tensor."""
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device).to(dtype)


def host(t):
    return t.detach().to(torch.float64).cpu().numpy()


def check_f32(gpu, ref, what=""):
    gpu = host(gpu) if isinstance(gpu, torch.Tensor) else gpu
    err = np.abs(gpu - ref)
    bound = F32_ATOL + F32_RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} elements outside "
                             f"1e-4 + 1e-5|ref|; worst at {i}: gpu={gpu[i]!r} ref={ref[i]!r}")


def check_bf16(gpu, ref, what=""):
    gpu = host(gpu) if isinstance(gpu, torch.Tensor) else gpu
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    assert err <= BF16_REL_MAX * scale + 1e-30, \
        f"{what}: max|err| = {err:.3e} > 2e-2 * max|ref| = {BF16_REL_MAX * scale:.3e}"


def check(io, gpu, ref, what=""):
    (check_f32 if io == "f32" else check_bf16)(gpu, ref, what)


def head_slice(d, h):
    """Inputs of one head h (all batches) of an SSD workload, for the oracle."""
    H = d["x"].shape[2]
    G = d["B"].shape[2]
    g = h // (H // G)
    return dict(x=d["x"][:, :, h:h + 1], dt=d["dt"][:, :, h:h + 1], A=d["A"][h:h + 1],
                B=d["B"][:, :, g:g + 1], C=d["C"][:, :, g:g + 1], D=d["D"][h:h + 1],
                init_state=None if d["init_state"] is None else d["init_state"][:, h:h + 1])
