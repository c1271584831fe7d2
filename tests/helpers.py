"""Shared test helpers: tensor marshalling and the error metric."""
from __future__ import annotations

import numpy as np

from selective_state_space_115_b300 import workloads as W

# Tolerances on the error metric below (max over elements):
#   fp32 io: 1e-4;  bf16 io with fp32 state: 2e-2.
TOL = {W.F32: 1e-4, W.BF16: 2e-2}
# The final state h_last is fp32 and never rounded to bf16, so with bf16 io the tests
# hold it to 1e-3 (stricter than the 2e-2 that covers y's bf16 rounding); fp32 io: 1e-4.
H_TOL = {W.F32: 1e-4, W.BF16: 1e-3}


def rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    """max_i |y_i - ref_i| / max(|ref_i|, rms(ref)): relative for typical elements,
    guarded against ref ~ 0 (the gate and D ~ N(0,1) make such elements common)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), rms if rms > 0 else 1.0)
    return float(np.max(np.abs(y - ref) / den))


def torch_io(x: np.ndarray, io: str, device="cuda"):
    """numpy array (fp32, or bf16 bits as uint16) -> torch tensor on device."""
    import torch
    if x is None:
        return None
    if io == W.BF16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device)


def torch_f32(x: np.ndarray, device="cuda"):
    import torch
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def from_torch(t) -> np.ndarray:
    """torch tensor (fp32 or bf16) -> float64 numpy (exact)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return W.bf16_bits_to_f32(t.view(torch.int16).numpy().view(np.uint16)).astype(np.float64)
    return t.numpy().astype(np.float64)
