"""GPU parity of the causal depthwise conv1d (+ silu) and its decode update
(through the C ABI) against the fp64 oracle.  Tolerances as for the scan: 1e-4
for fp32 io, 2e-2 for bf16 io (tests/helpers.py metric)."""
import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu


def S():
    from selective_state_space_115_b300 import binding
    return binding


def _inputs(io, batch, dim, seqlen, width, seed, state):
    rng = np.random.default_rng(seed)
    x = W.encode(rng.standard_normal((batch, dim, seqlen)).astype(np.float32), io)
    w = (rng.standard_normal((dim, width)) / np.sqrt(width)).astype(np.float32)
    bias = rng.standard_normal(dim).astype(np.float32)
    s0 = W.encode(rng.standard_normal((batch, dim, width - 1)).astype(np.float32), io) \
        if state else None
    return x, w, bias, s0


CASES = [
    # io, batch, dim, seqlen, width, state, silu
    (W.BF16, 2, 96, 2048, 4, False, True),    # the Mamba shape (d_conv = 4)
    (W.BF16, 3, 40, 1000, 4, True, True),     # carried state, 125 vectors per row
    (W.BF16, 2, 37, 64, 3, True, True),       # 8 vectors per row: row starts inside a warp
    (W.F32, 3, 21, 24, 7, True, True),        # fp32, two previous vectors per window
    (W.BF16, 1, 5, 8, 8, True, True),         # one vector per row: every window from the state
    (W.F32, 2, 3, 4, 5, False, True),         # one vector per row, zero history
    (W.BF16, 2, 64, 4096, 6, True, False),    # several CTAs per row
    (W.BF16, 1, 8, 1002, 4, True, True),      # L not a multiple of 8: element path
    (W.F32, 2, 33, 517, 4, True, False),      # unaligned rows: element path
    (W.F32, 1, 16, 64, 2, False, True),
    (W.BF16, 1, 8, 3, 7, True, True),         # L < width - 1: history from the state
    (W.F32, 2, 8, 256, 8, True, True),
    (W.BF16, 1, 4, 40, 1, False, False),      # width 1: a pointwise scale
]


@pytest.mark.parametrize("io,batch,dim,seqlen,width,state,silu", CASES)
def test_conv1d_fwd(io, batch, dim, seqlen, width, state, silu):
    import torch
    x, w, bias, s0 = _inputs(io, batch, dim, seqlen, width, seed=seqlen + width, state=state)
    out, st = S().conv1d_fwd(torch_io(x, io), torch_f32(w), torch_f32(bias),
                             conv_state=torch_io(s0, io), apply_silu=silu, return_state=True)
    torch.cuda.synchronize()
    f = lambda a: None if a is None else W.to_f64(a, io)  # noqa: E731
    ref, sref = oracle.conv1d_fwd(f(x), w, bias, state_in=f(s0), apply_silu=silu,
                                  return_state=True)
    assert rel_err(from_torch(out), ref) <= TOL[io]
    assert np.array_equal(from_torch(st), sref)  # the cache holds the raw inputs


@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_conv1d_update_matches_fwd(io):
    """The decode update, step by step, reproduces the full-sequence convolution and
    leaves the cache equal to the last width - 1 inputs."""
    import torch
    batch, dim, seqlen, width = 2, 50, 12, 4
    x, w, bias, s0 = _inputs(io, batch, dim, seqlen, width, seed=3, state=True)
    full = from_torch(S().conv1d_fwd(torch_io(x, io), torch_f32(w), torch_f32(bias),
                                     conv_state=torch_io(s0, io)))
    st = torch_io(s0, io).clone()
    f = lambda a: W.to_f64(a, io)  # noqa: E731
    sref = f(s0)
    for l in range(seqlen):
        xl = np.ascontiguousarray(x[..., l])
        y = S().conv1d_update(st, torch_io(xl, io), torch_f32(w), torch_f32(bias))
        torch.cuda.synchronize()
        yref, sref = oracle.conv1d_update(sref, f(xl), w, bias)
        assert rel_err(from_torch(y), yref) <= TOL[io], l
        assert np.array_equal(from_torch(y), full[..., l]), l
    assert np.array_equal(from_torch(st), sref)


def test_conv1d_guard_bands_untouched():
    import torch
    io = W.BF16
    batch, dim, seqlen, width = 2, 24, 520, 4
    x, w, bias, _ = _inputs(io, batch, dim, seqlen, width, seed=9, state=False)
    n = batch * dim * seqlen
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(batch, dim, seqlen)
    S().conv1d_fwd(torch_io(x, io), torch_f32(w), torch_f32(bias), out=out)
    torch.cuda.synchronize()
    b = from_torch(buf)
    assert np.isnan(b[:guard]).all() and np.isnan(b[guard + n:]).all()
    assert np.isfinite(b[guard:guard + n]).all()
