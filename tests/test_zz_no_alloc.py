"""The allocation-free scan entry point, through the C ABI.

Some callers cannot allocate device memory (code running under an allocator or
memory pool it does not control, or in a region where cudaMalloc is forbidden).
ssm_scan_fwd_noalloc serves them with a scratch array reserved statically in the
library instead of a caller-provided workspace.  This test calls it twice in a
row and checks each output against the workspace-taking ssm_scan_fwd on the same
inputs, within the tolerance the parity tests use.  It is collected last and must
also pass alone in a fresh process (the first call on the device does the set-up).
"""
import ctypes

import numpy as np
import pytest

from selective_state_space_115_b300 import workloads as W
from tests.helpers import TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu


def _noalloc(lib, x, io, y, stream):
    import torch
    t = lambda a: None if a is None else ctypes.c_void_p(a.data_ptr())  # noqa: E731
    b, d, L = x["u"].shape
    n = x["A"].shape[1]
    st = lib.ssm_scan_fwd_noalloc(b, d, n, L, 1 if io == W.BF16 else 0, t(x["u"]),
                                  t(x["delta"]), t(x["delta_bias"]), 1, t(x["A"]), t(x["B"]),
                                  t(x["C"]), t(x["D"]), t(x["z"]), t(x.get("h0")), None, t(y),
                                  ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("name,io,batch,dim,seqlen", [
    ("channel-kernel bf16", W.BF16, 2, 5120, 512),   # 10240 channels: TMA channel kernel
    ("chunk-kernel fp32", W.F32, 2, 96, 700),        # few channels, ragged L: chunk kernel
    # one channel of 8192 positions: the segmented two-pass plan, whose segment states
    # (2.5 KB) fit the static scratch
    ("segmented bf16", W.BF16, 1, 1, 8192),
])
def test_noalloc_matches_workspace_entry_point(name, io, batch, dim, seqlen):
    import torch
    from selective_state_space_115_b300 import binding
    lib = binding.library()
    cfg = W.ScanConfig("t", batch, dim, 16, seqlen, io, gate=True, dt_bias=True,
                       d_skip="normal", description=name)
    xn = W.make_scan_inputs(cfg, seed=31)
    x = {k: (torch_io(v, io) if k in ("u", "delta", "z", "B", "C") else torch_f32(v))
         for k, v in xn.items() if v is not None}
    x.setdefault("z", None)
    y_ref = binding.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                             delta_bias=x["delta_bias"])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full_like(x["u"], float("nan"))
        st = _noalloc(lib, x, io, y, stream)
        assert st == binding.SSM_OK, (call, binding.status_string(st),
                                      lib.ssm_last_cuda_error().decode())
        yv = from_torch(y)
        assert np.isfinite(yv).all(), call
        assert rel_err(yv, from_torch(y_ref)) <= TOL[io], call
