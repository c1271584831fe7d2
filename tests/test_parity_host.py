"""GPU parity of the host-buffer scan (ssm_scan_fwd_host through the C ABI)
against the fp64 oracle: pieces of whole batch rows and of channel ranges, more
pieces than staging slots, ragged last pieces, pinned and pageable host memory."""
import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import TOL, from_torch, rel_err

pytestmark = pytest.mark.gpu


def _host(a, io, pinned=True):
    import torch
    if a is None:
        return None
    if io == W.BF16 and a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.pin_memory() if pinned else t.clone()


CASES = [
    # io, batch, dim, dstate, seqlen, gate, h0, disc, pinned
    (W.BF16, 9, 40, 16, 256, True, True, "zoh", True),     # 2-row pieces, ragged last
    (W.F32, 1, 300, 8, 100, False, True, "zoh", True),     # channel ranges, unaligned rows
    (W.BF16, 3, 1000, 16, 512, True, False, "zoh", True),  # 9 pieces through 3 slots
    (W.F32, 2, 64, 4, 64, True, True, "euler", False),     # pageable host memory
]


@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,h0,disc,pinned", CASES)
def test_scan_fwd_host(io, batch, dim, dstate, seqlen, gate, h0, disc, pinned):
    from selective_state_space_115_b300 import binding
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=dim + seqlen, with_h0=h0)
    y, hl = binding.scan_fwd_host(
        _host(x["u"], io, pinned), _host(x["delta"], io, pinned), _host(x["A"], W.F32, pinned),
        _host(x["B"], io, pinned), _host(x["C"], io, pinned), D=_host(x["D"], W.F32, pinned),
        z=_host(x.get("z"), io, pinned), delta_bias=_host(x["delta_bias"], W.F32, pinned),
        h0=_host(x.get("h0"), W.F32, pinned), return_last_state=True, discretization=disc)
    f = lambda a: None if a is None else W.to_f64(a, io)  # noqa: E731
    ref, href = oracle.scan_fwd(f(x["u"]), f(x["delta"]), x["A"], f(x["B"]), f(x["C"]),
                                D=x["D"], z=f(x.get("z")), delta_bias=x["delta_bias"],
                                h0=x.get("h0"), return_last_state=True, discretization=disc)
    assert rel_err(from_torch(y), ref) <= TOL[io]
    assert rel_err(from_torch(hl), href) <= (1e-4 if io == W.F32 else 1e-3)
