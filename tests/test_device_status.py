"""The device-side timeout path, on the GPU without a fault: a bounded wait on an
mbarrier phase that nothing completes gives up at its limit, the kernel records
the timeout in the status words and returns, the host reads
SSM_ERR_DEVICE_TIMEOUT, and the context keeps working."""
import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu


def test_wait_that_completes_reports_ok():
    from selective_state_space_115_b300 import binding
    assert binding.selftest_wait(20_000_000, arrive=True) == binding.SSM_OK


def test_wait_that_never_completes_times_out_and_the_context_survives():
    import torch
    from selective_state_space_115_b300 import binding
    assert binding.selftest_wait(20_000_000, arrive=False) == binding.SSM_ERR_DEVICE_TIMEOUT
    # the same process and context run a scan correctly afterwards
    cfg = W.ScanConfig("t", 1, 64, 16, 256, W.BF16, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=4)
    y = binding.scan_fwd(torch_io(x["u"], W.BF16), torch_io(x["delta"], W.BF16),
                         torch_f32(x["A"]), torch_io(x["B"], W.BF16), torch_io(x["C"], W.BF16),
                         D=torch_f32(x["D"]), z=torch_io(x["z"], W.BF16),
                         delta_bias=torch_f32(x["delta_bias"]))
    torch.cuda.synchronize()
    assert binding.read_device_status() == binding.SSM_OK
    f = lambda a: W.to_f64(a, W.BF16)  # noqa: E731
    ref = oracle.scan_fwd(f(x["u"]), f(x["delta"]), x["A"], f(x["B"]), f(x["C"]), D=x["D"],
                          z=f(x["z"]), delta_bias=x["delta_bias"])
    assert rel_err(from_torch(y), ref) <= TOL[W.BF16]
    assert np.isfinite(from_torch(y)).all()
