"""GPU parity of the single-token state update (decode) against the fp64 oracle."""
import os

import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu
NTHREADS = os.cpu_count() or 1


def S():
    from selective_state_space_115_b300 import binding
    return binding


def gpu_step(h, st, static, io):
    return S().state_update(h, torch_io(st["u"], io), torch_io(st["delta"], io),
                            torch_f32(static["A"]), torch_io(st["B"], io), torch_io(st["C"], io),
                            D=torch_f32(static["D"]), z=torch_io(st.get("z"), io),
                            delta_bias=torch_f32(static["delta_bias"]))


def oracle_step(h, st, static, io):
    f = lambda a: None if a is None else W.to_f64(a, io)  # noqa: E731
    u, dl, z, B, C = (f(st.get(k)) for k in ("u", "delta", "z", "B", "C"))
    return oracle.state_update(h, u, dl, static["A"], B, C, D=static["D"], z=z,
                               delta_bias=static["delta_bias"], nthreads=NTHREADS)


def test_decode_all_rows_first_steps():
    """Full decode workload (B256 D5120 N16, bf16 io, fp32 state): every channel
    for the first 8 steps."""
    import torch
    cfg = W.DECODE_CONFIGS["decode"]
    static = W.make_decode_static(cfg, seed=0)
    h = torch_f32(static["h"])
    href = static["h"].astype(np.float64)
    for t in range(8):
        st = W.make_decode_step(cfg, t, seed=0)
        y = gpu_step(h, st, static, cfg.io)
        torch.cuda.synchronize()
        yref, href = oracle_step(href, st, static, cfg.io)
        e = rel_err(from_torch(y), yref)
        eh = rel_err(from_torch(h), href)
        assert e <= TOL[cfg.io], (t, e)
        assert eh <= 1e-5, (t, eh)


@pytest.mark.slow
def test_decode_1024_steps_all_rows():
    """The full 1024-step loop on the full batch (B256 D5120 N16, h in place); the oracle
    follows every channel through every step, and y and h are compared over all
    channels every 64 steps and at the last step."""
    import torch
    cfg = W.DECODE_CONFIGS["decode"]
    static = W.make_decode_static(cfg, seed=0)
    h = torch_f32(static["h"])
    href = static["h"].astype(np.float64)
    worst_y = worst_h = 0.0
    for t in range(cfg.steps):
        st = W.make_decode_step(cfg, t, seed=0)
        y = gpu_step(h, st, static, cfg.io)
        yref, href = oracle_step(href, st, static, cfg.io)
        if t % 64 == 63 or t == cfg.steps - 1:
            torch.cuda.synchronize()
            ey, eh = rel_err(from_torch(y), yref), rel_err(from_torch(h), href)
            worst_y, worst_h = max(worst_y, ey), max(worst_h, eh)
            assert ey <= TOL[cfg.io], (t, ey)
            assert eh <= 1e-4, (t, eh)
    torch.cuda.synchronize()
    print(f"decode 1024 steps, all channels: worst y err {worst_y:.3e}, h err {worst_h:.3e}")


@pytest.mark.parametrize("io", [W.F32, W.BF16])
@pytest.mark.parametrize("dstate", [4, 8, 16])
@pytest.mark.parametrize("gate", [True, False])
def test_decode_shapes(io, dstate, gate):
    import torch
    cfg = W.DecodeConfig("t", 3, 37, dstate, 5, io, gate=gate, h_std=0.1, description="")
    static = W.make_decode_static(cfg, seed=2)
    h = torch_f32(static["h"])
    href = static["h"].astype(np.float64)
    for t in range(cfg.steps):
        st = W.make_decode_step(cfg, t, seed=2)
        y = gpu_step(h, st, static, io)
        torch.cuda.synchronize()
        yref, href = oracle_step(href, st, static, io)
        assert rel_err(from_torch(y), yref) <= TOL[io]
        assert rel_err(from_torch(h), href) <= 1e-5


def test_decode_unaligned_state_falls_back():
    import torch
    io = W.BF16
    cfg = W.DecodeConfig("t", 2, 20, 16, 3, io, gate=True, h_std=0.1, description="")
    static = W.make_decode_static(cfg, seed=4)
    big = torch.zeros(static["h"].size + 1, dtype=torch.float32, device="cuda")
    h = big[1:].view(static["h"].shape)
    h.copy_(torch_f32(static["h"]))
    href = static["h"].astype(np.float64)
    for t in range(cfg.steps):
        st = W.make_decode_step(cfg, t, seed=4)
        y = gpu_step(h, st, static, io)
        torch.cuda.synchronize()
        yref, href = oracle_step(href, st, static, io)
        assert rel_err(from_torch(y), yref) <= TOL[io]
        assert rel_err(from_torch(h), href) <= 1e-5


@pytest.mark.parametrize("io", [W.F32, W.BF16])
@pytest.mark.parametrize("algo", ["channel", "channel_l1", "channel_l2", "chunk"])
def test_steps_equal_scan(io, algo):
    """L decode steps reproduce one scan over L (both on the GPU)."""
    import torch
    cfg = W.ScanConfig("t", 2, 40, 16, 96, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=21, with_h0=True)
    y_scan, h_scan = S().scan_fwd(torch_io(x["u"], io), torch_io(x["delta"], io),
                                  torch_f32(x["A"]), torch_io(x["B"], io), torch_io(x["C"], io),
                                  D=torch_f32(x["D"]), z=torch_io(x["z"], io),
                                  delta_bias=torch_f32(x["delta_bias"]), h0=torch_f32(x["h0"]),
                                  return_last_state=True, algo=algo)
    h = torch_f32(x["h0"]).clone()
    ys = []
    A, D, bias = torch_f32(x["A"]), torch_f32(x["D"]), torch_f32(x["delta_bias"])
    for l in range(cfg.seqlen):
        sl = lambda a: np.ascontiguousarray(a[..., l])  # noqa: E731
        ys.append(S().state_update(h, torch_io(sl(x["u"]), io), torch_io(sl(x["delta"]), io), A,
                                   torch_io(sl(x["B"]), io), torch_io(sl(x["C"]), io), D=D,
                                   z=torch_io(sl(x["z"]), io), delta_bias=bias))
    torch.cuda.synchronize()
    y_steps = np.stack([from_torch(t) for t in ys], axis=-1)
    assert rel_err(y_steps, from_torch(y_scan)) <= TOL[io]
    assert rel_err(from_torch(h), from_torch(h_scan)) <= (1e-5 if io == W.F32 else 1e-3)


@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_decode_euler_input_term(io):
    """Decode steps with Bbar = dt B against the oracle's Euler step."""
    import torch
    cfg = W.DecodeConfig("t", 3, 70, 16, 4, io, gate=True, h_std=0.1, description="")
    static = W.make_decode_static(cfg, seed=6)
    h = torch_f32(static["h"])
    href = static["h"].astype(np.float64)
    for t in range(cfg.steps):
        st = W.make_decode_step(cfg, t, seed=6)
        y = S().state_update(h, torch_io(st["u"], io), torch_io(st["delta"], io),
                             torch_f32(static["A"]), torch_io(st["B"], io),
                             torch_io(st["C"], io), D=torch_f32(static["D"]),
                             z=torch_io(st["z"], io), delta_bias=torch_f32(static["delta_bias"]),
                             discretization="euler")
        torch.cuda.synchronize()
        f = lambda a: W.to_f64(a, io)  # noqa: E731
        yref, href = oracle.state_update(href, f(st["u"]), f(st["delta"]), static["A"],
                                         f(st["B"]), f(st["C"]), D=static["D"], z=f(st["z"]),
                                         delta_bias=static["delta_bias"], discretization="euler")
        assert rel_err(from_torch(y), yref) <= TOL[io]
        assert rel_err(from_torch(h), href) <= 1e-5
