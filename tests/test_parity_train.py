"""GPU parity of the training step (through the C ABI): the forward that writes the
state checkpoints (ssm_scan_fwd_train) and the gradient that reads them
(ssm_scan_bwd_ckpt), against the fp64 oracle.

The checkpoint of block j is the state entering position 8 j, which the oracle gives
as the final state of the scan over positions [0, 8 j).  The training forward's y and
h_last equal the plain forward's bit for bit (the same kernels, with the checkpoint
stores added).  Tolerances as the other parity tests (tests/helpers.py).
"""
import os

import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import H_TOL, TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu
NTHREADS = os.cpu_count() or 1
ALGOS = ["auto", "channel_l1", "channel_l2", "channel_l4", "channel_mixed", "chunk", "segmented"]
MIN_DSTATE = {"channel_l2": 8, "channel_l4": 16, "channel_mixed": 16}


def S():
    from selective_state_space_115_b300 import binding
    return binding


def f64(x, io):
    return None if x is None else W.to_f64(x, io)


def dev_inputs(x, io):
    t = {k: torch_io(x.get(k), io) for k in ("u", "delta", "z", "B", "C")}
    t.update({k: torch_f32(x.get(k)) for k in ("A", "D", "delta_bias", "h0")})
    return t


def train_forward(t, algo="auto"):
    import torch
    b, d, L = t["u"].shape
    n = t["A"].shape[1]
    ck = torch.full(S().ckpt_shape(b, d, n, L), float("nan"), dtype=torch.float32, device="cuda")
    y, hl = S().scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                         delta_bias=t["delta_bias"], h0=t["h0"], return_last_state=True,
                         algo=algo, ckpt=ck)
    torch.cuda.synchronize()
    assert S().read_device_status() == 0
    return y, hl, ck


def oracle_checkpoints(x, io):
    """[nblk, b, d, n]: the state entering position 8 j, from the oracle's scan over
    positions [0, 8 j) (block 0: h0, or zero)."""
    b, d, L = x["u"].shape
    n = x["A"].shape[1]
    nblk = (L + 7) // 8
    out = np.empty((nblk, b, d, n))
    out[0] = x["h0"] if x.get("h0") is not None else 0.0
    cut = lambda a, m: None if a is None else a[..., :m]  # noqa: E731
    for j in range(1, nblk):
        m = 8 * j
        _, hl = oracle.scan_fwd(f64(cut(x["u"], m), io), f64(cut(x["delta"], m), io), x["A"],
                                f64(cut(x["B"], m), io), f64(cut(x["C"], m), io), D=x.get("D"),
                                z=f64(cut(x.get("z"), m), io), delta_bias=x.get("delta_bias"),
                                h0=x.get("h0"), return_last_state=True, nthreads=NTHREADS)
        out[j] = hl
    return out


SHAPES = [
    # io, batch, dim, dstate, seqlen, gate, h0
    (W.BF16, 2, 160, 16, 136, True, True),     # several 32-channel groups, ragged last block
    (W.F32, 2, 37, 16, 69, True, True),        # ragged tile and tail: the chunk kernel
    (W.BF16, 1, 40, 8, 512, False, False),
    (W.F32, 1, 64, 4, 264, True, False),
]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,h0", SHAPES)
def test_train_forward(algo, io, batch, dim, dstate, seqlen, gate, h0):
    """y and h_last bit for bit as the plain forward; every checkpoint against the
    oracle's state entering its block."""
    if dstate < MIN_DSTATE.get(algo, 0):
        pytest.skip(f"{algo} needs dstate >= {MIN_DSTATE[algo]}")
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=61 + seqlen, with_h0=h0)
    t = dev_inputs(x, io)
    y, hl, ck = train_forward(t, algo)
    y0, hl0 = S().scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                           delta_bias=t["delta_bias"], h0=t["h0"], return_last_state=True,
                           algo=algo)
    assert np.array_equal(from_torch(y), from_torch(y0))
    assert np.array_equal(from_torch(hl), from_torch(hl0))
    ckv = from_torch(ck)
    assert np.isfinite(ckv).all()          # every checkpoint written
    assert rel_err(ckv, oracle_checkpoints(x, io)) <= H_TOL[io]


GRAD_KEYS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


@pytest.mark.parametrize("segments", [0, 3])
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_gradient_from_checkpoints(io, segments):
    """ssm_scan_bwd_ckpt with the training forward's checkpoints against the oracle's
    gradient (unsplit and in three segments), and against the gradient that recomputes
    its states."""
    cfg = W.ScanConfig("t", 2, 96, 16, 520, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=71, with_h0=True)
    gr = W.make_scan_grads(cfg, seed=71)
    t = dev_inputs(x, io)
    _, _, ck = train_forward(t)
    dy, dhl = torch_io(gr["dy"], io), torch_f32(gr["dh_last"])
    kw = dict(D=t["D"], z=t["z"], delta_bias=t["delta_bias"], h0=t["h0"], dh_last=dhl,
              segments=segments)
    g = S().scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], dy, ckpt=ck, **kw)
    g0 = S().scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], dy, **kw)
    import torch
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                          f64(x["C"], io), f64(gr["dy"], io), D=x["D"], z=f64(x["z"], io),
                          delta_bias=x["delta_bias"], h0=x["h0"], dh_last=gr["dh_last"],
                          nthreads=NTHREADS)
    for k in GRAD_KEYS:
        got, base = from_torch(g[k]), from_torch(g0[k])
        assert np.isfinite(got).all(), k
        e = rel_err(got, ref[k])
        print(f"{io} seg {segments} {k}: max rel err {e:.3e}")
        assert e <= TOL[io], (k, e)
        assert rel_err(got, base) <= TOL[io], k


def test_gradient_from_checkpoints_vanishing_steps():
    """bf16, every step tiny (raw delta in [-60, -20]), no D, zero initial state: the
    checkpoints and the series coefficients of the gradient together."""
    io = W.BF16
    cfg = W.ScanConfig("t", 2, 40, 16, 256, io, gate=True, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=72)
    x["D"] = None
    rng = np.random.default_rng(11)
    x["delta"] = W.encode(rng.uniform(-60, -20, size=x["delta"].shape).astype(np.float32), io)
    gr = W.make_scan_grads(cfg, seed=72)
    t = dev_inputs(x, io)
    _, _, ck = train_forward(t)
    g = S().scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], torch_io(gr["dy"], io),
                     z=t["z"], dh_last=torch_f32(gr["dh_last"]), ckpt=ck)
    import torch
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                          f64(x["C"], io), f64(gr["dy"], io), z=f64(x["z"], io),
                          dh_last=gr["dh_last"], nthreads=NTHREADS)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dh0"):
        assert rel_err(from_torch(g[k]), ref[k]) <= TOL[io], k


# Shapes whose AUTO forward plan is the channel kernel (batch * dim >= 8192: four, two
# and one lanes per channel, both discretisations) or the segmented scan (few channels,
# L >= 8192): the gradient called without checkpoints forms them on those kernels, in
# their checkpoint-only mode, instead of in its own forward pass.
CKPT_FORWARD_CASES = [
    # io, batch, dim, dstate, seqlen, gate, disc
    (W.BF16, 2, 4096, 16, 256, True, "zoh"),
    (W.F32, 1, 8192, 8, 128, False, "zoh"),
    (W.BF16, 4, 2048, 4, 64, True, "euler"),
    (W.BF16, 1, 64, 16, 8192, True, "zoh"),
    (W.F32, 8, 5120, 16, 64, True, "zoh"),   # the mixed split (2 one-lane CTAs per SM + quarters)
]


@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,disc", CKPT_FORWARD_CASES)
def test_gradient_checkpoints_from_forward_kernels(io, batch, dim, dstate, seqlen, gate, disc):
    """ssm_scan_bwd without checkpoints where the forward's kernels form them: against
    the oracle's gradient, and bit for bit against the gradient from the training
    forward's checkpoints (the same kernels, the same plan, the same states)."""
    import torch
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=seqlen + dim, with_h0=True)
    gr = W.make_scan_grads(cfg, seed=seqlen + dim)
    t = dev_inputs(x, io)
    ck = torch.full(S().ckpt_shape(batch, dim, dstate, seqlen), float("nan"),
                    dtype=torch.float32, device="cuda")
    S().scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                 delta_bias=t["delta_bias"], h0=t["h0"], discretization=disc, ckpt=ck)
    dy, dhl = torch_io(gr["dy"], io), torch_f32(gr["dh_last"])
    kw = dict(D=t["D"], z=t["z"], delta_bias=t["delta_bias"], h0=t["h0"], dh_last=dhl,
              discretization=disc)
    g = S().scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], dy, **kw)
    gt = S().scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], dy, ckpt=ck, **kw)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                          f64(x["C"], io), f64(gr["dy"], io), D=x["D"], z=f64(x.get("z"), io),
                          delta_bias=x["delta_bias"], h0=x["h0"], dh_last=gr["dh_last"],
                          nthreads=NTHREADS, discretization=disc)
    for k in GRAD_KEYS:
        if ref.get(k) is None:
            continue
        got = from_torch(g[k])
        assert np.isfinite(got).all(), k
        e = rel_err(got, ref[k])
        print(f"{io} b{batch} d{dim} n{dstate} L{seqlen} {disc} {k}: max rel err {e:.3e}")
        assert e <= TOL[io], (k, e)
        assert np.array_equal(got, from_torch(gt[k])), k
