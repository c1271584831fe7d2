"""GPU parity of the scan's gradient (ssm_scan_bwd through the C ABI) against the
fp64 oracle's reverse-mode derivative.

Every gradient is compared with the error metric of tests/helpers.py: 1e-4 for
fp32 io, 2e-2 for bf16 io (fp32 state).  The shapes span several CTAs of
channels with a ragged last one, sequences with a ragged last block of 8
positions, unaligned rows (element staging) and aligned ones (cp.async staging),
every dstate, both discretisations, and the optional arguments present and absent.
"""
import os

import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu
NTHREADS = os.cpu_count() or 1
GRAD_KEYS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


def S():
    from selective_state_space_115_b300 import binding
    return binding


def f64(x, io):
    return None if x is None else W.to_f64(x, io)


def gpu_bwd(x, gr, io, softplus=True, disc="zoh", with_dh_last=True, segments=0):
    import torch
    g = S().scan_bwd(torch_io(x["u"], io), torch_io(x["delta"], io), torch_f32(x["A"]),
                     torch_io(x["B"], io), torch_io(x["C"], io), torch_io(gr["dy"], io),
                     D=torch_f32(x.get("D")), z=torch_io(x.get("z"), io),
                     delta_bias=torch_f32(x.get("delta_bias")), delta_softplus=softplus,
                     h0=torch_f32(x.get("h0")),
                     dh_last=torch_f32(gr["dh_last"]) if with_dh_last else None,
                     discretization=disc, segments=segments)
    torch.cuda.synchronize()
    return {k: (None if v is None else from_torch(v)) for k, v in g.items()}


def oracle_bwd(x, gr, io, softplus=True, disc="zoh", with_dh_last=True):
    return oracle.scan_bwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                           f64(x["C"], io), f64(gr["dy"], io), D=x.get("D"),
                           z=f64(x.get("z"), io), delta_bias=x.get("delta_bias"),
                           delta_softplus=softplus, h0=x.get("h0"),
                           dh_last=gr["dh_last"] if with_dh_last else None,
                           nthreads=NTHREADS, discretization=disc)


def check(got, ref, io, what="", keys=GRAD_KEYS, tol=None):
    tol = TOL[io] if tol is None else tol
    for k in keys:
        if ref.get(k) is None:
            assert got.get(k) is None, f"{what} {k}: not expected"
            continue
        assert got[k] is not None, f"{what} {k}: missing"
        assert got[k].shape == ref[k].shape, f"{what} {k}: shape {got[k].shape} vs {ref[k].shape}"
        assert np.isfinite(got[k]).all(), f"{what} {k}: non-finite values"
        e = rel_err(got[k], ref[k])
        print(f"{what} {k}: max rel err {e:.3e}")
        assert e <= tol, f"{what} {k}: max rel err {e:.3e} > {tol}"


SHAPES = [
    # io, batch, dim, dstate, seqlen, gate, h0
    (W.F32, 1, 1, 4, 1, False, False),
    (W.BF16, 1, 3, 8, 3, True, True),
    (W.F32, 2, 37, 16, 69, True, True),      # ragged channel tile, ragged last block
    (W.BF16, 3, 37, 16, 72, True, False),    # aligned rows (cp.async), ragged tile
    (W.BF16, 2, 100, 8, 1000, False, True),
    (W.F32, 1, 64, 4, 4096, True, False),    # two full CTAs of channels, long-ish L
    (W.BF16, 2, 33, 16, 517, True, True),    # L not a multiple of 8: element staging
    (W.F32, 1, 130, 16, 2, False, True),
    (W.BF16, 4, 96, 16, 256, True, True),    # three CTAs per batch row, four batch rows
]


@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,h0", SHAPES)
def test_bwd_shapes(io, batch, dim, dstate, seqlen, gate, h0):
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=seqlen + dim, with_h0=h0)
    gr = W.make_scan_grads(cfg, seed=seqlen + dim)
    check(gpu_bwd(x, gr, io), oracle_bwd(x, gr, io), io,
          what=f"{io} b{batch} d{dim} n{dstate} L{seqlen}")


@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_bwd_euler(io):
    cfg = W.ScanConfig("t", 2, 70, 16, 272, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=3, with_h0=True)
    gr = W.make_scan_grads(cfg, seed=3)
    check(gpu_bwd(x, gr, io, disc="euler"), oracle_bwd(x, gr, io, disc="euler"), io,
          what=f"euler {io}")


# (2, 40, 256): the gradient kernel forms its checkpoints; (2, 4096, 64): 8192 channels,
# the forward's channel kernel forms them in its checkpoint-only pass
@pytest.mark.parametrize("dim,seqlen", [(40, 256), (4096, 64)])
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_bwd_optional_arguments_absent(io, dim, seqlen):
    """No D, bias, gate, h0 or dh_last; delta used as dt directly (no softplus)."""
    cfg = W.ScanConfig("t", 2, dim, 16, seqlen, io, gate=False, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=5)
    x["D"] = None
    x["delta_bias"] = None
    x32 = np.abs(W.to_f64(x["delta"], io)).astype(np.float32) * np.float32(0.05)
    x["delta"] = W.encode(x32, io)
    gr = W.make_scan_grads(cfg, seed=5)
    got = gpu_bwd(x, gr, io, softplus=False, with_dh_last=False)
    ref = oracle_bwd(x, gr, io, softplus=False, with_dh_last=False)
    check(got, ref, io, what=f"no options {io} d{dim} L{seqlen}")


@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_bwd_zero_and_small_A(io):
    """A == 0 (the dt limit and dcoef/dA = dt^2 / 2) and tiny |A| (the series
    branches; bf16 leaves the fast path for the warps that hold them)."""
    cfg = W.ScanConfig("t", 1, 48, 8, 512, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=11)
    A = x["A"].copy()
    A[0, :] = 0.0
    A[5, 3] = -1e-7
    A[9, :] = -np.float32(1e-3) * np.arange(1, 9, dtype=np.float32)
    A[20, 1] = 0.0
    x["A"] = A
    gr = W.make_scan_grads(cfg, seed=11)
    check(gpu_bwd(x, gr, io), oracle_bwd(x, gr, io), io, what=f"small A {io}")


SEGMENT_CASES = [
    # io, batch, dim, dstate, seqlen, gate, h0, segments, disc
    (W.BF16, 2, 40, 16, 1000, True, True, 4, "zoh"),     # 125 blocks in 4 segments
    (W.F32, 1, 37, 16, 517, True, True, 3, "zoh"),       # ragged last segment, element staging
    (W.BF16, 1, 70, 8, 2048, False, False, 7, "euler"),
    (W.F32, 2, 33, 4, 96, True, True, 1000, "zoh"),      # capped at one block per segment
    (W.BF16, 3, 64, 16, 256, True, True, 2, "zoh"),
]


@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,h0,segments,disc", SEGMENT_CASES)
def test_bwd_segments(io, batch, dim, dstate, seqlen, gate, h0, segments, disc):
    """The sequence split into segments (first pass: each segment's end state, own
    adjoint and step-size sum; second pass: the segment with its combined entering
    state and end adjoint) against the oracle."""
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=seqlen + segments, with_h0=h0)
    gr = W.make_scan_grads(cfg, seed=seqlen + segments)
    check(gpu_bwd(x, gr, io, disc=disc, segments=segments),
          oracle_bwd(x, gr, io, disc=disc), io, what=f"{segments} segments {io} L{seqlen}")


def test_bwd_segments_match_unsplit():
    """A forced split and no split agree to rounding on the same inputs."""
    io = W.F32
    cfg = W.ScanConfig("t", 1, 64, 16, 2048, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=8, with_h0=True)
    gr = W.make_scan_grads(cfg, seed=8)
    a = gpu_bwd(x, gr, io, segments=1)
    b = gpu_bwd(x, gr, io, segments=6)
    for k in GRAD_KEYS:
        assert rel_err(b[k], a[k]) <= 1e-5, k


def test_bwd_long_sampled():
    """The long-sequence workload (bf16, B1 D1536 N16 L131072, no gate), which the
    library splits into segments: channel-local gradients, dA, dD, the bias gradient
    and dh0 on sampled channels against the oracle over those channels."""
    cfg = W.SCAN_CONFIGS["long"]
    io = cfg.io
    x = W.make_scan_inputs(cfg, seed=0)
    gr = W.make_scan_grads(cfg, seed=0)
    got = gpu_bwd(x, gr, io)
    ds = np.array([0, 31, 32, 777, 1535], dtype=np.int64)
    sub = dict(x)
    for k in ("u", "delta"):
        sub[k] = np.ascontiguousarray(x[k][:, ds, :])
    sub["A"] = np.ascontiguousarray(x["A"][ds])
    sub["D"] = np.ascontiguousarray(x["D"][ds])
    sub["delta_bias"] = np.ascontiguousarray(x["delta_bias"][ds])
    sgr = {"dy": np.ascontiguousarray(gr["dy"][:, ds, :]),
           "dh_last": np.ascontiguousarray(gr["dh_last"][:, ds, :])}
    ref = oracle_bwd(sub, sgr, io)
    gsub = {k: got[k][:, ds] for k in ("du", "ddelta", "dh0")}
    gsub.update({k: got[k][ds] for k in ("dA", "dD", "ddelta_bias")})
    check(gsub, ref, io, what="long sampled channels",
          keys=("du", "ddelta", "dh0", "dA", "dD", "ddelta_bias"))
    assert np.isfinite(got["dB"]).all() and np.isfinite(got["dC"]).all()


def test_bwd_is_deterministic():
    """Fixed-order reductions: two calls give the same bits."""
    io = W.BF16
    cfg = W.ScanConfig("t", 2, 200, 16, 528, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=21, with_h0=True)
    gr = W.make_scan_grads(cfg, seed=21)
    a = gpu_bwd(x, gr, io)
    b = gpu_bwd(x, gr, io)
    for k in GRAD_KEYS:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


def test_bwd_2p8b_size():
    """The 2.8B-like layer (bf16, B8 D5120 N16 L2048, gate) at full size.  Channel-
    local gradients and dA, dD, the bias gradient are checked on 24 sampled
    channels over all batch rows (their exact oracle needs only those channels);
    dB and dC of batch row 0 against the oracle over all 5120 channels of that row."""
    cfg = W.SCAN_CONFIGS["2p8b"]
    io = cfg.io
    x = W.make_scan_inputs(cfg, seed=0)
    gr = W.make_scan_grads(cfg, seed=0)
    got = gpu_bwd(x, gr, io)
    # sampled channels d (all batch rows)
    ds = np.array([0, 1, 31, 32, 777, 2048, 4095, 5119] +
                  list(np.random.default_rng(2).choice(5120, 16, replace=False)), dtype=np.int64)
    ds = np.unique(ds)
    sub = {k: (None if v is None else v) for k, v in x.items()}
    for k in ("u", "delta", "z"):
        sub[k] = np.ascontiguousarray(x[k][:, ds, :])
    sub["A"] = np.ascontiguousarray(x["A"][ds])
    sub["D"] = np.ascontiguousarray(x["D"][ds])
    sub["delta_bias"] = np.ascontiguousarray(x["delta_bias"][ds])
    sgr = {"dy": np.ascontiguousarray(gr["dy"][:, ds, :]),
           "dh_last": np.ascontiguousarray(gr["dh_last"][:, ds, :])}
    ref = oracle_bwd(sub, sgr, io)
    gsub = {k: got[k][:, ds] for k in ("du", "ddelta", "dz", "dh0")}
    gsub.update({k: got[k][ds] for k in ("dA", "dD", "ddelta_bias")})
    check(gsub, ref, io, what="2p8b sampled channels",
          keys=("du", "ddelta", "dz", "dh0", "dA", "dD", "ddelta_bias"))
    # dB, dC of batch row 0: all channels of that row
    row0 = {k: (v[:1] if k in ("u", "delta", "z", "B", "C") else v) for k, v in x.items()}
    gr0 = {"dy": gr["dy"][:1], "dh_last": gr["dh_last"][:1]}
    ref0 = oracle_bwd(row0, gr0, io)
    check({k: got[k][:1] for k in ("dB", "dC", "du")}, ref0, io, what="2p8b batch row 0",
          keys=("dB", "dC", "du"))


@pytest.mark.parametrize("segments", [0, 4])
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_bwd_large_and_tiny_dt(io, segments):
    """softplus saturation (raw delta up to +60) and vanishing dt (raw down to -60), no D
    skip, zero initial state; unsplit and in four segments."""
    cfg = W.ScanConfig("t", 2, 40, 16, 256, io, gate=True, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=51)
    x["D"] = None
    rng = np.random.default_rng(8)
    x["delta"] = W.encode(rng.uniform(-60, 60, size=x["delta"].shape).astype(np.float32), io)
    gr = W.make_scan_grads(cfg, seed=51)
    check(gpu_bwd(x, gr, io, segments=segments), oracle_bwd(x, gr, io), io,
          what=f"large/tiny dt {io} seg {segments}")


@pytest.mark.parametrize("segments", [0, 4])
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_bwd_vanishing_dt(io, segments):
    """Every step tiny (raw delta in [-60, -20]), no D skip, zero initial state: every
    gradient is built from tiny steps only, so the scale-free error metric sees any
    absolute error of the coefficients (bf16: these CTAs take the series coefficients)."""
    cfg = W.ScanConfig("t", 2, 40, 16, 256, io, gate=True, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=52)
    x["D"] = None
    rng = np.random.default_rng(9)
    x["delta"] = W.encode(rng.uniform(-60, -20, size=x["delta"].shape).astype(np.float32), io)
    gr = W.make_scan_grads(cfg, seed=52)
    check(gpu_bwd(x, gr, io, segments=segments), oracle_bwd(x, gr, io), io,
          what=f"vanishing dt {io} seg {segments}")


def test_bwd_mixed_fast_and_series_ctas():
    """bf16: one 32-channel CTA of each batch row holds a channel of vanishing steps (it
    takes the series coefficients, launched first) next to CTAs on the fast coefficients
    (launched to overlap it); every gradient, including the dB / dC sums over both kinds
    of CTA, against the oracle."""
    io = W.BF16
    cfg = W.ScanConfig("t", 2, 96, 16, 512, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=53, with_h0=True)
    dl = W.to_f64(x["delta"], io).astype(np.float32)
    dl[:, 40, :] = -45.0  # channel 40 (second CTA): dt ~ 3e-20 after the bias
    x["delta"] = W.encode(dl, io)
    gr = W.make_scan_grads(cfg, seed=53)
    check(gpu_bwd(x, gr, io), oracle_bwd(x, gr, io), io, what="mixed CTAs")


def test_bwd_steps_near_fast_threshold():
    """bf16: every step with |dt A| log2(e) from 0.5x to 4x of 2^-16, the lower limit of
    the fast coefficients per CTA, no D skip, zero initial state: CTAs with a step
    below it take the series, the others the fast coefficients."""
    io = W.BF16
    cfg = W.ScanConfig("t", 2, 64, 16, 512, io, gate=False, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=54)
    x["D"] = None
    rng = np.random.default_rng(10)
    q = 2.0 ** -16 * np.exp(rng.uniform(np.log(0.5), np.log(4.0), size=x["delta"].shape))
    # the first CTA's 32 channels stay above the limit throughout (fast coefficients at
    # steps just above it); the second CTA's reach below it (series)
    q[:, :32, :] = np.maximum(q[:, :32, :], 1.05 * 2.0 ** -16)
    dt = q / np.log2(np.e)
    x["delta"] = W.encode(np.log(np.expm1(dt)).astype(np.float32), io)
    gr = W.make_scan_grads(cfg, seed=54)
    check(gpu_bwd(x, gr, io), oracle_bwd(x, gr, io), io, what="near-threshold steps")
