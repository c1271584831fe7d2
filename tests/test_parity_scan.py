"""GPU parity of the selective-scan forward (through the C ABI) against the fp64 oracle.

Tolerances (error metric in tests/helpers.py): 1e-4 for fp32 io, 2e-2 for bf16 io
with fp32 state.  Every configuration runs both kernel families, the channel
kernel at each of its lanes-per-channel splits (1, 2, 4 lanes; a split that would
leave a lane fewer than 4 states is skipped).
"""
import os

import numpy as np
import pytest

import oracle
from selective_state_space_115_b300 import workloads as W
from tests.helpers import H_TOL, TOL, from_torch, rel_err, torch_f32, torch_io

pytestmark = pytest.mark.gpu
ALGOS = ["channel_l1", "channel_l2", "channel_l4", "channel_mixed", "chunk", "segmented"]
FULL_ALGOS = ALGOS + ["auto"]
MIN_DSTATE = {"channel_l2": 8, "channel_l4": 16, "channel_mixed": 16}
NTHREADS = os.cpu_count() or 1
_ORACLE_CACHE = {}
_INPUT_CACHE = {}


def workload_inputs(name):
    """Seeded inputs of a named workload, drawn once per test session."""
    if name not in _INPUT_CACHE:
        _INPUT_CACHE[name] = W.make_scan_inputs(W.SCAN_CONFIGS[name], seed=0)
    return _INPUT_CACHE[name]


def S():
    from selective_state_space_115_b300 import binding
    return binding


def gpu_scan(x, io, algo, softplus=True, return_last_state=False, out=None):
    import torch
    if x["A"].shape[1] < MIN_DSTATE.get(algo, 0):
        pytest.skip(f"{algo} needs dstate >= {MIN_DSTATE[algo]}")
    r = S().scan_fwd(torch_io(x["u"], io), torch_io(x["delta"], io), torch_f32(x["A"]),
                     torch_io(x["B"], io), torch_io(x["C"], io), D=torch_f32(x.get("D")),
                     z=torch_io(x.get("z"), io), delta_bias=torch_f32(x.get("delta_bias")),
                     delta_softplus=softplus, h0=torch_f32(x.get("h0")),
                     return_last_state=return_last_state, algo=algo, out=out)
    torch.cuda.synchronize()
    assert S().read_device_status() == 0
    return r


def f64(x, io):
    return None if x is None else W.to_f64(x, io)


def oracle_full(x, io, softplus=True, return_last_state=False, cache_key=None):
    """The fp64 oracle on all rows (memoised per `cache_key` when given)."""
    if cache_key is not None:
        key = (cache_key, softplus, return_last_state)
        if key not in _ORACLE_CACHE:
            _ORACLE_CACHE[key] = oracle_full(x, io, softplus, return_last_state)
        return _ORACLE_CACHE[key]
    return oracle.scan_fwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                           f64(x["C"], io), D=x.get("D"), z=f64(x.get("z"), io),
                           delta_bias=x.get("delta_bias"), delta_softplus=softplus,
                           h0=x.get("h0"), return_last_state=return_last_state,
                           nthreads=NTHREADS)


def oracle_rows(x, io, rows, return_last_state=False):
    b, d, L = x["u"].shape
    take = lambda a: None if a is None else W.to_f64(a, io).reshape(b * d, L)[rows]  # noqa: E731
    return oracle.scan_rows(rows, take(x["u"]), take(x["delta"]), x["A"], f64(x["B"], io),
                            f64(x["C"], io), b, d, D=x.get("D"), z_rows=take(x.get("z")),
                            delta_bias=x.get("delta_bias"), h0=x.get("h0"),
                            return_last_state=return_last_state)


# ---------------------------------------------------------------------------
# the workloads at full size
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("algo", ALGOS)
def test_tiny(algo):
    cfg = W.SCAN_CONFIGS["tiny"]
    x = W.make_scan_inputs(cfg, seed=0)
    y, hl = gpu_scan(x, cfg.io, algo, return_last_state=True)
    ref, hr = oracle_full(x, cfg.io, return_last_state=True)
    assert rel_err(from_torch(y), ref) <= TOL[cfg.io]
    assert rel_err(from_torch(hl), hr) <= TOL[cfg.io]


@pytest.mark.parametrize("algo", FULL_ALGOS)
def test_130m_full(algo):
    cfg = W.SCAN_CONFIGS["130m"]
    x = workload_inputs("130m")
    y, hl = gpu_scan(x, cfg.io, algo, return_last_state=True)
    ref, hr = oracle_full(x, cfg.io, return_last_state=True, cache_key="130m")
    e = rel_err(from_torch(y), ref)
    print(f"130m {algo}: max rel err {e:.3e}")
    assert e <= TOL[cfg.io]
    assert rel_err(from_torch(hl), hr) <= TOL[cfg.io]


@pytest.mark.parametrize("algo", FULL_ALGOS)
def test_2p8b_full(algo):
    """Mamba-2.8B-like layer (B8 D5120 N16 L2048, bf16 io, gate) at full size: every
    element of y and of h_last against the oracle."""
    cfg = W.SCAN_CONFIGS["2p8b"]
    x = workload_inputs("2p8b")
    y, hl = gpu_scan(x, cfg.io, algo, return_last_state=True)
    ref, hr = oracle_full(x, cfg.io, return_last_state=True, cache_key="2p8b")
    yg = from_torch(y)
    assert np.isfinite(yg).all()
    e, eh = rel_err(yg, ref), rel_err(from_torch(hl), hr)
    print(f"2p8b {algo}: max rel err y {e:.3e}, h_last {eh:.3e} (all {yg.size} elements)")
    assert e <= TOL[cfg.io]
    assert eh <= H_TOL[cfg.io]


@pytest.mark.parametrize("algo", FULL_ALGOS)
def test_long_full(algo):
    """Long-sequence scan (B1 D1536 N16 L131072, bf16 io) at full size: every element
    of y and of h_last against the oracle."""
    cfg = W.SCAN_CONFIGS["long"]
    x = workload_inputs("long")
    y, hl = gpu_scan(x, cfg.io, algo, return_last_state=True)
    ref, hr = oracle_full(x, cfg.io, return_last_state=True, cache_key="long")
    yg = from_torch(y)
    assert np.isfinite(yg).all()
    e, eh = rel_err(yg, ref), rel_err(from_torch(hl), hr)
    print(f"long {algo}: max rel err y {e:.3e}, h_last {eh:.3e} (all {yg.size} elements)")
    assert e <= TOL[cfg.io]
    assert eh <= H_TOL[cfg.io]


# ---------------------------------------------------------------------------
# odd shapes, optional arguments, both dtypes
# ---------------------------------------------------------------------------
SHAPES = [
    # io, batch, dim, dstate, seqlen, gate, h0
    (W.F32, 1, 1, 4, 1, False, False),
    (W.BF16, 1, 3, 8, 3, True, True),
    (W.F32, 2, 37, 16, 69, True, True),       # ragged dim tile and ragged L tail
    (W.BF16, 3, 37, 16, 72, True, False),     # TMA-eligible L, ragged dim
    (W.BF16, 2, 100, 8, 1000, False, True),
    (W.F32, 1, 64, 4, 4096, True, False),
    (W.BF16, 2, 33, 16, 517, True, True),     # L not a multiple of 8: no TMA
    (W.F32, 1, 130, 16, 2, False, True),
]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,h0", SHAPES)
def test_shapes(algo, io, batch, dim, dstate, seqlen, gate, h0):
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=seqlen + dim, with_h0=h0)
    y, hl = gpu_scan(x, io, algo, return_last_state=True)
    ref, hr = oracle_full(x, io, return_last_state=True)
    assert rel_err(from_torch(y), ref) <= TOL[io]
    assert rel_err(from_torch(hl), hr) <= (1e-4 if io == W.F32 else 1e-3)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_optional_arguments_absent(algo, io):
    cfg = W.ScanConfig("t", 2, 40, 16, 256, io, gate=False, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=5)
    x["D"] = None
    x["delta_bias"] = None
    # delta used as dt directly (no softplus): keep it positive
    x32 = np.abs(W.to_f64(x["delta"], io)).astype(np.float32) * np.float32(0.05)
    x["delta"] = W.encode(x32, io)
    y = gpu_scan(x, io, algo, softplus=False)
    ref = oracle_full(x, io, softplus=False)
    assert rel_err(from_torch(y), ref) <= TOL[io]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_zero_and_small_A(algo, io):
    """A == 0 uses the dt limit; tiny |A| must stay accurate (bf16 switches to the
    accurate path)."""
    cfg = W.ScanConfig("t", 1, 48, 8, 512, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=11)
    A = x["A"].copy()
    A[0, :] = 0.0
    A[5, 3] = -1e-7
    A[9, :] = -np.float32(1e-3) * np.arange(1, 9, dtype=np.float32)
    A[20, 1] = 0.0
    x["A"] = A
    y = gpu_scan(x, io, algo)
    ref = oracle_full(x, io)
    assert rel_err(from_torch(y), ref) <= TOL[io]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_large_and_tiny_dt(algo, io):
    """softplus saturation (raw delta up to +60) and vanishing dt (raw down to -60),
    with no D skip and a zero initial state."""
    cfg = W.ScanConfig("t", 1, 32, 16, 256, io, gate=True, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=12)
    x["D"] = None
    rng = np.random.default_rng(3)
    x["delta"] = W.encode(rng.uniform(-60, 60, size=x["delta"].shape).astype(np.float32), io)
    y = gpu_scan(x, io, algo)
    assert rel_err(from_torch(y), oracle_full(x, io)) <= TOL[io]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_vanishing_dt(algo, io):
    """Every step tiny (raw delta in [-60, -20]: dt between 1e-26 and 2e-9), no D skip,
    zero initial state: the state and the output are built from tiny steps only (the
    "keep the state" end of the selection mechanism), so the output is tiny too and the
    scale-free error metric sees any absolute error of the update."""
    cfg = W.ScanConfig("t", 2, 40, 16, 512, io, gate=True, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=18)
    x["D"] = None
    rng = np.random.default_rng(4)
    x["delta"] = W.encode(rng.uniform(-60, -20, size=x["delta"].shape).astype(np.float32), io)
    y = from_torch(gpu_scan(x, io, algo))
    ref = oracle_full(x, io)
    assert np.abs(y).max() > 0
    assert rel_err(y, ref) <= TOL[io]


@pytest.mark.parametrize("algo", ALGOS)
def test_steps_near_fast_threshold(algo):
    """bf16: steps with |dt A| log2(e) from 0.5x to 4x of the fast update's lower limit
    (2^-15), no D skip, zero initial state.  Blocks whose smallest step is below the
    limit take the accurate update, the rest the fast one; both must stay within
    tolerance when the state is built only from such steps."""
    io = W.BF16
    cfg = W.ScanConfig("t", 2, 64, 16, 1024, io, gate=False, dt_bias=False, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=19)
    x["D"] = None
    rng = np.random.default_rng(5)
    q = 2.0 ** -15 * np.exp(rng.uniform(np.log(0.5), np.log(4.0), size=x["delta"].shape))
    dt = q / np.log2(np.e)  # min |A| = 1: q = dt * log2(e) at the state with A = -1
    x["delta"] = W.encode(np.log(np.expm1(dt)).astype(np.float32), io)
    y = from_torch(gpu_scan(x, io, algo))
    ref = oracle_full(x, io)
    e = rel_err(y, ref)
    print(f"near-threshold steps {algo}: max rel err {e:.3e}")
    assert e <= TOL[io]


# ---------------------------------------------------------------------------
# memory safety, fallbacks, properties
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io", [W.F32, W.BF16])
def test_guard_bands_untouched(algo, io):
    """y lives inside a NaN-filled buffer: the bands around it must stay NaN and y
    must be fully written (no NaN left)."""
    import torch
    cfg = W.ScanConfig("t", 2, 37, 16, 136, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=13)
    n = cfg.batch * cfg.dim * cfg.seqlen
    guard = 4096
    dt = torch.float32 if io == W.F32 else torch.bfloat16
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=dt, device="cuda")
    y = buf[guard:guard + n].view(cfg.batch, cfg.dim, cfg.seqlen)
    gpu_scan(x, io, algo, out=y)
    b = from_torch(buf)
    assert np.isnan(b[:guard]).all() and np.isnan(b[guard + n:]).all()
    assert np.isfinite(b[guard:guard + n]).all()
    ref = oracle_full(x, io)
    assert rel_err(from_torch(y), ref) <= TOL[io]


@pytest.mark.parametrize("algo", ALGOS)
def test_unaligned_pointers_fall_back(algo):
    """Tensors offset by one element from a 16-byte boundary take the element-load path."""
    import torch
    io = W.BF16
    cfg = W.ScanConfig("t", 1, 24, 16, 128, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=14)

    def shifted(a):
        t = torch_io(a, io)
        big = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = big[1:].view(t.shape)
        v.copy_(t)
        return v

    r = S().scan_fwd(shifted(x["u"]), shifted(x["delta"]), torch_f32(x["A"]), shifted(x["B"]),
                     shifted(x["C"]), D=torch_f32(x["D"]), z=shifted(x["z"]),
                     delta_bias=torch_f32(x["delta_bias"]), algo=algo)
    torch.cuda.synchronize()
    assert rel_err(from_torch(r), oracle_full(x, io)) <= TOL[io]


@pytest.mark.parametrize("algo", ALGOS)
def test_split_invariance(algo):
    """scan(0..L) == scan(0..m) then scan(m..L) from h_last (checkpoint / resume)."""
    io = W.F32
    cfg = W.ScanConfig("t", 2, 40, 16, 1024, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=15)
    m = 384
    part = lambda a, sl: None if a is None else np.ascontiguousarray(a[..., sl])  # noqa: E731
    xa = {k: (part(v, slice(0, m)) if k in ("u", "delta", "z", "B", "C") else v)
          for k, v in x.items()}
    xb = {k: (part(v, slice(m, None)) if k in ("u", "delta", "z", "B", "C") else v)
          for k, v in x.items()}
    y, hl = gpu_scan(x, io, algo, return_last_state=True)
    ya, ha = gpu_scan(xa, io, algo, return_last_state=True)
    xb["h0"] = from_torch(ha).astype(np.float32)
    yb, hb = gpu_scan(xb, io, algo, return_last_state=True)
    yy = np.concatenate([from_torch(ya), from_torch(yb)], axis=-1)
    assert rel_err(yy, from_torch(y)) <= 1e-5
    assert rel_err(from_torch(hb), from_torch(hl)) <= 1e-5


@pytest.mark.parametrize("algo", ALGOS)
def test_linearity_in_u(algo):
    io = W.F32
    cfg = W.ScanConfig("t", 1, 64, 16, 512, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x1 = W.make_scan_inputs(cfg, seed=16)
    x2 = dict(x1)
    x2["u"] = np.random.default_rng(7).standard_normal(x1["u"].shape).astype(np.float32)
    x12 = dict(x1)
    x12["u"] = (np.float32(1.5) * x1["u"] - np.float32(0.5) * x2["u"]).astype(np.float32)
    y1 = from_torch(gpu_scan(x1, io, algo))
    y2 = from_torch(gpu_scan(x2, io, algo))
    y12 = from_torch(gpu_scan(x12, io, algo))
    assert rel_err(y12, 1.5 * y1 - 0.5 * y2) <= 1e-4


@pytest.mark.parametrize("algo", ALGOS)
def test_deterministic(algo):
    cfg = W.ScanConfig("t", 2, 96, 16, 640, W.BF16, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=17)
    a = from_torch(gpu_scan(x, cfg.io, algo))
    b = from_torch(gpu_scan(x, cfg.io, algo))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("io,dstate", [(W.BF16, 16), (W.F32, 16), (W.BF16, 8)])
def test_lane_splits_are_bit_identical(io, dstate):
    """1, 2 and 4 lanes per channel evaluate every state update, the contraction
    (per-4-state pair sums, then a tree) and the per-position work in the same order,
    so they agree bit for bit -- including a channel group that takes the accurate
    arithmetic (small |A|) next to groups on the fast path."""
    cfg = W.ScanConfig("t", 2, 160, dstate, 512, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=23, with_h0=True)
    A = x["A"].copy()
    A[40, 2] = -1e-3  # channels 32..63 take the accurate path
    x["A"] = A
    outs = []
    for algo in ("channel_l1", "channel_l2", "channel_l4"):
        if dstate < MIN_DSTATE.get(algo, 0):
            continue
        y, hl = gpu_scan(x, io, algo, return_last_state=True)
        outs.append((algo, from_torch(y), from_torch(hl)))
    for algo, y, hl in outs[1:]:
        assert np.array_equal(y, outs[0][1]), algo
        assert np.array_equal(hl, outs[0][2]), algo
    assert rel_err(outs[0][1], oracle_full(x, io)) <= TOL[io]


def test_mixed_split_matches_one_lane_bit_for_bit():
    """150 tiles of 128 channels on a 148-SM B300: one one-lane CTA per SM plus 2
    tiles run as eight 32-channel four-lane CTAs; the roles are taken at run time,
    and the result equals the one-lane-per-channel launch bit for bit."""
    io = W.BF16
    cfg = W.ScanConfig("t", 2, 9600, 16, 256, io, gate=True, dt_bias=True, d_skip="normal",
                       description="")
    x = W.make_scan_inputs(cfg, seed=29, with_h0=True)
    ym, hm = gpu_scan(x, io, "channel_mixed", return_last_state=True)
    y1, h1 = gpu_scan(x, io, "channel_l1", return_last_state=True)
    assert np.array_equal(from_torch(ym), from_torch(y1))
    assert np.array_equal(from_torch(hm), from_torch(h1))
    rows = np.array([0, 127, 128, 9599, 9600 + 9471, 9600 + 9472, 2 * 9600 - 1], dtype=np.int64)
    ref = oracle_rows(x, io, rows)
    assert rel_err(from_torch(ym).reshape(-1, cfg.seqlen)[rows], ref) <= TOL[io]


EULER_CASES = [
    # io, batch, dim, dstate, seqlen, gate, h0
    (W.F32, 2, 37, 16, 69, True, True),
    (W.BF16, 2, 160, 16, 512, True, True),
    (W.BF16, 1, 40, 8, 1000, False, False),
]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("io,batch,dim,dstate,seqlen,gate,h0", EULER_CASES)
def test_euler_input_term(algo, io, batch, dim, dstate, seqlen, gate, h0):
    """Bbar = dt B (Mamba_Model_Report.md section 4.2) on every kernel family."""
    import torch
    if dstate < MIN_DSTATE.get(algo, 0):
        pytest.skip(f"{algo} needs dstate >= {MIN_DSTATE[algo]}")
    cfg = W.ScanConfig("t", batch, dim, dstate, seqlen, io, gate=gate, dt_bias=True,
                       d_skip="normal", description="")
    x = W.make_scan_inputs(cfg, seed=41 + seqlen, with_h0=h0)
    y, hl = S().scan_fwd(torch_io(x["u"], io), torch_io(x["delta"], io), torch_f32(x["A"]),
                         torch_io(x["B"], io), torch_io(x["C"], io), D=torch_f32(x["D"]),
                         z=torch_io(x.get("z"), io), delta_bias=torch_f32(x["delta_bias"]),
                         h0=torch_f32(x.get("h0")), return_last_state=True, algo=algo,
                         discretization="euler")
    torch.cuda.synchronize()
    assert S().read_device_status() == 0
    ref, hr = oracle.scan_fwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                              f64(x["C"], io), D=x["D"], z=f64(x.get("z"), io),
                              delta_bias=x["delta_bias"], h0=x.get("h0"), return_last_state=True,
                              nthreads=NTHREADS, discretization="euler")
    assert rel_err(from_torch(y), ref) <= TOL[io]
    assert rel_err(from_torch(hl), hr) <= (1e-4 if io == W.F32 else 1e-3)
    # and it is not the ZOH result
    zoh = oracle.scan_fwd(f64(x["u"], io), f64(x["delta"], io), x["A"], f64(x["B"], io),
                          f64(x["C"], io), D=x["D"], z=f64(x.get("z"), io),
                          delta_bias=x["delta_bias"], h0=x.get("h0"), nthreads=NTHREADS)
    assert rel_err(from_torch(y), zoh) > 10 * TOL[io]


def test_auto_matches_explicit_choice():
    cfg = W.SCAN_CONFIGS["2p8b"]
    x = W.make_scan_inputs(cfg, seed=0, batch=2)  # 10240 channels: the channel kernel
    a = from_torch(gpu_scan(x, cfg.io, "auto"))
    b = from_torch(gpu_scan(x, cfg.io, "channel"))
    assert np.array_equal(a, b)
    cfg = W.SCAN_CONFIGS["130m"]
    x = W.make_scan_inputs(cfg, seed=0, seqlen=256)  # 3072 channels: the chunk kernel
    a = from_torch(gpu_scan(x, cfg.io, "auto"))
    b = from_torch(gpu_scan(x, cfg.io, "chunk"))
    assert np.array_equal(a, b)
