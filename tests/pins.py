"""Pins for the fp64 oracle: checks against facts fixed by the pages and by
mathematics, independent of the oracle's own loop.

Each pin takes an ``oracle.Oracle`` and raises AssertionError on a mismatch, so
the same pins can be run against deliberately broken copies of the oracle
(tests/test_oracle_pins.py::test_pins_catch_planted_mistakes).

Sources of each fact:
  * continuous system h'(t) = A h(t) + B x(t), y = C h (+ D x), input held over
    each step (zero-order hold) of length delta_k:
    "mamba 学习" (fakeeyes2wo), sections "MAMBA" and "引入可变步长 Δ_k";
    velog Mamba review, section 2 "Discretization".
  * inclusive recurrence h_k = Abar h_{k-1} + Bbar x_k, y_k = C h_k:
    velog Mamba review, section 2 "Discretization", item 3.
  * unrolled sum h_k = Abar^k h_0 + sum_j Abar^{k-1-j} Bbar x_j and the
    convolution kernel K_l = C Abar^l Bbar for constant parameters:
    "mamba 学习", section "离散 SSM 的卷积形式与时不变性" (shifted to the
    inclusive convention above).
  * ZOH integral needs invertible A; its A -> 0 limit is delta * B:
    "mamba 学习", section "MAMBA".
  * linearity of the SSM in its input: velog Mamba review, section 2 "LTI".
  * dt = softplus(raw + bias): velog Mamba review, section 3.2; the D skip:
    "mamba 学习", section "SSM 状态空间模型"; gate y * silu(z):
    Mamba_Model_Report.md, section 3 (MambaBlock.forward).
  * single-token step equals the scan: Mamba_Model_Report.md, section 6.
  * Euler input term Bbar = delta * B with the same Abar = exp(delta A):
    Mamba_Model_Report.md, section 4.2 (selective_scan: deltaB = delta * B).
  * causal depthwise conv1d (groups = channels, padding W - 1, first L outputs)
    then silu, and its decode cache of the last W - 1 inputs:
    Mamba_Model_Report.md, sections 3 (MambaBlock.forward) and 6 (step).
  * the scan's gradient (Mamba_Model_Report.md, section 4.1: the backward of
    the recurrence through a reverse scan) is the derivative of the forward:
    central finite differences of the pinned forward oracle fix every partial
    derivative; a function linear in some inputs equals the sum of each input
    times its gradient (Euler's theorem on homogeneous functions), exactly.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.integrate import solve_ivp


def _rng(seed):
    return np.random.default_rng(1000 + seed)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    if not np.all(err <= lim):
        i = int(np.argmax(err - lim))
        raise AssertionError(f"{what}: max excess at flat index {i}: got {a.flat[i]!r}, "
                             f"expected {b.flat[i]!r}")


# ---------------------------------------------------------------------------
# 1. zero-order hold, checked by integrating the continuous system
# ---------------------------------------------------------------------------
def pin_zoh_matches_ode(orc):
    """Integrate h' = A h + B_k x_k over [t_k, t_k + delta_k] with an ODE solver
    (no closed form used) and compare y_k = C_k h(t_k + delta_k) + D x_k."""
    rng = _rng(1)
    n, L = 4, 7
    A = np.array([[-1.0, -2.5, -0.003, 0.0]])          # includes A = 0 exactly
    dts = rng.uniform(0.05, 0.9, size=L)
    x = rng.standard_normal(L)
    B = rng.standard_normal((n, L))
    C = rng.standard_normal((n, L))
    Dd = 0.7
    h0 = rng.standard_normal(n) * 0.5
    h = h0.copy()
    y_ref = np.empty(L)
    a = A[0]
    for k in range(L):
        bx = B[:, k] * x[k]
        sol = solve_ivp(lambda t, hh: a * hh + bx, (0.0, dts[k]), h, method="DOP853",
                        rtol=1e-13, atol=1e-15)
        h = sol.y[:, -1]
        y_ref[k] = C[:, k] @ h + Dd * x[k]
    y = orc.scan_fwd(x[None, None, :], dts[None, None, :], A, B[None], C[None],
                     D=np.array([Dd]), delta_softplus=False, h0=h0[None, None, :])
    _close(y[0, 0], y_ref, rtol=1e-9, atol=1e-11, what="ZOH vs ODE")


# ---------------------------------------------------------------------------
# 2. brute-force unrolled sum (no loop-carried state)
# ---------------------------------------------------------------------------
def _unrolled(u, dt, A, B, C, D, h0, euler=False):
    """y_k = sum_n C[n,k] (prod_{i<=k} Abar_i h0 + sum_{j<=k} prod_{j<i<=k} Abar_i Bbar_j u_j) + D u_k"""
    L = u.shape[0]
    n = A.shape[0]
    Abar = np.exp(dt[:, None] * A[None, :])                        # [L, n]
    with np.errstate(divide="ignore", invalid="ignore"):
        coef = np.where(A[None, :] == 0.0, dt[:, None],
                        np.expm1(dt[:, None] * A[None, :]) / A[None, :])
    if euler:
        coef = np.broadcast_to(dt[:, None], (L, n))
    Bbar_u = coef * B.T * u[:, None]                                # [L, n]
    y = np.empty(L)
    for k in range(L):
        hk = np.prod(Abar[: k + 1], axis=0) * h0
        for j in range(k + 1):
            hk = hk + np.prod(Abar[j + 1: k + 1], axis=0) * Bbar_u[j]
        y[k] = C[:, k] @ hk + D * u[k]
    return y


def pin_unrolled_sum(orc):
    rng = _rng(2)
    b, d, n, L = 2, 3, 5, 37
    u = rng.standard_normal((b, d, L))
    raw = rng.standard_normal((b, d, L))
    bias = rng.uniform(-3.0, 0.5, size=d)
    A = -rng.uniform(0.2, 4.0, size=(d, n))
    A[1, 2] = 0.0
    B = rng.standard_normal((b, n, L))
    C = rng.standard_normal((b, n, L))
    D = rng.standard_normal(d)
    h0 = rng.standard_normal((b, d, n))
    y, hl = orc.scan_fwd(u, raw, A, B, C, D=D, delta_bias=bias, h0=h0, return_last_state=True)
    for bi in range(b):
        for di in range(d):
            x = raw[bi, di] + bias[di]
            dt = np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)   # softplus, stable form
            y_ref = _unrolled(u[bi, di], dt, A[di], B[bi], C[bi], D[di], h0[bi, di])
            _close(y[bi, di], y_ref, rtol=1e-11, atol=1e-12, what=f"unrolled sum ({bi},{di})")


# ---------------------------------------------------------------------------
# 3. LTI special case: convolution with K_l = sum_n C_n Abar_n^l Bbar_n
# ---------------------------------------------------------------------------
def pin_lti_convolution(orc):
    rng = _rng(3)
    n, L = 6, 64
    A = -np.arange(1, n + 1, dtype=np.float64)[None, :] * 0.7
    dt = 0.13
    Bc = rng.standard_normal(n)
    Cc = rng.standard_normal(n)
    Dd = -0.4
    u = rng.standard_normal(L)
    B = np.repeat(Bc[:, None], L, axis=1)[None]
    C = np.repeat(Cc[:, None], L, axis=1)[None]
    y = orc.scan_fwd(u[None, None], np.full((1, 1, L), dt), A, B, C, D=np.array([Dd]),
                     delta_softplus=False)[0, 0]
    Abar = np.exp(dt * A[0])
    Bbar = np.expm1(dt * A[0]) / A[0] * Bc
    K = np.array([np.sum(Cc * Abar ** l * Bbar) for l in range(L)])
    y_ref = np.convolve(u, K)[:L] + Dd * u
    _close(y, y_ref, rtol=1e-11, atol=1e-12, what="LTI convolution")


# ---------------------------------------------------------------------------
# 4. geometric series: N = 1, x = 1, constant parameters
# ---------------------------------------------------------------------------
def pin_geometric_series(orc):
    L = 50
    for a, dt, bval, cval in [(-1.0, 0.1, 1.0, 1.0), (-3.0, 0.02, 0.5, -2.0),
                              (-0.25, 1.7, -1.5, 0.3)]:
        A = np.array([[a]])
        y = orc.scan_fwd(np.ones((1, 1, L)), np.full((1, 1, L), dt), A,
                         np.full((1, 1, L), bval), np.full((1, 1, L), cval),
                         delta_softplus=False)[0, 0]
        Abar = math.exp(a * dt)
        Bbar = (Abar - 1.0) / a * bval
        k = np.arange(L)
        h_ref = Bbar * (1.0 - Abar ** (k + 1)) / (1.0 - Abar)
        _close(y, cval * h_ref, rtol=1e-11, atol=1e-13, what=f"geometric series a={a}")


# ---------------------------------------------------------------------------
# 5. A -> 0 limit of the ZOH input coefficient
# ---------------------------------------------------------------------------
def pin_zoh_small_A(orc):
    dt, bval, uval = 0.37, 1.3, -0.8
    # A == 0 exactly: Bbar = dt * B (the integral of e^{0 tau} over [0, dt])
    y0 = orc.scan_fwd(np.full((1, 1, 1), uval), np.full((1, 1, 1), dt), np.zeros((1, 1)),
                      np.full((1, 1, 1), bval), np.ones((1, 1, 1)), delta_softplus=False)
    if y0[0, 0, 0] != dt * bval * uval:
        raise AssertionError(f"A=0: got {y0[0, 0, 0]!r}, expected {dt * bval * uval!r}")
    # tiny A: coef = dt * (1 + q/2 + q^2/6 + q^3/24), q = dt*A, truncation < q^4
    for p in range(3, 13):
        a = -(10.0 ** -p)
        q = dt * a
        ref = dt * (1 + q / 2 + q * q / 6 + q ** 3 / 24) * bval * uval
        y = orc.scan_fwd(np.full((1, 1, 1), uval), np.full((1, 1, 1), dt), np.array([[a]]),
                         np.full((1, 1, 1), bval), np.ones((1, 1, 1)), delta_softplus=False)
        _close(y[0, 0, 0], ref, rtol=1e-13, what=f"A=-1e-{p}")


# ---------------------------------------------------------------------------
# 6. linearity in u (delta, B, C, z fixed; h0 = 0)
# ---------------------------------------------------------------------------
def pin_linearity(orc):
    rng = _rng(6)
    b, d, n, L = 1, 3, 4, 40
    raw = rng.standard_normal((b, d, L))
    A = -rng.uniform(0.5, 3.0, size=(d, n))
    B = rng.standard_normal((b, n, L))
    C = rng.standard_normal((b, n, L))
    D = rng.standard_normal(d)
    z = rng.standard_normal((b, d, L))
    u1 = rng.standard_normal((b, d, L))
    u2 = rng.standard_normal((b, d, L))
    al, be = 1.7, -0.6
    y1 = orc.scan_fwd(u1, raw, A, B, C, D=D, z=z)
    y2 = orc.scan_fwd(u2, raw, A, B, C, D=D, z=z)
    y12 = orc.scan_fwd(al * u1 + be * u2, raw, A, B, C, D=D, z=z)
    _close(y12, al * y1 + be * y2, rtol=1e-11, atol=1e-12, what="linearity in u")


# ---------------------------------------------------------------------------
# 7. parameter plumbing: softplus(raw + bias), D skip, silu gate order
# ---------------------------------------------------------------------------
def pin_softplus_bias_gate(orc):
    import torch
    import torch.nn.functional as F

    rng = _rng(7)
    L = 64
    raw = rng.uniform(-25.0, 25.0, size=L)
    bias = 0.75
    # A = 0, B = C = u = 1, h0 = 0, one step per row: y = dt = softplus(raw + bias)
    y = orc.scan_fwd(np.ones((1, L, 1)), raw[None, :, None], np.zeros((L, 1)),
                     np.ones((1, 1, 1)), np.ones((1, 1, 1)),
                     delta_bias=np.full(L, bias))[0, :, 0]
    ref = F.softplus(torch.tensor(raw + bias, dtype=torch.float64), beta=1.0,
                     threshold=1e9).numpy()
    _close(y, ref, rtol=1e-14, atol=1e-300, what="softplus(raw + bias)")
    # B = 0 keeps h = 0, so y = D u silu(z): D skip enters before the gate
    u = rng.standard_normal(L)
    z = rng.uniform(-12.0, 12.0, size=L)
    Dv = rng.standard_normal(L)
    y = orc.scan_fwd(u[None, :, None], np.zeros((1, L, 1)), -np.ones((L, 1)),
                     np.zeros((1, 1, 1)), np.ones((1, 1, 1)), D=Dv, z=z[None, :, None])[0, :, 0]
    ref = Dv * u * F.silu(torch.tensor(z, dtype=torch.float64)).numpy()
    _close(y, ref, rtol=1e-14, atol=1e-300, what="D skip then silu gate")


# ---------------------------------------------------------------------------
# 8. decode step == scan, and split invariance through h0 / h_last
# ---------------------------------------------------------------------------
def pin_step_equals_scan(orc):
    rng = _rng(8)
    b, d, n, L = 2, 3, 4, 12
    u = rng.standard_normal((b, d, L))
    raw = rng.standard_normal((b, d, L))
    bias = rng.uniform(-4, 0, size=d)
    A = -rng.uniform(0.5, 3.0, size=(d, n))
    B = rng.standard_normal((b, n, L))
    C = rng.standard_normal((b, n, L))
    D = rng.standard_normal(d)
    z = rng.standard_normal((b, d, L))
    h0 = rng.standard_normal((b, d, n)) * 0.3
    y, hl = orc.scan_fwd(u, raw, A, B, C, D=D, z=z, delta_bias=bias, h0=h0,
                         return_last_state=True)
    h = h0.copy()
    for l in range(L):
        yl, h = orc.state_update(h, u[:, :, l], raw[:, :, l], A, B[:, :, l], C[:, :, l], D=D,
                                 z=z[:, :, l], delta_bias=bias)
        _close(yl, y[:, :, l], rtol=1e-13, atol=1e-14, what=f"step {l} vs scan")
    _close(h, hl, rtol=1e-13, atol=1e-14, what="final state: steps vs scan")


def pin_split_invariance(orc):
    rng = _rng(9)
    b, d, n, L, m = 1, 2, 4, 30, 11
    u = rng.standard_normal((b, d, L))
    raw = rng.standard_normal((b, d, L))
    A = -rng.uniform(0.5, 3.0, size=(d, n))
    B = rng.standard_normal((b, n, L))
    C = rng.standard_normal((b, n, L))
    D = rng.standard_normal(d)
    y, hl = orc.scan_fwd(u, raw, A, B, C, D=D, return_last_state=True)
    ya, ha = orc.scan_fwd(u[..., :m], raw[..., :m], A, B[..., :m], C[..., :m], D=D,
                          return_last_state=True)
    yb, hb = orc.scan_fwd(u[..., m:], raw[..., m:], A, B[..., m:], C[..., m:], D=D, h0=ha,
                          return_last_state=True)
    _close(np.concatenate([ya, yb], axis=-1), y, rtol=1e-13, atol=1e-14, what="split y")
    _close(hb, hl, rtol=1e-13, atol=1e-14, what="split h_last")


def pin_rows_match_full(orc):
    rng = _rng(10)
    b, d, n, L = 2, 5, 4, 20
    u = rng.standard_normal((b, d, L))
    raw = rng.standard_normal((b, d, L))
    A = -rng.uniform(0.5, 3.0, size=(d, n))
    B = rng.standard_normal((b, n, L))
    C = rng.standard_normal((b, n, L))
    z = rng.standard_normal((b, d, L))
    h0 = rng.standard_normal((b, d, n))
    y, hl = orc.scan_fwd(u, raw, A, B, C, z=z, h0=h0, return_last_state=True)
    rows = [0, 3, 7, 9]
    uf, rf, zf = u.reshape(b * d, L), raw.reshape(b * d, L), z.reshape(b * d, L)
    yr, hr = orc.scan_rows(rows, uf[rows], rf[rows], A, B, C, b, d, z_rows=zf[rows], h0=h0,
                           return_last_state=True)
    _close(yr, y.reshape(b * d, L)[rows], rtol=0, atol=0, what="scan_rows")
    _close(hr, hl.reshape(b * d, n)[rows], rtol=0, atol=0, what="scan_rows h_last")


# ---------------------------------------------------------------------------
# 10. the Euler input term (Bbar = dt B, Abar unchanged)
# ---------------------------------------------------------------------------
def pin_euler_unrolled_sum(orc):
    """Brute-force unrolled sum with Bbar_j = dt_j B_j, through the scan and the
    decode step (no loop-carried state in the reference)."""
    rng = _rng(11)
    b, d, n, L = 1, 3, 4, 29
    u = rng.standard_normal((b, d, L))
    raw = rng.standard_normal((b, d, L))
    bias = rng.uniform(-3.0, 0.5, size=d)
    A = -rng.uniform(0.2, 4.0, size=(d, n))
    A[2, 1] = 0.0
    B = rng.standard_normal((b, n, L))
    C = rng.standard_normal((b, n, L))
    D = rng.standard_normal(d)
    h0 = rng.standard_normal((b, d, n))
    y = orc.scan_fwd(u, raw, A, B, C, D=D, delta_bias=bias, h0=h0, discretization="euler")
    h = h0.copy()
    for l in range(L):
        yl, h = orc.state_update(h, u[:, :, l], raw[:, :, l], A, B[:, :, l], C[:, :, l], D=D,
                                 delta_bias=bias, discretization="euler")
        _close(yl, y[:, :, l], rtol=1e-13, atol=1e-14, what=f"euler step {l} vs scan")
    for di in range(d):
        x = raw[0, di] + bias[di]
        dt = np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)
        y_ref = _unrolled(u[0, di], dt, A[di], B[0], C[0], D[di], h0[0, di], euler=True)
        _close(y[0, di], y_ref, rtol=1e-11, atol=1e-12, what=f"euler unrolled sum (0,{di})")


def pin_euler_geometric_and_first_order(orc):
    """N = 1, x = 1, constant parameters: h_k = dt B (1 - Abar^{k+1}) / (1 - Abar).
    One step from h = 0: ZOH minus Euler is (expm1(q)/q - 1) dt B u = (q/2 + q^2/6 +
    ...) dt B u, q = dt A (both input terms pinned against each other)."""
    L = 40
    for a, dt, bval in [(-1.0, 0.1, 1.0), (-2.5, 0.37, -0.7)]:
        A = np.array([[a]])
        y = orc.scan_fwd(np.ones((1, 1, L)), np.full((1, 1, L), dt), A,
                         np.full((1, 1, L), bval), np.ones((1, 1, L)), delta_softplus=False,
                         discretization="euler")[0, 0]
        Abar = math.exp(a * dt)
        k = np.arange(L)
        _close(y, dt * bval * (1.0 - Abar ** (k + 1)) / (1.0 - Abar), rtol=1e-12, atol=1e-14,
               what=f"euler geometric series a={a}")
    dt, bval, uval = 1e-3, 0.9, 1.3
    for a in (-0.5, -3.0):
        args = (np.full((1, 1, 1), uval), np.full((1, 1, 1), dt), np.array([[a]]),
                np.full((1, 1, 1), bval), np.ones((1, 1, 1)))
        yz = orc.scan_fwd(*args, delta_softplus=False)[0, 0, 0]
        ye = orc.scan_fwd(*args, delta_softplus=False, discretization="euler")[0, 0, 0]
        q = dt * a
        _close(ye, dt * bval * uval, rtol=1e-15, what="euler one step")
        _close(yz - ye, (q / 2 + q * q / 6 + q ** 3 / 24) * dt * bval * uval, rtol=1e-6,
               what="zoh - euler, first order")


# ---------------------------------------------------------------------------
# 11. causal depthwise convolution (MambaBlock conv1d, and its decode cache)
# ---------------------------------------------------------------------------
def pin_conv1d_matches_convolution(orc):
    """Each channel's output is the full linear convolution of its input with the
    reversed filter, truncated to the first L outputs (np.convolve), plus the bias,
    then silu; and the same as torch's grouped Conv1d with padding W - 1."""
    import torch
    import torch.nn.functional as F

    rng = _rng(12)
    b, d, L = 2, 5, 23
    for width in (2, 4, 7):
        x = rng.standard_normal((b, d, L))
        w = rng.standard_normal((d, width))
        bias = rng.standard_normal(d)
        out = orc.conv1d_fwd(x, w, bias, apply_silu=False)
        outs = orc.conv1d_fwd(x, w, bias, apply_silu=True)
        for bi in range(b):
            for di in range(d):
                ref = np.convolve(x[bi, di], w[di, ::-1])[:L] + bias[di]
                _close(out[bi, di], ref, rtol=1e-13, atol=1e-13, what=f"conv W={width}")
        tx = torch.tensor(x, dtype=torch.float64)
        ref = F.conv1d(tx, torch.tensor(w[:, None, :]), torch.tensor(bias), padding=width - 1,
                       groups=d)[:, :, :L]
        _close(out, ref.numpy(), rtol=1e-13, atol=1e-13, what=f"torch conv1d W={width}")
        _close(outs, F.silu(ref).numpy(), rtol=1e-13, atol=1e-13, what=f"conv + silu W={width}")


def pin_conv1d_state_and_step(orc):
    """A carried-in window continues the sequence (two halves with the state passed
    on equal one pass), and the decode update applied position by position equals
    the full convolution, its cache equal to the last W - 1 inputs."""
    rng = _rng(13)
    b, d, L, m, width = 2, 3, 17, 6, 4
    x = rng.standard_normal((b, d, L))
    w = rng.standard_normal((d, width))
    bias = rng.standard_normal(d)
    s0 = rng.standard_normal((b, d, width - 1))
    full, s_end = orc.conv1d_fwd(x, w, bias, state_in=s0, return_state=True)
    ya, sa = orc.conv1d_fwd(x[..., :m], w, bias, state_in=s0, return_state=True)
    yb, sb = orc.conv1d_fwd(x[..., m:], w, bias, state_in=sa, return_state=True)
    _close(np.concatenate([ya, yb], -1), full, rtol=1e-14, atol=1e-14, what="conv halves")
    _close(sb, s_end, rtol=0, atol=0, what="conv state after halves")
    _close(s_end, x[..., L - (width - 1):], rtol=0, atol=0, what="conv state = last inputs")
    st = s0.copy()
    for l in range(L):
        yl, st = orc.conv1d_update(st, x[..., l], w, bias)
        _close(yl, full[..., l], rtol=1e-14, atol=1e-14, what=f"conv step {l}")
    _close(st, s_end, rtol=0, atol=0, what="conv cache after steps")
    # without a state the inputs before position 0 are zero: a lone first position
    y1 = orc.conv1d_fwd(x[..., :1], w, bias, apply_silu=False)
    _close(y1[..., 0], w[None, :, -1] * x[..., 0] + bias[None, :], rtol=1e-15, atol=1e-15,
           what="first position, zero history")


# ---------------------------------------------------------------------------
# gradient of the scan
# ---------------------------------------------------------------------------
def _bwd_case(seed, euler=False, softplus=True, gate=True, skip=True):
    rng = _rng(seed)
    b, d, n, L = 2, 3, 4, 6
    case = {
        "u": rng.standard_normal((b, d, L)),
        "delta": (rng.standard_normal((b, d, L)) if softplus
                  else rng.uniform(0.05, 0.8, size=(b, d, L))),
        "A": -rng.uniform(0.5, 3.0, size=(d, n)),
        "B": rng.standard_normal((b, n, L)),
        "C": rng.standard_normal((b, n, L)),
        "D": rng.standard_normal(d) if skip else None,
        "z": rng.standard_normal((b, d, L)) if gate else None,
        "delta_bias": rng.uniform(-1.0, 0.5, size=d),
        "h0": rng.standard_normal((b, d, n)) * 0.5,
    }
    # the A -> 0 limit and the small-|dt A| series branch of dcoef/dA
    case["A"][0, 1] = 0.0
    case["A"][1, 2] = -5e-4
    case["A"][2, 0] = 3e-4
    dy = rng.standard_normal((b, d, L))
    dhl = rng.standard_normal((b, d, n))
    return case, dy, dhl, dict(delta_softplus=softplus,
                               discretization="euler" if euler else "zoh")


def _loss(orc, case, dy, dhl, kw):
    y, hl = orc.scan_fwd(case["u"], case["delta"], case["A"], case["B"], case["C"],
                         D=case["D"], z=case["z"], delta_bias=case["delta_bias"],
                         h0=case["h0"], return_last_state=True, **kw)
    return float(np.sum(dy * y) + np.sum(dhl * hl))


def pin_bwd_finite_differences(orc):
    """Every gradient against central differences of the forward oracle's
    loss sum(dy * y) + sum(dh_last * h_last), with and without each option."""
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}
    variants = [dict(), dict(euler=True), dict(softplus=False, gate=False, skip=False)]
    for k, var in enumerate(variants):
        case, dy, dhl, kw = _bwd_case(40 + k, **var)
        g = orc.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dy,
                         D=case["D"], z=case["z"], delta_bias=case["delta_bias"],
                         h0=case["h0"], dh_last=dhl, **kw)
        for key, gname in names.items():
            if case[key] is None:
                continue
            x = case[key]
            fd = np.empty_like(x)
            for i in range(x.size):
                old = x.flat[i]
                step = 1e-6 * max(1.0, abs(old))
                x.flat[i] = old + step
                fp = _loss(orc, case, dy, dhl, kw)
                x.flat[i] = old - step
                fm = _loss(orc, case, dy, dhl, kw)
                x.flat[i] = old
                fd.flat[i] = (fp - fm) / (2 * step)
            _close(g[gname], fd, rtol=1e-6, atol=2e-7, what=f"{gname} vs finite differences "
                                                              f"({var or 'zoh, all options'})")


def pin_bwd_homogeneity(orc):
    """Exact identities: the loss is linear in (u, h0) jointly, in B (h0 = 0) and
    in C (no D, dh_last = 0), so it equals sum(input * gradient) over those."""
    for k, euler in enumerate((False, True)):
        case, dy, dhl, kw = _bwd_case(50 + k, euler=euler)
        f = _loss(orc, case, dy, dhl, kw)
        g = orc.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dy,
                         D=case["D"], z=case["z"], delta_bias=case["delta_bias"],
                         h0=case["h0"], dh_last=dhl, **kw)
        _close(np.sum(g["du"] * case["u"]) + np.sum(g["dh0"] * case["h0"]), f, rtol=1e-12,
               atol=1e-12, what="linear in (u, h0)")
        case["h0"] = np.zeros_like(case["h0"])
        case["D"] = None
        f = _loss(orc, case, dy, dhl, kw)
        g = orc.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dy,
                         z=case["z"], delta_bias=case["delta_bias"], h0=case["h0"],
                         dh_last=dhl, **kw)
        _close(np.sum(g["dB"] * case["B"]), f, rtol=1e-12, atol=1e-12, what="linear in B")
        f = _loss(orc, case, dy, np.zeros_like(dhl), kw)
        g = orc.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dy,
                         z=case["z"], delta_bias=case["delta_bias"], h0=case["h0"], **kw)
        _close(np.sum(g["dC"] * case["C"]), f, rtol=1e-12, atol=1e-12, what="linear in C")


def pin_bwd_split_chain(orc):
    """The gradient over [0, L) equals the gradient over [m, L) chained into the
    one over [0, m) through the state at m (its dh0 becomes the first part's
    dh_last)."""
    case, dy, dhl, kw = _bwd_case(60)
    m = 2
    c = {k: case[k] for k in ("A", "D", "delta_bias")}
    full = orc.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dy,
                        D=case["D"], z=case["z"], delta_bias=case["delta_bias"], h0=case["h0"],
                        dh_last=dhl, **kw)
    _, hm = orc.scan_fwd(case["u"][..., :m], case["delta"][..., :m], case["A"],
                         case["B"][..., :m], case["C"][..., :m], D=case["D"],
                         z=case["z"][..., :m], delta_bias=case["delta_bias"], h0=case["h0"],
                         return_last_state=True, **kw)
    part = lambda sl, h0, dh: orc.scan_bwd(  # noqa: E731
        case["u"][..., sl], case["delta"][..., sl], c["A"], case["B"][..., sl],
        case["C"][..., sl], dy[..., sl], D=c["D"], z=case["z"][..., sl],
        delta_bias=c["delta_bias"], h0=h0, dh_last=dh, **kw)
    second = part(slice(m, None), hm, dhl)
    first = part(slice(0, m), case["h0"], second["dh0"])
    for key in ("du", "ddelta", "dz", "dB", "dC"):
        _close(np.concatenate([first[key], second[key]], axis=-1), full[key], rtol=1e-12,
               atol=1e-13, what=f"split {key}")
    for key in ("dA", "dD", "ddelta_bias"):
        _close(first[key] + second[key], full[key], rtol=1e-12, atol=1e-13,
               what=f"split {key}")
    _close(first["dh0"], full["dh0"], rtol=1e-12, atol=1e-13, what="split dh0")


ALL_PINS = [pin_zoh_matches_ode, pin_unrolled_sum, pin_lti_convolution, pin_geometric_series,
            pin_zoh_small_A, pin_linearity, pin_softplus_bias_gate, pin_step_equals_scan,
            pin_split_invariance, pin_rows_match_full, pin_euler_unrolled_sum,
            pin_euler_geometric_and_first_order, pin_conv1d_matches_convolution,
            pin_conv1d_state_and_step, pin_bwd_finite_differences, pin_bwd_homogeneity,
            pin_bwd_split_chain]
