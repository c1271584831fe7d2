"""Randomised properties of the oracle (no GPU): the fixed pins of tests/pins.py at
random shapes, split points and options, drawn by hypothesis with a fixed seed.

  * the scan is split-invariant: [0, L) equals [0, m) then [m, L) from its state;
  * the gradient chains through a split: [m, L)'s dh0 is [0, m)'s dh_last;
  * the loss is linear in (u, h0) jointly: sum(u du) + sum(h0 dh0) equals it;
  * the conv1d carried window chains: [0, L) equals [0, m) then [m, L) with the
    first part's last W - 1 inputs as the state.
"""
import numpy as np
from hypothesis import given, settings, strategies as st

import oracle

SETTINGS = settings(max_examples=25, deadline=None, derandomize=True)


def _case(seed, b, d, n, L, gate, euler):
    rng = np.random.default_rng(seed)
    x = {
        "u": rng.standard_normal((b, d, L)),
        "delta": rng.standard_normal((b, d, L)),
        "A": -rng.uniform(0.1, 4.0, size=(d, n)),
        "B": rng.standard_normal((b, n, L)),
        "C": rng.standard_normal((b, n, L)),
        "D": rng.standard_normal(d),
        "z": rng.standard_normal((b, d, L)) if gate else None,
        "delta_bias": rng.uniform(-3.0, 0.5, size=d),
        "h0": rng.standard_normal((b, d, n)) * 0.3,
    }
    return x, rng, dict(discretization="euler" if euler else "zoh")


def _sl(x, lo, hi):
    return {k: (v[..., lo:hi] if k in ("u", "delta", "z", "B", "C") and v is not None else v)
            for k, v in x.items()}


shapes = st.tuples(st.integers(0, 10_000), st.integers(1, 2), st.integers(1, 4),
                   st.sampled_from([1, 2, 4, 8]), st.integers(2, 24), st.booleans(),
                   st.booleans())


@SETTINGS
@given(shapes, st.data())
def test_forward_split_invariance(shape, data):
    seed, b, d, n, L, gate, euler = shape
    m = data.draw(st.integers(1, L - 1))
    x, _, kw = _case(seed, b, d, n, L, gate, euler)
    full, hl = oracle.scan_fwd(**x, return_last_state=True, **kw)
    a, ha = oracle.scan_fwd(**_sl(x, 0, m), return_last_state=True, **kw)
    second = dict(_sl(x, m, L), h0=ha)
    c, hc = oracle.scan_fwd(**second, return_last_state=True, **kw)
    np.testing.assert_allclose(np.concatenate([a, c], axis=-1), full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hc, hl, rtol=1e-12, atol=1e-12)


@SETTINGS
@given(shapes, st.data())
def test_gradient_chains_through_a_split(shape, data):
    seed, b, d, n, L, gate, euler = shape
    m = data.draw(st.integers(1, L - 1))
    x, rng, kw = _case(seed, b, d, n, L, gate, euler)
    dy = rng.standard_normal((b, d, L))
    dhl = rng.standard_normal((b, d, n))
    full = oracle.scan_bwd(**x, dy=dy, dh_last=dhl, **kw)
    _, hm = oracle.scan_fwd(**_sl(x, 0, m), return_last_state=True, **kw)
    second = oracle.scan_bwd(**dict(_sl(x, m, L), h0=hm), dy=dy[..., m:], dh_last=dhl, **kw)
    first = oracle.scan_bwd(**_sl(x, 0, m), dy=dy[..., :m], dh_last=second["dh0"], **kw)
    for k in ("du", "ddelta", "dB", "dC") + (("dz",) if gate else ()):
        np.testing.assert_allclose(np.concatenate([first[k], second[k]], axis=-1), full[k],
                                   rtol=1e-10, atol=1e-11)
    for k in ("dA", "dD", "ddelta_bias"):
        np.testing.assert_allclose(first[k] + second[k], full[k], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(first["dh0"], full["dh0"], rtol=1e-10, atol=1e-11)


@SETTINGS
@given(shapes)
def test_loss_is_linear_in_u_and_h0(shape):
    seed, b, d, n, L, gate, euler = shape
    x, rng, kw = _case(seed, b, d, n, L, gate, euler)
    dy = rng.standard_normal((b, d, L))
    dhl = rng.standard_normal((b, d, n))
    y, hl = oracle.scan_fwd(**x, return_last_state=True, **kw)
    loss = float(np.sum(dy * y) + np.sum(dhl * hl))
    g = oracle.scan_bwd(**x, dy=dy, dh_last=dhl, **kw)
    lin = float(np.sum(g["du"] * x["u"]) + np.sum(g["dh0"] * x["h0"]))
    assert abs(lin - loss) <= 1e-10 * max(1.0, abs(loss))


@SETTINGS
@given(st.integers(0, 10_000), st.integers(1, 3), st.integers(1, 8), st.integers(2, 30),
       st.booleans(), st.data())
def test_conv1d_state_chains(seed, d, width, L, silu, data):
    m = data.draw(st.integers(1, L - 1))
    rng = np.random.default_rng(seed)
    xv = rng.standard_normal((2, d, L))
    w = rng.standard_normal((d, width))
    bias = rng.standard_normal(d)
    s0 = rng.standard_normal((2, d, width - 1))
    full = oracle.conv1d_fwd(xv, w, bias, state_in=s0, apply_silu=silu)
    a, sa = oracle.conv1d_fwd(xv[..., :m], w, bias, state_in=s0, apply_silu=silu,
                              return_state=True)
    c = oracle.conv1d_fwd(xv[..., m:], w, bias, state_in=sa, apply_silu=silu)
    np.testing.assert_allclose(np.concatenate([a, c], axis=-1), full, rtol=1e-13, atol=1e-13)
