"""fp64 CPU oracle for the selective scan (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never does; the two share no code.  Inputs come from the seeded
generators in ``selective_state_space_115_b300.workloads``.

The arithmetic lives in ``ssm_oracle.c`` (plain sequential fp64 loops); this
file compiles it with gcc and marshals numpy arrays.  See that file's header
for the passages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ssm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
             "-ffp-contract=off"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library at `out`."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, IEEE semantics, OpenMP over rows)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _f64(x: Optional[np.ndarray]) -> Optional[np.ndarray]:
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x: Optional[np.ndarray]):
    if x is None:
        return None
    return x.ctypes.data_as(_dp)


def _euler(discretization: str) -> int:
    if discretization not in ("zoh", "euler"):
        raise ValueError(f"unknown discretization {discretization!r}")
    return int(discretization == "euler")


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_scan_fwd.restype = ctypes.c_int
        lib.oracle_scan_fwd.argtypes = [_i64, _i64, _i64, _i64, _dp, _dp, _dp, ctypes.c_int,
                                        _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                        ctypes.c_int]
        lib.oracle_scan_rows.restype = ctypes.c_int
        lib.oracle_scan_rows.argtypes = [_i64, _i64, _i64, _i64,
                                         ctypes.POINTER(ctypes.c_int64), _i64,
                                         _dp, _dp, _dp, ctypes.c_int, _dp, _dp, _dp, _dp,
                                         _dp, _dp, _dp, _dp, ctypes.c_int]
        lib.oracle_state_update.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [_i64, _i64, _i64, _dp, _dp, _dp, _dp,
                                            ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _dp,
                                            ctypes.c_int, ctypes.c_int]
        lib.oracle_scan_bwd.restype = ctypes.c_int
        lib.oracle_scan_bwd.argtypes = [_i64, _i64, _i64, _i64, _dp, _dp, _dp, ctypes.c_int,
                                        _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                        _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                        ctypes.c_int]
        lib.oracle_conv1d_fwd.restype = ctypes.c_int
        lib.oracle_conv1d_fwd.argtypes = [_i64, _i64, _i64, _i64, _dp, _dp, _dp, _dp,
                                          ctypes.c_int, _dp, _dp]
        lib.oracle_conv1d_update.restype = ctypes.c_int
        lib.oracle_conv1d_update.argtypes = [_i64, _i64, _i64, _dp, _dp, _dp, _dp, ctypes.c_int,
                                             _dp]
        self.lib = lib
        self.path = path

    def scan_fwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                 delta_softplus=True, h0=None, return_last_state=False, nthreads: int = 1,
                 discretization: str = "zoh"):
        """Selective scan in fp64.  u, delta, z [b,d,l]; B, C [b,n,l]; A [d,n];
        D, delta_bias [d]; h0 [b,d,n].  Returns y [b,d,l] (and h_last [b,d,n]).
        discretization: "zoh" (Bbar = (Abar - 1) / A * B) or "euler" (Bbar = dt * B)."""
        u, delta, A, B, C = (_f64(a) for a in (u, delta, A, B, C))
        D, z, delta_bias, h0 = (_f64(a) for a in (D, z, delta_bias, h0))
        batch, dim, seqlen = u.shape
        dstate = A.shape[1]
        assert delta.shape == u.shape and A.shape == (dim, dstate)
        assert B.shape == (batch, dstate, seqlen) and C.shape == (batch, dstate, seqlen)
        assert z is None or z.shape == u.shape
        y = np.empty_like(u)
        h_last = np.empty((batch, dim, dstate)) if return_last_state else None
        rc = self.lib.oracle_scan_fwd(batch, dim, dstate, seqlen, _ptr(u), _ptr(delta),
                                      _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A),
                                      _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(h0),
                                      _ptr(h_last), _ptr(y), int(nthreads),
                                      _euler(discretization))
        if rc != 0:
            raise RuntimeError("oracle_scan_fwd failed")
        return (y, h_last) if return_last_state else y

    def scan_rows(self, rows: Sequence[int], u_rows, delta_rows, A, B, C, batch: int, dim: int,
                  D=None, z_rows=None, delta_bias=None, delta_softplus=True, h0=None,
                  return_last_state=False, discretization: str = "zoh"):
        """Scan only the listed rows (row = b*dim + d).  u_rows, delta_rows, z_rows
        are the [nrows, L] slices of those rows; B, C are the full [b,n,l]."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        u_rows, delta_rows, A, B, C = (_f64(a) for a in (u_rows, delta_rows, A, B, C))
        D, z_rows, delta_bias, h0 = (_f64(a) for a in (D, z_rows, delta_bias, h0))
        nrows, seqlen = u_rows.shape
        dstate = A.shape[1]
        y = np.empty((nrows, seqlen))
        h_last = np.empty((nrows, dstate)) if return_last_state else None
        rc = self.lib.oracle_scan_rows(batch, dim, dstate, seqlen,
                                       rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), nrows,
                                       _ptr(u_rows), _ptr(delta_rows), _ptr(delta_bias),
                                       int(bool(delta_softplus)), _ptr(A), _ptr(B), _ptr(C),
                                       _ptr(D), _ptr(z_rows), _ptr(h0), _ptr(h_last), _ptr(y),
                                       _euler(discretization))
        if rc != 0:
            raise RuntimeError("oracle_scan_rows failed")
        return (y, h_last) if return_last_state else y

    def state_update(self, h, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                     delta_softplus=True, discretization: str = "zoh", nthreads: int = 1):
        """One decode step in fp64.  h [b,d,n] (copied, not modified); u, delta, z [b,d];
        B, C [b,n].  Returns (y [b,d], h_new [b,d,n])."""
        h = np.array(h, dtype=np.float64, copy=True, order="C")
        u, delta, A, B, C = (_f64(a) for a in (u, delta, A, B, C))
        D, z, delta_bias = (_f64(a) for a in (D, z, delta_bias))
        batch, dim = u.shape
        dstate = A.shape[1]
        assert h.shape == (batch, dim, dstate) and B.shape == (batch, dstate)
        y = np.empty_like(u)
        rc = self.lib.oracle_state_update(batch, dim, dstate, _ptr(h), _ptr(u), _ptr(delta),
                                          _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A),
                                          _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(y),
                                          _euler(discretization), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_state_update failed")
        return y, h


    def scan_bwd(self, u, delta, A, B, C, dy, D=None, z=None, delta_bias=None,
                 delta_softplus=True, h0=None, dh_last=None, nthreads: int = 1,
                 discretization: str = "zoh"):
        """Gradient of the scan in fp64 for the loss sum(dy * y) (+ sum(dh_last * h_last)).
        Returns a dict with du, ddelta [b,d,l], dA [d,n], dB, dC [b,n,l], dD (when D),
        dz (when z), ddelta_bias (when delta_bias), dh0 [b,d,n]."""
        u, delta, A, B, C, dy = (_f64(a) for a in (u, delta, A, B, C, dy))
        D, z, delta_bias, h0, dh_last = (_f64(a) for a in (D, z, delta_bias, h0, dh_last))
        batch, dim, seqlen = u.shape
        dstate = A.shape[1]
        assert delta.shape == u.shape and dy.shape == u.shape and A.shape == (dim, dstate)
        assert B.shape == (batch, dstate, seqlen) and C.shape == (batch, dstate, seqlen)
        assert z is None or z.shape == u.shape
        out = {"du": np.empty_like(u), "ddelta": np.empty_like(u),
               "dA": np.empty((dim, dstate)), "dB": np.empty_like(B), "dC": np.empty_like(C),
               "dD": np.empty(dim) if D is not None else None,
               "dz": np.empty_like(u) if z is not None else None,
               "ddelta_bias": np.empty(dim) if delta_bias is not None else None,
               "dh0": np.empty((batch, dim, dstate))}
        rc = self.lib.oracle_scan_bwd(batch, dim, dstate, seqlen, _ptr(u), _ptr(delta),
                                      _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A),
                                      _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(h0), _ptr(dy),
                                      _ptr(dh_last), _ptr(out["du"]), _ptr(out["ddelta"]),
                                      _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
                                      _ptr(out["dD"]), _ptr(out["dz"]), _ptr(out["ddelta_bias"]),
                                      _ptr(out["dh0"]), int(nthreads), _euler(discretization))
        if rc != 0:
            raise RuntimeError("oracle_scan_bwd failed")
        return out

    def conv1d_fwd(self, x, weight, bias=None, state_in=None, apply_silu=True,
                   return_state=False):
        """Causal depthwise convolution over time in fp64.  x [b,d,l]; weight [d,W];
        bias [d]; state_in [b,d,W-1] (inputs before position 0).  Returns out [b,d,l]
        (and the last W-1 inputs [b,d,W-1])."""
        x, weight, bias, state_in = (_f64(a) for a in (x, weight, bias, state_in))
        batch, dim, seqlen = x.shape
        width = weight.shape[1]
        assert weight.shape == (dim, width)
        assert state_in is None or state_in.shape == (batch, dim, width - 1)
        out = np.empty_like(x)
        state_out = np.empty((batch, dim, width - 1)) if return_state else None
        rc = self.lib.oracle_conv1d_fwd(batch, dim, seqlen, width, _ptr(x), _ptr(weight),
                                        _ptr(bias), _ptr(state_in), int(bool(apply_silu)),
                                        _ptr(out), _ptr(state_out))
        if rc != 0:
            raise RuntimeError("oracle_conv1d_fwd failed")
        return (out, state_out) if return_state else out

    def conv1d_update(self, state, x, weight, bias=None, apply_silu=True):
        """One decode position: state [b,d,W-1] (copied, not modified), x [b,d].
        Returns (out [b,d], new state [b,d,W-1])."""
        state = np.array(state, dtype=np.float64, copy=True, order="C")
        x, weight, bias = (_f64(a) for a in (x, weight, bias))
        batch, dim = x.shape
        width = weight.shape[1]
        assert state.shape == (batch, dim, width - 1)
        out = np.empty_like(x)
        rc = self.lib.oracle_conv1d_update(batch, dim, width, _ptr(state), _ptr(x), _ptr(weight),
                                           _ptr(bias), int(bool(apply_silu)), _ptr(out))
        if rc != 0:
            raise RuntimeError("oracle_conv1d_update failed")
        return out, state


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def scan_fwd(*args, **kwargs):
    return default().scan_fwd(*args, **kwargs)


def scan_rows(*args, **kwargs):
    return default().scan_rows(*args, **kwargs)


def state_update(*args, **kwargs):
    return default().state_update(*args, **kwargs)


def scan_bwd(*args, **kwargs):
    return default().scan_bwd(*args, **kwargs)


def conv1d_fwd(*args, **kwargs):
    return default().conv1d_fwd(*args, **kwargs)


def conv1d_update(*args, **kwargs):
    return default().conv1d_update(*args, **kwargs)
