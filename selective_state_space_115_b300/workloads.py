"""Seeded synthetic workloads for the selective scan and the decode state update.

This module only draws random inputs.  It holds none of the scan's arithmetic,
so both the CUDA path and the fp64 oracle can take their inputs from it.

Shapes follow the selection section of the velog review of "Mamba: Linear-Time
Sequence Modeling with Selective State Spaces" (section 3.2: delta is (B, L, D),
A is (D, N), B and C are (B, L, N)), stored here channel-major with l fastest:

    u, delta, z : [batch, dim, seqlen]      (io dtype)
    B, C        : [batch, dstate, seqlen]   (io dtype)
    A           : [dim, dstate]             float32, A[d, n] = -(n + 1)
    D, bias     : [dim]                     float32
    h           : [batch, dim, dstate]      float32

A[d, n] = -(n + 1) is the "S4D real" initialisation of the Mamba_Model_Report.md
MambaBlock (section 3, A_log = log(arange(1, N+1))).  The per-channel step bias
is the inverse softplus of a log-uniform dt, as that report's dt_proj bias
initialisation describes (section 3, "inv_dt").

bf16 values are carried as uint16 bit patterns (numpy has no bfloat16); they are
produced from float32 draws with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    io: str                 # "f32" or "bf16"
    gate: bool              # silu(z) gate on
    dt_bias: bool           # bias = inverse softplus of log-uniform dt (else 0)
    d_skip: str             # "normal" (D ~ N(0,1)) or "ones"
    description: str

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen

    @property
    def updates(self) -> int:
        return self.elements * self.dstate


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    io: str
    gate: bool
    h_std: float
    description: str


SCAN_CONFIGS: Dict[str, ScanConfig] = {
    "tiny": ScanConfig("tiny", 1, 4, 4, 64, F32, gate=False, dt_bias=False, d_skip="ones",
                       description="tiny fp32 scan B1 D4 N4 L64, bias 0, D=1, no gate"),
    "130m": ScanConfig("130m", 2, 1536, 16, 2048, F32, gate=True, dt_bias=True, d_skip="normal",
                       description="fp32 scan, Mamba-130M-like layer B2 D1536 N16 L2048, gate"),
    "2p8b": ScanConfig("2p8b", 8, 5120, 16, 2048, BF16, gate=True, dt_bias=True, d_skip="normal",
                       description="bf16 I/O fp32 state, Mamba-2.8B-like layer B8 D5120 N16 L2048, gate"),
    "long": ScanConfig("long", 1, 1536, 16, 131072, BF16, gate=False, dt_bias=True, d_skip="normal",
                       description="long bf16 scan B1 D1536 N16 L131072, no gate"),
}

DECODE_CONFIGS: Dict[str, DecodeConfig] = {
    "decode": DecodeConfig("decode", 256, 5120, 16, 1024, BF16, gate=True, h_std=0.1,
                           description="decode state update B256 D5120 N16, 1024 steps"),
}


# ----------------------------------------------------------------------------
# bf16 bit helpers (input encoding only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_f64(x: np.ndarray, io: str) -> np.ndarray:
    """Exact float64 value of an io-typed array (float32 or bf16 bits)."""
    if io == BF16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def encode(x32: np.ndarray, io: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if io == BF16 else np.ascontiguousarray(x32, dtype=np.float32)


# ----------------------------------------------------------------------------
# parameter recipes
# ----------------------------------------------------------------------------
def s4d_real_A(dim: int, dstate: int) -> np.ndarray:
    """A[d, n] = -(n + 1) (S4D-real initialisation, A = -exp(log(n+1)))."""
    return -np.tile(np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))


def dt_bias_from(rng: np.random.Generator, dim: int,
                 dt_min: float = 1e-3, dt_max: float = 1e-1) -> np.ndarray:
    """Per-channel bias = inverse softplus of dt, dt log-uniform in [dt_min, dt_max]."""
    log_dt = rng.uniform(math.log(dt_min), math.log(dt_max), size=dim)
    dt = np.exp(log_dt)
    return np.log(np.expm1(dt)).astype(np.float32)


def make_scan_inputs(cfg: ScanConfig, seed: int = 0, with_h0: bool = False,
                     batch: Optional[int] = None, dim: Optional[int] = None,
                     seqlen: Optional[int] = None, dstate: Optional[int] = None,
                     gate: Optional[bool] = None) -> Dict[str, np.ndarray]:
    """Draw one scan problem.  Draw order: u, delta_raw, B, C, z, D, dt, h0.

    Size overrides let tests build odd shapes with a config's distributions.
    """
    b = cfg.batch if batch is None else batch
    d = cfg.dim if dim is None else dim
    n = cfg.dstate if dstate is None else dstate
    L = cfg.seqlen if seqlen is None else seqlen
    g = cfg.gate if gate is None else gate
    rng = np.random.default_rng(seed)
    f32 = np.float32
    u = rng.standard_normal((b, d, L), dtype=f32)
    delta = rng.standard_normal((b, d, L), dtype=f32)
    Bm = rng.standard_normal((b, n, L), dtype=f32)
    Cm = rng.standard_normal((b, n, L), dtype=f32)
    z = rng.standard_normal((b, d, L), dtype=f32) if g else None
    if cfg.d_skip == "normal":
        Dv = rng.standard_normal(d, dtype=f32)
    else:
        Dv = np.ones(d, dtype=f32)
    bias = dt_bias_from(rng, d) if cfg.dt_bias else np.zeros(d, dtype=f32)
    h0 = (rng.standard_normal((b, d, n), dtype=f32) * f32(0.1)).astype(f32) if with_h0 else None
    out = {
        "u": encode(u, cfg.io),
        "delta": encode(delta, cfg.io),
        "B": encode(Bm, cfg.io),
        "C": encode(Cm, cfg.io),
        "z": None if z is None else encode(z, cfg.io),
        "A": s4d_real_A(d, n),
        "D": Dv,
        "delta_bias": bias,
        "h0": h0,
    }
    return out


def make_decode_static(cfg: DecodeConfig, seed: int = 0, batch: Optional[int] = None,
                       dim: Optional[int] = None) -> Dict[str, np.ndarray]:
    """A, D, bias and the initial state h (std cfg.h_std) for the decode loop."""
    b = cfg.batch if batch is None else batch
    d = cfg.dim if dim is None else dim
    rng = np.random.default_rng([seed, 0])
    h = (rng.standard_normal((b, d, cfg.dstate), dtype=np.float32) * np.float32(cfg.h_std))
    Dv = rng.standard_normal(d, dtype=np.float32)
    bias = dt_bias_from(rng, d)
    return {"A": s4d_real_A(d, cfg.dstate), "D": Dv, "delta_bias": bias,
            "h": h.astype(np.float32)}


def make_decode_step(cfg: DecodeConfig, step: int, seed: int = 0, batch: Optional[int] = None,
                     dim: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Per-token inputs of decode step `step`: u, delta_raw, z [b, d]; B, C [b, n]."""
    b = cfg.batch if batch is None else batch
    d = cfg.dim if dim is None else dim
    rng = np.random.default_rng([seed, step + 1])
    f32 = np.float32
    u = rng.standard_normal((b, d), dtype=f32)
    delta = rng.standard_normal((b, d), dtype=f32)
    Bm = rng.standard_normal((b, cfg.dstate), dtype=f32)
    Cm = rng.standard_normal((b, cfg.dstate), dtype=f32)
    z = rng.standard_normal((b, d), dtype=f32) if cfg.gate else None
    return {"u": encode(u, cfg.io), "delta": encode(delta, cfg.io), "B": encode(Bm, cfg.io),
            "C": encode(Cm, cfg.io), "z": None if z is None else encode(z, cfg.io)}


def make_scan_grads(cfg: ScanConfig, seed: int = 0, batch: Optional[int] = None,
                    dim: Optional[int] = None, seqlen: Optional[int] = None,
                    dstate: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Upstream gradients for the scan's backward: dy [b, d, L] ~ N(0, 1) in the io
    dtype and dh_last [b, d, n] ~ N(0, 1) float32, from their own stream
    (default_rng([seed, 7])) so they do not disturb the forward inputs' draws."""
    b = cfg.batch if batch is None else batch
    d = cfg.dim if dim is None else dim
    n = cfg.dstate if dstate is None else dstate
    L = cfg.seqlen if seqlen is None else seqlen
    rng = np.random.default_rng([seed, 7])
    dy = rng.standard_normal((b, d, L), dtype=np.float32)
    dh_last = rng.standard_normal((b, d, n), dtype=np.float32)
    return {"dy": encode(dy, cfg.io), "dh_last": dh_last}
