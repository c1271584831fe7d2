"""Writes the stored expected values under tests/golden/ by calling only the oracle.

The pages print no worked numeric example, so the only stored values are
oracle outputs kept as a regression guard.  Run from the repository root:

    python -m tests.golden.make_golden
"""
from __future__ import annotations

import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def tiny_scan_values(orc) -> np.ndarray:
    """y of the tiny fp32 workload (B1 D4 N4 L64, seed 0), flattened, plus h_last."""
    from selective_state_space_115_b300 import workloads as W
    cfg = W.SCAN_CONFIGS["tiny"]
    x = W.make_scan_inputs(cfg, seed=0)
    y, hl = orc.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                         delta_bias=x["delta_bias"], delta_softplus=True,
                         return_last_state=True)
    return np.concatenate([y.ravel(), hl.ravel()])


def main():
    import oracle
    vals = tiny_scan_values(oracle.default())
    path = os.path.join(HERE, "tiny_scan.txt")
    header = ("oracle output of the tiny workload (batch 1, dim 4, dstate 4, seqlen 64, fp32,\n"
              "seed 0, bias 0, D = 1, no gate): 256 values of y in [b,d,l] order, then the\n"
              "16 values of h_last in [b,d,n] order.  Written by tests/golden/make_golden.py.")
    np.savetxt(path, vals, fmt="%.17e", header=header)
    print(f"wrote {path} ({vals.size} values)")


if __name__ == "__main__":
    main()
