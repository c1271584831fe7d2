"""The oracle against its pins, and the pins against planted mistakes.

Every pin in tests/pins.py is checked against the real oracle.  Then each of a
list of plausible mistakes (a dropped term, a wrong sign, a wrong index, a
swapped operand, a wrong convention) is planted in a temporary copy of the
oracle source on the CPU, compiled, and the pins must reject it.
"""
import os

import numpy as np
import pytest

import oracle
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


# (name, text in ssm_oracle.c, replacement)
MUTANTS = [
    ("euler_instead_of_zoh",
     "double coef = (a == 0.0) ? dt : expm1(dt * a) / a;", "double coef = dt;"),
    ("sign_of_Abar", "double a = A_row[n];\n        double Abar = exp(dt * a);",
     "double a = A_row[n];\n        double Abar = exp(-dt * a);"),
    ("exclusive_output_convention",
     "h[n] = Abar * h[n] + coef * B_col[n * bc_stride] * u;\n"
     "        acc += C_col[n * bc_stride] * h[n];",
     "acc += C_col[n * bc_stride] * h[n];\n"
     "        h[n] = Abar * h[n] + coef * B_col[n * bc_stride] * u;"),
    ("dropped_D_skip", "double y = acc + Dd * u;", "double y = acc;"),
    ("gate_before_D_skip",
     "double y = acc + Dd * u;\n    if (z)\n        y *= oracle_silu(*z);",
     "double y = acc;\n    if (z)\n        y *= oracle_silu(*z);\n    y += Dd * u;"),
    ("bias_after_softplus",
     "double x = delta_raw + bias;\n    double dt = delta_softplus ? oracle_softplus(x) : x;",
     "double x = delta_raw;\n    double dt = (delta_softplus ? oracle_softplus(x) : x) + bias;"),
    ("wrong_BC_stride", "Bcol, Ccol, seqlen, Dd,", "Bcol, Ccol, 1, Dd,"),
    ("swapped_B_C", "Bcol, Ccol, seqlen, Dd,", "Ccol, Bcol, seqlen, Dd,"),
    ("ignored_h0", "h[n] = h0 ? h0[row * dstate + n] : 0.0;", "h[n] = 0.0;"),
    ("wrong_A_row", "A + d * dstate,\n                           Bcol",
     "A + d,\n                           Bcol"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("softplus_branch", "return x + log1p(exp(-x));", "return x + log1p(exp(x));"),
    ("dropped_input_u", "coef * B_col[n * bc_stride] * u;\n        acc",
     "coef * B_col[n * bc_stride];\n        acc"),
    ("expm1_without_divide", "(a == 0.0) ? dt : expm1(dt * a) / a;",
     "(a == 0.0) ? dt : expm1(dt * a);"),
    ("bwd_forward_expm1_without_divide", "(a == 0.0 ? dt : expm1(dt * a) / a);",
     "(a == 0.0 ? dt : expm1(dt * a));"),
    ("bwd_reverse_expm1_without_divide", "                coef = expm1(dt * a) / a;",
     "                coef = expm1(dt * a);"),
    ("decode_stride", "A + d * dstate, B + b * dstate, C + b * dstate, 1,",
     "A + d * dstate, B + b * dstate, C + b * dstate, dstate,"),
    ("euler_coef_times_A", "        if (euler)\n            coef = dt;",
     "        if (euler)\n            coef = dt * a;"),
    ("euler_flag_ignored", "        if (euler)\n            coef = dt;", ""),
    ("euler_flag_dropped_in_decode", "D ? D[d] : 0.0, z ? z + i : NULL, euler);",
     "D ? D[d] : 0.0, z ? z + i : NULL, 0);"),
    ("euler_half_step", "        if (euler)\n            coef = dt;",
     "        if (euler)\n            coef = 0.5 * dt;"),
    ("conv_anticausal", "l - (width - 1) + k);", "l + k);"),
    ("conv_reversed_taps", "acc += weight[d * width + k] * oracle_conv_input(",
     "acc += weight[d * width + (width - 1 - k)] * oracle_conv_input("),
    ("conv_dropped_bias", "                double acc = bias ? bias[d] : 0.0;\n",
     "                double acc = 0.0;\n"),
    ("conv_state_ignored", "    if (p < -(width - 1) || !state_row)", "    if (1)"),
    ("conv_update_no_shift", "                s[k] = s[k + 1];", "                ;"),
    ("conv_silu_before_bias",
     "                out[row * seqlen + l] = apply_silu ? oracle_silu(acc) : acc;",
     "                out[row * seqlen + l] = apply_silu ? oracle_silu(acc - (bias ? bias[d] : 0.0))"
     " + (bias ? bias[d] : 0.0) : acc;"),
    ("bwd_no_state_decay", "            g[n] = Abar * g[n];", "            g[n] = g[n];"),
    ("bwd_h_l_for_h_prev", "const double p = g[n] * h_prev[n];", "const double p = g[n] * h_l[n];"),
    ("bwd_no_softplus_derivative", "ddt * oracle_sigmoid(x) : ddt;", "ddt : ddt;"),
    ("bwd_dcoef_ddt_one", "                dcoef_ddt = Abar;", "                dcoef_ddt = 1.0;"),
    ("bwd_dC_from_h_prev", "+= dy0 * h_l[n];", "+= dy0 * h_prev[n];"),
    ("bwd_gate_derivative_sigmoid_only", "dy[i] * y0 * sg * (1.0 + z[i] * (1.0 - sg));",
     "dy[i] * y0 * sg;"),
    ("bwd_series_coefficient", "q * (1.0 / 3.0 + q", "q * (1.0 / 6.0 + q"),
    ("bwd_dA_without_Abar", "p * dt * Abar + r * dcoef_da", "p * dt + r * dcoef_da"),
    ("bwd_dh_last_ignored", "g[n] = dh_last ? dh_last[row * dstate + n] : 0.0;", "g[n] = 0.0;"),
    ("bwd_dB_without_u", "+= g[n] * coef * u[i];", "+= g[n] * coef;"),
    ("bwd_dD_before_gate", "dD_acc[d] += dy0 * u[i];", "dD_acc[d] += dy[i] * u[i];"),
    ("bwd_bias_grad_dropped", "        dbias_acc[d] += dx;\n", ""),
    ("bwd_euler_dcoef_ddt", "                coef = dt;\n                dcoef_ddt = 1.0;\n"
     "                dcoef_da = 0.0;",
     "                coef = dt;\n                dcoef_ddt = Abar;\n                dcoef_da = 0.0;"),
    ("bwd_zero_A_limit", "        return 0.5 * dt * dt;", "        return 0.0;"),
    ("bwd_gate_grad_before_contraction", "        double y0 = Dd * u[i];", "        double y0 = 0.0;"),
    ("bwd_du_missing_skip", "double du_l = Dd * dy0;", "double du_l = 0.0;"),
]


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(tmp_path, name, find, repl):
    src = open(oracle.SOURCE).read()
    assert src.count(find) == 1, f"mutation site for {name} not unique/present"
    mutant = tmp_path / f"mutant_{name}.c"
    mutant.write_text(src.replace(find, repl))
    lib = oracle.compile_source(str(mutant), str(tmp_path / f"lib_{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except (AssertionError, FloatingPointError, ValueError) as e:  # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, f"no pin rejects the planted mistake '{name}'"


def test_golden_tiny_regression(orc):
    """tests/golden/tiny_scan.txt was written by tests/golden/make_golden.py from
    the oracle; this guards the oracle against silent drift."""
    from tests.golden import make_golden
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_scan.txt")
    stored = np.loadtxt(path)
    fresh = make_golden.tiny_scan_values(orc)
    np.testing.assert_allclose(fresh, stored, rtol=1e-13, atol=1e-15)
