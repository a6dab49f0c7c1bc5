"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of conv1d_oracle.c (a wrong tap offset,
reversed state order, a sign flip in the SiLU derivative, transposed taps in
the input gradient, a transposed full-channel weight, ...), compiles it, and
runs the pin suites (depthwise and full-channel) against it in a subprocess:
the suites have to fail.  Every planted mistake keeps all memory
accesses in bounds.
"""

import os
import subprocess
import sys
import tempfile

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "conv1d_oracle.c")

MUTANTS = {
    "tap_offset": ("p += w[k] * xe(x, init, W - 1, t - (W - 1) + k);",
                   "p += w[k] * xe(x, init, W - 1, t - (W - 1) + (k + 1) % W);"),
    "init_order_reversed": ("return init ? init[j + S] : 0.0;",
                            "return init ? init[S - 1 - (j + S)] : 0.0;"),
    "silu_grad_sign": ("return s * (1.0 + p * (1.0 - s));", "return s * (1.0 - p * (1.0 - s));"),
    "silu_forward": ("return act ? p * sigmoid(p) : p;", "return act ? sigmoid(p) : p;"),
    "dx_taps_transposed": ("acc += wd[k] * gp[t];", "acc += wd[W - 1 - k] * gp[t];"),
    "dfinal_reversed": ("acc += gfs[j - (len - S)];", "acc += gfs[len - 1 - j];"),
    "final_state_reversed": ("fs[i] = xe(xs, is, S, len - S + i);",
                             "fs[S - 1 - i] = xe(xs, is, S, len - S + i);"),
    "dw_taps_reversed": ("double term = gp[t] * xe(xs, is, S, t - (W - 1) + k);",
                         "double term = gp[t] * xe(xs, is, S, t - k);"),
    "db_without_act_grad": ("sdb += gp[t];", "sdb += gs[t];"),
    "empty_sequence_accepted": ("if (cu[n + 1] <= cu[n])", "if (cu[n + 1] < cu[n])"),
    "update_shift": ("s[i] = ext[i + 1];", "s[i] = ext[i];"),
    "update_drops_bias": ("double p = bias ? bias[d] : 0.0;\n            for (int k = 0; k < W; ++k)\n                p += wd[k] * ext[k];",
                          "double p = 0.0;\n            for (int k = 0; k < W; ++k)\n                p += wd[k] * ext[k];"),
    "bf16_truncates": ("double r = rint(ldexp(a, -qexp));", "double r = floor(ldexp(a, -qexp));"),
    "bias_dropped": ("double p = b;\n    for (int k = 0; k < W; ++k)\n        if (same_seq",
                     "double p = 0.0 * b;\n    for (int k = 0; k < W; ++k)\n        if (same_seq"),
    "dw_abs_shifted_tap": ("sdw_abs[k] += fabs(term);", "sdw_abs[(k + 1) % W] += fabs(term);"),
    "dw_abs_doubled": ("sdw_abs[k] += fabs(term);", "sdw_abs[k] += 2.0 * fabs(term);"),
    "db_abs_without_act_grad": ("sdb_abs += fabs(gp[t]);", "sdb_abs += fabs(gs[t]);"),
    "seq_idx_ordered_not_equal": ("return !ids || j < 0 || ids[j] == ids[t];",
                                  "return !ids || j < 0 || ids[j] <= ids[t];"),
    "seq_idx_dx_unmasked": ("if (t >= 0 && t < len && same_seq(ids, j, t))", "if (t >= 0 && t < len)"),
    "seq_idx_dw_unmasked": ("if (!same_seq(ids, t - (W - 1) + k, t))\n                        term = 0.0;",
                            "if (0)\n                        term = 0.0;"),
    "fullconv_padding_sign": ("int64_t pos = t + (int64_t)k * dil - P;", "int64_t pos = t - (int64_t)k * dil;"),
    "fullconv_no_dilation": ("int64_t pos = t + (int64_t)k * dil - P;", "int64_t pos = t + (int64_t)k - P;"),
    "fullconv_weight_transposed": ("double term = w[(oc * Cin + ic) * K + k] * x[(b * Cin + ic) * T + pos];",
                                   "double term = w[(ic * Cout + oc) * K + k] * x[(b * Cin + ic) * T + pos];"),
    "fullconv_bias_dropped": ("double s = bias ? bias[oc] : 0.0;", "double s = 0.0;"),
    "fullconv_abs_without_bias": ("double a = bias ? fabs(bias[oc]) : 0.0;", "double a = 0.0;"),
    "width_state_offset": ("const double *is = init ? init + ((int64_t)n * D + d) * S : NULL;\n            const int32_t *ids",
                           "const double *is = init ? init + ((int64_t)n * D + d) * 3 : NULL;\n            const int32_t *ids"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as d:
        msrc = os.path.join(d, "mutant.c")
        lib = os.path.join(d, "libmutant.so")
        with open(msrc, "w") as f:
            f.write(src.replace(old, new))
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                               msrc, "-o", lib, "-lm"])
        env = dict(os.environ, CCC_ORACLE_LIB=lib)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                            os.path.join(ROOT, "tests", "test_oracle_pins_fullconv.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
