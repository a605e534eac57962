"""The oracle pins must reject a broken oracle (CPU only).

Each case below plants one plausible mistake in a private copy of the oracle
source (a wrong mean divisor, eps in the wrong place, a swapped sign, a wrong
partner index, swapped q/k weights, a double rounding, ...), compiles it with
gcc, and runs the pin suite against it.  The suite must fail for every
mutant; a mutant that survives means the pins have a blind spot.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rn_oracle.c")

MUTANTS = {
    "mean_divisor_n_minus_1": ("double ms = ss / (double)N;", "double ms = ss / (double)(N - 1);"),
    "eps_on_sum": ("double ms = ss / (double)N;\n        double rs = 1.0 / sqrt(ms + deps);",
                   "double ms = ss / (double)N;\n        double rs = 1.0 / sqrt((ss + deps) / (double)N);"),
    "eps_outside_sqrt": ("double rs = 1.0 / sqrt(ms + deps);", "double rs = 1.0 / (sqrt(ms) + deps);"),
    "rstd_eps_outside_sqrt": ("rstd[r] = 1.0 / sqrt(ss / (double)N + (double)eps);",
                              "rstd[r] = 1.0 / (sqrt(ss / (double)N) + (double)eps);"),
    "rstd_eps_on_sum": ("rstd[r] = 1.0 / sqrt(ss / (double)N + (double)eps);",
                        "rstd[r] = 1.0 / sqrt((ss + (double)eps) / (double)N);"),
    "rstd_eps_dropped": ("rstd[r] = 1.0 / sqrt(ss / (double)N + (double)eps);",
                         "rstd[r] = 1.0 / sqrt(ss / (double)N);"),
    "rstd_mean_divisor_n_minus_1": ("rstd[r] = 1.0 / sqrt(ss / (double)N + (double)eps);",
                                    "rstd[r] = 1.0 / sqrt(ss / (double)(N > 1 ? N - 1 : 1) + (double)eps);"),
    "no_weight": ("yr[j] = narrow(v * rs * g, f16);", "yr[j] = narrow(v * rs + 0.0 * g, f16);"),
    "round_via_float": ("double n = nearbyint(v / q);", "double n = nearbyint((double)(float)v / q);"),
    "ties_away": ("double n = nearbyint(v / q);", "double n = round(v / q);"),
    "rope_sign_first": ("o[a] = n[a] * c - n[b] * s;", "o[a] = n[a] * c + n[b] * s;"),
    "rope_sign_second": ("o[b] = n[b] * c + n[a] * s;", "o[b] = n[b] * c - n[a] * s;"),
    "rope_partner_d_half": ("int b = style ? 2 * i + 1 : i + half;", "int b = style ? 2 * i + 1 : i + D / 2;"),
    "rope_cos_sin_swapped": ("double c = (double)cs[i];\n                double s = (double)cs[half + i];",
                             "double s = (double)cs[i];\n                double c = (double)cs[half + i];"),
    "qk_weights_swapped": ("const uint16_t *w = (h < Hq) ? wq : wk;", "const uint16_t *w = (h < Hq) ? wk : wq;"),
    "qk_mean_over_rotary": ("double rs = 1.0 / sqrt(ss / (double)D + deps);",
                            "double rs = 1.0 / sqrt(ss / (double)rotary_dim + deps);"),
    "qk_tail_dropped": ("for (int j = rotary_dim; j < D; ++j) o[j] = n[j];",
                        "for (int j = rotary_dim; j < D; ++j) o[j] = 0.0;"),
    "qk_touches_v": ("for (int h = 0; h < Hq + Hkv; ++h) {", "for (int h = 0; h < Hq + 2 * Hkv; ++h) {"),
    "table_freq_over_d": ("double f = pow(theta, -2.0 * (double)i / (double)rotary_dim);",
                          "double f = pow(theta, -1.0 * (double)i / (double)rotary_dim);"),
    "table_sin_first": ("row[i] = (float)cos(a);\n            row[half + i] = (float)sin(a);",
                        "row[i] = (float)sin(a);\n            row[half + i] = (float)cos(a);"),
    "table_bf16_through_float": ("row[i] = rn_oracle_double_to_bf16(cos(a));\n            row[half + i] = rn_oracle_double_to_bf16(sin(a));",
                                 "row[i] = rn_oracle_double_to_bf16((double)(float)cos(a));\n            row[half + i] = rn_oracle_double_to_bf16((double)(float)sin(a));"),
    "table_bf16_sin_first": ("row[i] = rn_oracle_double_to_bf16(cos(a));\n            row[half + i] = rn_oracle_double_to_bf16(sin(a));",
                             "row[i] = rn_oracle_double_to_bf16(sin(a));\n            row[half + i] = rn_oracle_double_to_bf16(cos(a));"),
    "gptj_partner": ("int b = style ? 2 * i + 1 : i + half;", "int b = style ? 2 * i + 2 - (2 * i + 2) / rotary_dim : i + half;"),
    "gptj_cos_index": ("int a = style ? 2 * i : i;", "int a = style ? 2 * i + 1 : i;"),
    "l2_norm_squared": ("double nrm = sqrt(ss);", "double nrm = ss;"),
    "l2_eps_added": ("double d = nrm > (double)eps ? nrm : (double)eps;", "double d = nrm + (double)eps;"),
    "add_sum_not_rounded": ("h[r * N + j] = narrow(widen(x[r * N + j], f16) + widen(res[r * N + j], f16), f16);",
                            "h[r * N + j] = narrow(0.999 * widen(x[r * N + j], f16) + widen(res[r * N + j], f16), f16);"),
    "add_norm_of_x_only": ("return rn_oracle_rmsnorm_fmt(h, w, eps, M, N, y, f16);", "return rn_oracle_rmsnorm_fmt(x, w, eps, M, N, y, f16);"),
    "layernorm_unbiased": ("double rs = 1.0 / sqrt(m2 / (double)N + (double)eps);",
                           "double rs = 1.0 / sqrt(m2 / (double)(N - 1) + (double)eps);"),
    "layernorm_bias_dropped": ("if (b) v += widen(b[j], f16);", "(void)b;"),
    "f16_round_via_float": ("double r = nearbyint(a / q) * q;                 /* ties to even */",
                            "double r = nearbyint((double)(float)a / q) * q;"),
    "f16_exponent_bias": ("return sign | (uint16_t)((E + 15) << 10) | mant;", "return sign | (uint16_t)((E + 14) << 10) | mant;"),
    "f16_subnormal_quantum": ("if (qexp < -24) qexp = -24;", "if (qexp < -25) qexp = -25;"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = mutant_dir / f"{name}.c"
    so_path = mutant_dir / f"{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so_path), str(c_path), "-lm"], check=True)
    env = dict(os.environ, RN_ORACLE_LIB=str(so_path))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant {name} survived the pins:\n{res.stdout[-2000:]}"
