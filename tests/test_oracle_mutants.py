"""The pins have teeth: plausible mistakes planted in a copy of the oracle (on the
CPU, in a temporary directory) must each fail at least one pin.

Each mutant rewrites one spot of oracle.c -- a dropped term, a wrong sign, a
wrong index or divisor, a swapped operand -- compiles the copy with the same
flags and runs every pin against it.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (id, text in oracle.c, replacement, which occurrence (0-based))
MUTANTS = [
    ("ln_var_unbiased", "const double var = orc_sum_get(&q) / (double)N;",
     "const double var = orc_sum_get(&q) / (double)(N - 1);", 0),
    ("ln_mean_wrong_divisor", "const double mean = orc_sum_get(&s) / (double)N;",
     "const double mean = orc_sum_get(&s) / (double)(N + 1);", 0),
    ("ln_eps_outside_sqrt", "const double rstd = 1.0 / sqrt(var + (double)eps);",
     "const double rstd = 1.0 / (sqrt(var) + (double)eps);", 0),
    ("ln_drop_beta", "const double out = (orc_get(dt, x, base + i) - mean) * rstd * g + b;",
     "const double out = (orc_get(dt, x, base + i) - mean) * rstd * g;", 0),
    ("ln_sign", "const double out = (orc_get(dt, x, base + i) - mean) * rstd * g + b;",
     "const double out = (mean - orc_get(dt, x, base + i)) * rstd * g + b;", 0),
    ("ln_gamma_reversed", "const double g = gamma ? orc_get(dt, gamma, i) : 1.0;",
     "const double g = gamma ? orc_get(dt, gamma, N - 1 - i) : 1.0;", 0),
    ("rms_sum_not_squared", "orc_sum_add(&s, v * v);", "orc_sum_add(&s, v);", 0),
    ("rms_eps_outside_sqrt", "const double rstd = 1.0 / sqrt(ms + (double)eps);",
     "const double rstd = 1.0 / (sqrt(ms) + (double)eps);", 0),
    ("rms_drop_weight", "const double out = orc_get(dt, x, base + i) * rstd * wi;",
     "const double out = orc_get(dt, x, base + i) * rstd;", 0),
    ("add_rms_wrong_sign", "const float sum = a + b;", "const float sum = a - b;", 0),
    ("add_rms_stats_unrounded", "const double v = orc_get(dt, residual_out, base + i);",
     "const double v = (double)sum;", 0),
    ("add_rms_normalizes_x",
     "const double out = orc_get(dt, residual_out, base + i) * rstd * wi;",
     "const double out = orc_get(dt, x, base + i) * rstd * wi;", 0),
    ("add_rms_eps_dropped", "const double rstd = 1.0 / sqrt(ms + (double)eps);",
     "const double rstd = 1.0 / sqrt(ms);", 1),
    ("bn_transposed_index", "orc_sum_add(&s, orc_get(dt, x, (n * C + c) * HW + k));",
     "orc_sum_add(&s, orc_get(dt, x, (c * batch + n) * HW + k));", 0),
    ("bn_var_unbiased", "const double var = orc_sum_get(&q) / (double)cnt;",
     "const double var = orc_sum_get(&q) / (double)(cnt - 1);", 0),
    ("bn_gamma_index", "const double g = gamma ? orc_get(dt, gamma, c) : 1.0;",
     "const double g = gamma ? orc_get(dt, gamma, 0) : 1.0;", 0),
    ("bn_running_var_biased", "+ m * var * (double)cnt / (double)(cnt - 1);", "+ m * var;", 0),
    ("bn_momentum_swapped",
     "running_mean[c] = (1.0 - m) * running_mean[c] + m * mean;",
     "running_mean[c] = m * running_mean[c] + (1.0 - m) * mean;", 0),
    ("bn_infer_eps_dropped",
     "const double rstd = 1.0 / sqrt((double)running_var[c] + (double)eps);",
     "const double rstd = 1.0 / sqrt((double)running_var[c]);", 0),
    ("bn_infer_drop_beta", "const double out = (orc_get(dt, x, i) - mean) * rstd * g + b;",
     "const double out = (orc_get(dt, x, i) - mean) * rstd * g;", 1),
    ("bn_infer_channel_index", "const double mean = (double)running_mean[c];",
     "const double mean = (double)running_mean[0];", 0),
    ("bn_bwd_drop_gamma",
     "g * rstd[c] * (orc_get(dt, dy, i) - db / cnt - xhat * dg / cnt);",
     "rstd[c] * (orc_get(dt, dy, i) - db / cnt - xhat * dg / cnt);", 0),
    ("bn_bwd_xhat_term_sign", "- xhat * dg / cnt);", "+ xhat * dg / cnt);", 0),
    ("bn_bwd_dbeta_not_averaged", "(orc_get(dt, dy, i) - db / cnt", "(orc_get(dt, dy, i) - db", 0),
    ("bn_bwd_dgamma_uses_x", "orc_sum_add(&s2, g_out * xhat);",
     "orc_sum_add(&s2, g_out * orc_get(dt, x, i));", 0),
    ("bn_bwd_xhat_unscaled", "const double xhat = (orc_get(dt, x, i) - mean[c]) * rstd[c];",
     "const double xhat = (orc_get(dt, x, i) - mean[c]);", 0),
    ("bn_bwd_biased_count", "const double cnt = (double)(batch * HW);",
     "const double cnt = (double)(batch * HW - 1);", 0),
    ("softmax_no_max", "double m = -INFINITY;", "double m = 0.0; if (0)", 0),
    ("softmax_sum_skips_last", "orc_sum_add(&s, exp(orc_get(dt, x, r * N + j) - m));",
     "if (j + 1 < N) orc_sum_add(&s, exp(orc_get(dt, x, r * N + j) - m));", 0),
    ("softmax_eps_in_denominator", "const double out = exp(orc_get(dt, x, r * N + j) - m) / d;",
     "const double out = exp(orc_get(dt, x, r * N + j) - m) / (d + 1e-12);", 0),
    ("softmax_uses_min", "if (v > m)", "if (v < m || m == -INFINITY)", 0),
    ("rn_ties_away", "if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) == 1.0))",
     "if (r >= 0.5)", 0),
    ("rn_flush_subnormals", "        E = emin;                  /* subnormal range",
     "        return (uint16_t)sign;  /* subnormal range", 0),
    ("rn_no_overflow", "if (biased >= all_ones)", "if (biased > all_ones)", 0),
    ("f16_decode_exponent", "mag = ldexp((double)(f + 1024), e - 25);",
     "mag = ldexp((double)(f + 1024), e - 24);", 0),
    ("bf16_decode_subnormal", "mag = ldexp((double)f, -133);", "mag = ldexp((double)f, -126);", 0),
]


def _replace_nth(text, old, new, k):
    start = -1
    for _ in range(k + 1):
        start = text.find(old, start + 1)
        if start < 0:
            return None
    return text[:start] + new + text[start + len(old):]


@pytest.mark.parametrize("mid,old,new,k", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, mid, old, new, k):
    src = open(SRC).read()
    mutated = _replace_nth(src, old, new, k)
    assert mutated is not None, f"mutation site for {mid} not found in oracle.c"
    msrc = tmp_path / f"oracle_{mid}.c"
    msrc.write_text(mutated)
    so = oracle.compile_oracle(str(msrc), str(tmp_path / f"liboracle_{mid}.so"))
    orc = oracle.Oracle(oracle.load_library(so))
    failed = []
    for pin in oracle_pins.PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, OverflowError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mid} passed every pin"
