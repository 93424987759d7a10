"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutant is the committed oracle source with one plausible mistake planted by
text substitution (a dropped term, a wrong sign or index, a transposed operand,
a wrong variance kind ...).  It is compiled into a temporary library and every
pin is run against it; at least one pin must fail.  Nothing here touches the
committed oracle or the CUDA path.
"""
import os

import pytest

import oracle
from tests.oracle_pins import ALL_PINS

# (name, text to find, replacement, which occurrence (0-based))
MUTANTS = [
    ("exp_without_max_shift", "s += exp((double)v[k * stride] - m);",
     "s += exp((double)v[k * stride]);", 0),
    ("transposed_strided_index", "lse_strided_float(x + o * R * inner + i, R, inner)",
     "lse_strided_float(x + o * R * inner + i * R, R, 1)", 0),
    ("max_as_min", "else if (a > m) m = a;", "else if (a < m) m = a;", 1),
    ("all_ninf_not_special", "if (m == -INFINITY) return -INFINITY;", "", 1),
    ("nan_not_first", "if (has_nan) return NAN;", "", 1),
    ("row_off_by_one", "lse_strided_float(row, cols, 1)", "lse_strided_float(row, cols - 1, 1)", 0),
    ("log_softmax_sign", "(double)row[j] - lse", "(double)row[j] + lse", 0),
    ("lse_drops_log", "return m + log(s);", "return m + s;", 1),
    ("unbiased_variance", "sq / (double)count", "sq / (double)(count - 1)", 0),
    ("eps_outside_sqrt", "1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)", 0),
    ("hardswish_div3", "t * c / 6.0", "t * c / 3.0", 0),
    ("hardswish_shift", "double c = t + 3.0;", "double c = t + 6.0;", 0),
    ("no_residual", "r[c] = v + hardswish(tanh(z));", "r[c] = hardswish(tanh(z));", 0),
    ("no_tanh", "r[c] = v + hardswish(tanh(z));", "r[c] = v + hardswish(z);", 0),
    ("group_by_modulo", "int64_t g = c / cpg;", "int64_t g = c % G;", 0),
    ("affine_per_group", "(double)gamma[c] + (double)beta[c]", "(double)gamma[g] + (double)beta[g]", 0),
    ("group_offset", "group_stats(yn + g * cpg * HW,", "group_stats(yn + g * HW,", 0),
    ("channel_lse_drops_max", "return m + log(s);", "return log(s);", 0),
    ("mean_not_subtracted", "double d = (double)p[k] - mean;", "double d = (double)p[k];", 0),
    ("stats_skip_non_finite",
     "double sum = 0.0;\n    for (int64_t k = 0; k < count; ++k) sum += (double)p[k];\n"
     "    double mean = sum / (double)count;\n    double sq = 0.0;\n"
     "    for (int64_t k = 0; k < count; ++k) {\n        double d = (double)p[k] - mean;",
     "double sum = 0.0;\n    int64_t nf = 0;\n"
     "    for (int64_t k = 0; k < count; ++k) if (isfinite(p[k])) { sum += (double)p[k]; ++nf; }\n"
     "    double mean = nf ? sum / (double)nf : 0.0;\n    double sq = 0.0;\n"
     "    for (int64_t k = 0; k < count; ++k) {\n        if (!isfinite(p[k])) continue;\n"
     "        double d = (double)p[k] - mean;", 0),
    ("beta_dropped", " + (double)beta[c];", ";", 0),
    ("softmax_without_exp", "out[r * cols + j] = exp((double)row[j] - lse);",
     "out[r * cols + j] = (double)row[j] - lse;", 0),
    ("softmax_unshifted", "exp((double)row[j] - lse)", "exp((double)row[j])", 0),
    ("dim_softmax_stride", "lse_strided_float(col, R, inner)", "lse_strided_float(col, R, 1)", 0),
    ("dim_softmax_index", "(double)col[r * inner] - lse", "(double)col[r] - lse", 0),
    ("groupnorm_eps_dropped", "double rs = 1.0 / sqrt(var + eps);", "double rs = 1.0 / sqrt(var);", 0),
    ("chain_no_residual", "act ? v + hardswish(tanh(z)) : z", "act ? hardswish(tanh(z)) : z", 0),
    ("groupnorm_affine_swapped", "(v - mu) * rs * (double)gamma[c] + (double)beta[c]",
     "(v - mu) * rs * (double)beta[c] + (double)gamma[c]", 0),
    ("conv_no_bias", "double acc = (double)b[co];", "double acc = 0.0;", 0),
    ("conv_taps_transposed", "x[((n * Cin + ci) * H + i + u) * W + j + v]",
     "x[((n * Cin + ci) * H + i + v) * W + j + u]", 0),
    ("conv_kernel_flipped", "w[((co * Cin + ci) * KH + u) * KW + v]",
     "w[((co * Cin + ci) * KH + (KH - 1 - u)) * KW + (KW - 1 - v)]", 0),
    ("conv_chain_unbiased", "rstd[g] = 1.0 / sqrt(sq / (double)count + eps);",
     "rstd[g] = 1.0 / sqrt(sq / (double)(count - 1) + eps);", 0),
    ("conv_chain_no_residual", "r[c] = v + hardswish(tanh(z));", "r[c] = hardswish(tanh(z));", 1),
]


def _replace_nth(text, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"mutation anchor not found: {old!r} (occurrence {n})"
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, nth):
    with open(oracle.SOURCE) as f:
        src = f.read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    c_path = os.path.join(tmp_path, f"{name}.c")
    with open(c_path, "w") as f:
        f.write(mutated)
    lib = oracle.compile_oracle(c_path, os.path.join(tmp_path, f"lib{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
            break
    assert caught, f"mutant {name} passed every pin"
