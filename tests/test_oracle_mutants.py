"""Plant plausible mistakes in copies of the CPU oracle and show that the pins
catch every one of them.

Each mutant is a textual edit of oracle/zero_oracle.c compiled to a temporary
library; the real oracle is never modified.  A mutant "survives" if every
check in tests/oracle_checks.py still passes on it, which would mean the pins
could not tell that mistake from the method.
"""
import os
import shutil
import subprocess

import pytest

import oracle as oracle_pkg
import oracle_checks

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "zero_oracle.c")

MUTANTS = {
    "m_sign": ("(1.0 - beta1) * gi", "(1.0 + beta1) * gi"),
    "no_bias_correction_m": ("double m_hat = (double)m_new / bc1;", "double m_hat = (double)m_new;"),
    "no_bias_correction_v": ("double v_hat = (double)v_new / bc2;", "double v_hat = (double)v_new;"),
    "bias_exponent_off_by_one": ("pow(beta1, (double)step)", "pow(beta1, (double)(step + 1))"),
    "eps_inside_sqrt": ("(sqrt(v_hat) + eps)", "sqrt(v_hat + eps)"),
    "no_weight_decay": ("(1.0 - lr * weight_decay)", "(1.0)"),
    "v_uses_g": ("(1.0 - beta2) * gi * gi", "(1.0 - beta2) * gi"),
    "sum_not_mean": ("(float)(sum / (double)n_ranks)", "(float)sum"),
    "mean_over_wrong_count": ("(float)(sum / (double)n_ranks)", "(float)(sum / (double)(n_ranks + 1))"),
    "rs_transposed_stride": ("mean_over_ranks(grads, n_ranks, P_pad, e);\n        }\n    }\n}",
                             "mean_over_ranks(grads, n_ranks, S, e);\n        }\n    }\n}"),
    "bf16_truncate": ("u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    "bf16_ties_away": ("u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;"),
    "layout_offsets_shifted": ("offsets[i] = running;", "offsets[i] = running + (i > 0);"),
    "layout_extra_pad": ("int64_t P_pad = P + pad;", "int64_t P_pad = P + pad + (pad == 0 ? 0 : n_ranks);"),
    "gather_wrong_rank": ("full[(int64_t)r * S + i] = shards[(int64_t)r * S + i];",
                          "full[(int64_t)r * S + i] = shards[(int64_t)((r + 1) % n_ranks) * S + i];"),
    "accum_not_reset": ("if (first) {", "if (0) {"),
    "accum_no_average": ("(double)acc[i] / (double)n_micro", "(double)acc[i]"),
    "clip_no_sqrt": ("double norm = sqrt(total_sum_squares);", "double norm = total_sum_squares;"),
    "clip_no_clamp": ("if (coef >= 1.0) {", "if (coef >= 1e300) {"),
    "clip_no_eps": ("double coef = max_norm / (norm + 1e-6);", "double coef = max_norm / norm;"),
    "clip_scale_ignored": ("g[i] = (float)((double)g[i] * (double)coef);", "g[i] = g[i];"),
    "clip_nan_coefficient_ignored": ("if (coef >= 1.0) {", "if (!(coef < 1.0)) {"),
    "zero1_accum_not_reset": ("double prev = first ? 0.0 : (double)acc_full[idx];",
                              "double prev = (double)acc_full[idx];"),
    "zero1_no_micro_average": ("g[e] = (float)((double)mean / (double)n_micro);", "g[e] = mean;"),
    "fsdp2_floor_chunk": ("int64_t chunk = (dim0 + n_ranks - 1) / n_ranks;",
                          "int64_t chunk = dim0 / n_ranks + (dim0 % n_ranks > 1);"),
    "fsdp2_rows_not_scaled": ("*begin = first_row * row_numel;", "*begin = first_row;"),
    "decay_after_update": ("double updated = decayed - lr * m_hat / (sqrt(v_hat) + eps);",
                           "double updated = ((double)theta[i] - lr * m_hat / (sqrt(v_hat) + eps)) * (1.0 - lr * weight_decay * 1.5);"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return tmp_path_factory.mktemp("oracle_mutants")


def _build_mutant(tmpdir, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    text = text.replace(old, new, 1)
    src = os.path.join(str(tmpdir), f"{name}.c")
    with open(src, "w") as f:
        f.write(text)
    out = os.path.join(str(tmpdir), f"lib{name}.so")
    subprocess.run(["gcc", *oracle_pkg.CFLAGS, "-o", out, src, "-lm"], check=True,
                   capture_output=True)
    return out


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(mutant_dir, name):
    old, new = MUTANTS[name]
    lib = oracle_pkg.load(_build_mutant(mutant_dir, name, old, new))
    o = oracle_pkg.Oracle(lib)
    caught = []
    for check in oracle_checks.ALL_CHECKS:
        try:
            check(o)
        except Exception as exc:   # an assertion, or an error the mistake provokes
            caught.append((check.__name__, type(exc).__name__))
    assert caught, f"planted mistake '{name}' passed every pin"
