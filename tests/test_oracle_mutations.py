"""The pins are strong enough: each plausible mistake planted in a copy of
the oracle's C source (on the CPU) makes at least one pin fail.

Every mutant is compiled from a temporary copy of ``oracle/gn_oracle.c``
with one textual edit; the real oracle file is never touched.
"""
import os

import pytest

import oracle
from tests import oracle_pins

# (name, original text, replacement, which occurrence (0-based))
MUTATIONS = [
    ("unbiased_variance", "const double v = sq / m;", "const double v = sq / (m - 1.0);", 0),
    ("eps_outside_sqrt", "1.0 / sqrt(v + eps)", "1.0 / sqrt(v) + eps", 0),
    ("no_sqrt", "1.0 / sqrt(v + eps)", "1.0 / (v + eps)", 0),
    ("dropped_beta", "* r * gam + bet;", "* r * gam;", 0),
    ("dropped_gamma", "* r * gam + bet;", "* r + bet;", 0),
    ("mean_not_subtracted", "(xv - mu) * r", "(xv) * r", 0),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));", 0),
    ("silu_without_z", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));", 0),
    ("mean_over_rows_only", "const double mu = sum / m;", "const double mu = sum / (double)L;", 0),
    ("row_stride", "sum += bf16_to_f64(xn[l * C + c]);", "sum += bf16_to_f64(xn[l * Cg + c]);", 0),
    ("group_of_channel", "const int64_t g = c / Cg;", "const int64_t g = c % G;", 0),
    ("gamma_by_group", "(double)gamma[c], (double)beta[c], apply_silu);",
     "(double)gamma[g], (double)beta[c], apply_silu);", 0),
    ("beta_transposed", "(double)gamma[c], (double)beta[c], apply_silu);",
     "(double)beta[c], (double)gamma[c], apply_silu);", 0),
    ("batch_offset", "const uint16_t *xn = x + n * L * C;", "const uint16_t *xn = x + n * C;", 0),
    ("stats_index", "mean[n * G + g], rstd[n * G + g]", "mean[g], rstd[g]", 0),
    ("bf16_decode", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15", 0),
    ("second_pass_not_centered", "const double d = bf16_to_f64(xn[l * C + c]) - mu;",
     "const double d = bf16_to_f64(xn[l * C + c]);", 0),
    ("apply_at_batch", "const int64_t n = at / (L * C);", "const int64_t n = at / L;", 0),
    ("apply_at_channel", "const int64_t c = at % C;", "const int64_t c = at % L;", 0),
    ("apply_at_group", "const int64_t g = c / Cg;", "const int64_t g = c / G;", 1),
]


def _mutate(text, old, new, occurrence):
    start = -1
    for _ in range(occurrence + 1):
        start = text.find(old, start + 1)
        if start < 0:
            raise AssertionError(f"mutation anchor not found: {old!r} #{occurrence}")
    return text[:start] + new + text[start + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, occ):
    src = open(oracle.SOURCE).read()
    code_start = src.index("#include")      # anchors must not land in the header comment
    mutated = src[:code_start] + _mutate(src[code_start:], old, new, occ)
    assert mutated != src
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.build(source=path, out=os.path.join(tmp_path, f"libmut_{name}.so"), force=True)
    failed = oracle_pins.failing_pins(oracle.Oracle(lib))
    assert failed, f"no pin caught the planted mistake {name!r}"
