"""The attention-block oracle against its pins (CPU), and the pins'
strength: plausible mistakes planted in copies of attn_oracle.c each fail a
pin."""
import os

import pytest

import oracle
from tests import attn_pins


@pytest.mark.parametrize("pin", attn_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(oracle.attn()) == []


MUTATIONS = [
    # (name, original text, replacement)
    ("no_scale", "const double scale = 1.0 / sqrt((double)D);", "const double scale = 1.0;"),
    ("scale_one_over_d", "const double scale = 1.0 / sqrt((double)D);", "const double scale = 1.0 / (double)D;"),
    ("no_value_bias", "double acc = bf(bv[c]), mag = fabs(bf(bv[c]));", "double acc = 0.0, mag = fabs(bf(bv[c]));"),
    ("no_output_bias", "double acc = t->bo[e], m = fabs(t->bo[e]) + fabs(rv);",
     "double acc = 0.0, m = fabs(t->bo[e]) + fabs(rv);"),
    ("value_weight_transposed", "const double p = bf(xn[j * D + i]) * wvd[c * D + i];",
     "const double p = bf(xn[j * D + i]) * wvd[i * D + c];"),
    ("output_weight_transposed", "acc += o[c] * t->wo[e * D + c];", "acc += o[c] * t->wo[c * D + e];"),
    ("residual_dropped", "out[e] = acc + rv;", "out[e] = acc;"),
    ("not_normalised", "for (int64_t j = 0; j < S; ++j) a[j] /= l;", "for (int64_t j = 0; j < S; ++j) a[j] /= 1.0;"),
    ("query_is_key", "s += bf(t->q[r * D + d]) * bf(t->k[j * D + d]);",
     "s += bf(t->k[r * D + d]) * bf(t->k[j * D + d]);"),
    ("rows_ignored", "att_row(&t, rows ? rows[i] : i,", "att_row(&t, i,"),
    ("magnitude_signed", "m += oa[c] * fabs(t->wo[e * D + c]);", "m += oa[c] * t->wo[e * D + c];"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(oracle.ATTN_SOURCE).read()
    code_start = src.index("#include")
    body = src[code_start:]
    assert body.count(old) == 1, f"mutation anchor for {name!r} not unique"
    mutated = src[:code_start] + body.replace(old, new)
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.build(source=path, out=os.path.join(tmp_path, f"libmut_{name}.so"), force=True)
    failed = attn_pins.failing_pins(oracle.AttnOracle(lib))
    assert failed, f"no pin caught the planted mistake {name!r}"
