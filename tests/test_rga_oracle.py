"""The residual-gate oracle against its pins (CPU), and the pins' strength:
plausible mistakes planted in copies of rga_oracle.c each fail a pin."""
import os

import pytest

import oracle
from tests import rga_pins


@pytest.mark.parametrize("pin", rga_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(oracle.rga()) == []


MUTATIONS = [
    # (name, original text, replacement)
    ("single_rounding", "    const uint16_t p = round_half((float)prod, fmt);            /* (float) is exact here */\n"
     "    const double sum = decode(res, fmt) + decode(p, fmt);",
     "    const double sum = decode(res, fmt) + prod;"),
    ("product_not_rounded_to_half", "const double sum = decode(res, fmt) + decode(p, fmt);",
     "const double sum = decode(res, fmt) + (double)(float)prod + 0.0 * p;"),
    ("bf16_ties_up", "    w += 0x7fffu + lsb;", "    w += 0x8000u + 0 * lsb;"),
    ("f16_ties_up", "if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;",
     "if (rem >= 0.5) fl += 1.0;"),
    ("f16_no_subnormals", "    if (q < -24) q = -24;", "    if (q < -24) q = -14 - 10 + 0 * q;\n    if (e - 1 < -14) return sign;"),
    ("gate_by_row", "out[at] = residual_gate_one(residual[at], update[at], gate[d], fmt);",
     "out[at] = residual_gate_one(residual[at], update[at], gate[r % D], fmt);"),
    ("operands_swapped", "out[at] = residual_gate_one(residual[at], update[at], gate[d], fmt);",
     "out[at] = residual_gate_one(update[at], residual[at], gate[d], fmt);"),
    ("f16_decode_bias", "v = ldexp((double)(man | 0x400), ex - 25);", "v = ldexp((double)(man | 0x400), ex - 24);"),
    ("at_gate_index", "gate[at % D]", "gate[at / D % D]"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(oracle.RGA_SOURCE).read()
    code_start = src.index("#include")
    body = src[code_start:]
    assert body.count(old) == 1, f"mutation anchor for {name!r} not unique"
    mutated = src[:code_start] + body.replace(old, new)
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.build(source=path, out=os.path.join(tmp_path, f"libmut_{name}.so"), force=True)
    failed = rga_pins.failing_pins(oracle.RgaOracle(lib))
    assert failed, f"no pin caught the planted mistake {name!r}"
