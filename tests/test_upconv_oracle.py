"""The upsample + 3x3 conv oracle against its pins (CPU), and the pins'
strength: plausible mistakes planted in copies of upconv_oracle.c each fail
a pin."""
import os

import pytest

import oracle
from tests import upconv_pins


@pytest.mark.parametrize("pin", upconv_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(oracle.upconv()) == []


MUTATIONS = [
    # (name, original text, replacement)
    ("upsample_rounds_up", "const int64_t i = p / 2, j = q / 2;",
     "const int64_t i = (p + 1) / 2 < pr->H ? (p + 1) / 2 : pr->H - 1, j = q / 2;"),
    ("no_zero_padding", "if (p < 0 || q < 0 || p >= 2 * pr->H || q >= 2 * pr->W) return 0.0;",
     "if (p < 0) p = 0;\n    if (q < 0) q = 0;\n    if (p >= 2 * pr->H) p = 2 * pr->H - 1;\n"
     "    if (q >= 2 * pr->W) q = 2 * pr->W - 1;"),
    ("window_not_centered", "upsampled(pr, n, P + ky - 1, Q + kx - 1, ci)",
     "upsampled(pr, n, P + ky, Q + kx - 1, ci)"),
    ("kernel_transposed", "pr->wd[((co * pr->Cin + ci) * 3 + ky) * 3 + kx]",
     "pr->wd[((co * pr->Cin + ci) * 3 + kx) * 3 + ky]"),
    ("kernel_flipped", "pr->wd[((co * pr->Cin + ci) * 3 + ky) * 3 + kx]",
     "pr->wd[((co * pr->Cin + ci) * 3 + (2 - ky)) * 3 + (2 - kx)]"),
    ("dropped_bias", "double s = pr->bias ? bf16_value(pr->bias[co]) : 0.0;", "double s = 0.0;"),
    ("channel_stride", "return bf16_value(pr->x[((n * pr->H + i) * pr->W + j) * pr->Cin + ci]);",
     "return bf16_value(pr->x[((n * pr->H + i) * pr->W + j) + ci * pr->H * pr->W * 0]);"),
    ("batch_ignored", "return bf16_value(pr->x[((n * pr->H + i) * pr->W + j) * pr->Cin + ci]);",
     "return bf16_value(pr->x[((0 * n * pr->H + i) * pr->W + j) * pr->Cin + ci]);"),
    ("weight_in_out_swapped", "pr->wd[((co * pr->Cin + ci) * 3 + ky) * 3 + kx]",
     "pr->wd[((ci * pr->Cout + co) * 3 + ky) * 3 + kx]"),
    ("at_channel", "const int64_t co = at % Cout, pix = at / Cout;",
     "const int64_t co = at / (N * OH * OW) % Cout, pix = at % (N * OH * OW);"),
    ("abs_of_sum", "t += fabs(u * w);", "t += u * w;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(oracle.UPCONV_SOURCE).read()
    code_start = src.index("#include")
    body = src[code_start:]
    assert body.count(old) == 1, f"mutation anchor for {name!r} not unique"
    mutated = src[:code_start] + body.replace(old, new)
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.build(source=path, out=os.path.join(tmp_path, f"libmut_{name}.so"), force=True)
    failed = upconv_pins.failing_pins(oracle.UpconvOracle(lib))
    assert failed, f"no pin caught the planted mistake {name!r}"
