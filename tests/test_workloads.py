"""Seeded input generator: bf16 rounding, determinism, and the shapes and
timings printed on the pages (CPU only)."""
import os

import numpy as np
import torch

from channels_last_groupnorm_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "speedup_table_h200.txt")


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 10,
        # exact ties: the low 16 bits are 0x8000
        (((rng.integers(0, 1 << 15, 2000, dtype=np.uint32) << 16) | 0x8000)
         .astype(np.uint32).view(np.float32)),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40], np.float32),
    ])
    v = v[np.isfinite(v)]
    ours = wl.f32_to_bf16_bits(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(wl.bf16_bits_to_f32(ours),
                          torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_workloads_are_deterministic():
    w = wl.WORKLOADS[0]
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert a["x_bits"].shape == (w.N, w.L, w.C)
    assert a["gamma"].dtype == np.float32 and a["beta"].dtype == np.float32


def test_distributions_look_right():
    w = wl.WORKLOADS[0]
    inp = wl.make_inputs(w)
    x = wl.bf16_bits_to_f32(inp["x_bits"])
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert inp["gamma"].min() >= 0.5 and inp["gamma"].max() <= 1.5
    assert abs(inp["beta"].std() - 0.1) < 0.03


def test_offset_stress_case_has_channel_offsets():
    case = wl.make_case(1, 4096, 64, 3, mean=4.0, std=0.25, channel_offset=1.0)
    x = wl.bf16_bits_to_f32(case["x_bits"])[0]
    per_channel = x.mean(axis=0)
    assert per_channel.std() > 0.3          # U(-1,1) offsets: std ~0.58
    assert abs(x.std(axis=0).mean() - 0.25) < 0.02


def test_shapes_and_timings_match_the_pages_table():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        n, c, h, w, aten, old, new = line.split()
        rows.append(((int(n), int(c), int(h), int(w)), float(new)))
    table = dict(rows)
    quoted = [w for w in wl.WORKLOADS if w.pages_us_h200 is not None]
    assert len(quoted) == len(table) == 5
    for w in quoted:
        assert w.nchw in table, w.name
        assert table[w.nchw] == w.pages_us_h200


def test_general_workloads_draw_whole_rows_deterministically():
    w = wl.Workload("probe_c960", 10, 1, 960, 8, 8, D=3)
    assert w.general and w.L == 3 * 8 * 8
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    assert a["x_bits"].shape == (1, 192, 960)
    assert np.array_equal(a["x_bits"], b["x_bits"])
    assert {x.name for x in wl.GENERAL_WORKLOADS} <= set(wl.BY_NAME)
    assert all(x.general or x.D > 1 for x in wl.GENERAL_WORKLOADS)


def test_upconv_inputs_are_seeded_and_scaled():
    a = wl.make_upconv_case(1, 8, 4, 64, 128, 3)
    b = wl.make_upconv_case(1, 8, 4, 64, 128, 3)
    for k in ("x_bits", "w_bits", "bias_bits"):
        assert np.array_equal(a[k], b[k]), k
    assert a["x_bits"].shape == (1, 8, 4, 64) and a["w_bits"].shape == (128, 64, 3, 3)
    bound = 1.0 / np.sqrt(9 * 64)
    w = wl.bf16_bits_to_f32(a["w_bits"])
    assert np.abs(w).max() <= bound * (1 + 2 ** -8) and np.abs(w).max() > 0.9 * bound
    assert wl.make_upconv_case(1, 2, 2, 64, 128, 3, bias=False)["bias_bits"] is None
    big = wl.UPCONV_BY_NAME["upconv_c512_256x256"]
    assert (big.N, big.H, big.W, big.Cin, big.Cout) == (1, 256, 256, 512, 512)
    assert big.flops == 2 * 512 * 512 * 512 * 4 * 512
