"""Fused nearest-2x upsample + 3x3 conv on the GPU (gn_upconv_fold +
gn_upconv_nhwc, tcgen05 tensor cores) against the fp64 oracle, which
evaluates the upsample and the convolution as defined (sglang PR #33451,
"FLUX.2 VAE decoder fast path behind quality=high", section "Modifications",
item 2).

Acceptance bound, per output, derived from the arithmetic (bf16 keeps 8
significant bits: one rounding errs by at most u = 2^-8 relative): the
summed taps are rounded to bf16 (so the products they enter err by at most
2^-8 of the sum of |x * w| over their constituent 3x3 taps), the tensor
cores accumulate in fp32 (at most K 2^-24 of the same sum, K = 4 Cin <=
2048 here: 2^-13), and the result is rounded to bf16 (2^-8 |y|); together
less than
    |y_gpu - y_ref| <= 2^-7 (S + |y_ref|),   S = |bias| + sum |u * w|
(S is returned by the oracle).  Wrong indexing or a wrong tap moves outputs
by about |y| (~0.6 here), far above the bound (~0.08); the rms check below
is tighter still.
"""
import numpy as np
import pytest
import torch

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu
from tests import upconv_pins as up

pytestmark = pytest.mark.gpu

BOUND = 2.0 ** -7


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    gs.lib()
    yield
    gu.assert_clean_device()


def to_dev(bits, shape=None):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    return t if shape is None else t.reshape(shape)


def device_case(c):
    N, H, W, Cin = c["x_bits"].shape
    x = to_dev(c["x_bits"]).reshape(N, H, W, Cin).permute(0, 3, 1, 2)   # channels_last view
    w = to_dev(c["w_bits"]).contiguous()
    b = None if c["bias_bits"] is None else to_dev(c["bias_bits"])
    return x, w, b


def run_device(c, stream=None):
    """y as a device tensor [N, 2H, 2W, Cout] (the NHWC view of the result)."""
    x, w, b = device_case(c)
    wf = gs.upconv_fold(w, stream=stream)
    assert wf is not None, "upconv_fold rejected a supported weight"
    y = gs.upsample_conv_nhwc(x, wf, b, stream=stream)
    assert y is not None, "upsample_conv_nhwc rejected a supported input"
    torch.cuda.synchronize()
    return y.permute(0, 2, 3, 1)


def run(c, stream=None):
    return run_device(c, stream).float().cpu().numpy().astype(np.float64)


def check(got, ref, absum, what):
    err = np.abs(got - ref)
    bound = BOUND * (absum + np.abs(ref))
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outputs outside the bound; worst "
                           f"err {err.max():.3e} (bound there {bound.reshape(-1)[np.argmax(err)]:.3e})")
    # typical quality: the rms error is a small fraction of the rms output
    rel = np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    assert rel < 2.0 ** -7, f"{what}: rms error {rel:.3e} of the rms output"


SMALL = [
    # (N, H, W, Cin, Cout, bias): several tiles, each tiling mode, ragged image groups
    (1, 16, 16, 64, 128, True),      # W < 128: 8-row boxes
    (3, 8, 8, 64, 256, True),        # two images per tile, last tile half outside N
    (1, 4, 128, 128, 128, False),    # W = 128: one row per tile, no bias
    (2, 2, 32, 64, 384, True),       # Cout 384: three 128-wide channel tiles
    (1, 1, 256, 64, 128, True),      # a single input row (every tap row but one is padding)
    (2, 16, 8, 192, 256, True),      # Cin 192: three K chunks per tap
    (1, 1, 1, 64, 128, True),        # one input pixel, one tile mostly outside the image
    (2, 2, 128, 64, 256, False),     # W = 128, two images, CTA pairs, no bias
    (3, 1, 128, 128, 512, True),     # odd number of pixel tiles: the last pair's second tile is past the batch
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:5])) + ("" if s[5] else "-nobias"))
def test_matches_oracle(shape):
    N, H, W, Cin, Cout, bias = shape
    c = wl.make_upconv_case(N, H, W, Cin, Cout, sum(shape[:5]), bias)
    ref, absum = oracle.upconv().forward(c["x_bits"], c["w_bits"], c["bias_bits"], with_abs=True)
    check(run(c), ref, absum, str(shape))


def test_fold_layout_and_rounding():
    """The folded weight [4 parities][Cout][4 taps][Cin] equals the summed
    3x3 taps (the transposed-conv identity's 4x4 kernel read per parity),
    rounded once to bf16."""
    Cin, Cout = 64, 128
    c = wl.make_upconv_case(1, 1, 1, Cin, Cout, 77)
    w = wl.bf16_bits_to_f32(c["w_bits"]).astype(np.float64).reshape(Cout, Cin, 3, 3)
    wf = gs.upconv_fold(to_dev(c["w_bits"]).contiguous())
    torch.cuda.synchronize()
    got = wf.float().cpu().numpy().astype(np.float64).reshape(4, Cout, 2, 2, Cin)
    # output row P = 2i + a reads input row i + a - 1 + r; the transposed
    # convolution (P = 2 i_in - 1 + k) reaches it through tap k = 3 - a - 2r
    for a in range(2):
        for b in range(2):
            for r in range(2):
                for s in range(2):
                    k1, k2 = 3 - a - 2 * r, 3 - b - 2 * s
                    want = np.zeros((Cout, Cin))
                    for ky in up._SUMMED_ROWS[k1]:
                        for kx in up._SUMMED_ROWS[k2]:
                            want += w[:, :, ky, kx]
                    g = got[2 * a + b, :, r, s, :]
                    assert np.all(np.abs(g - want) <= 2.0 ** -8 * np.abs(want) + 1e-30), (a, b, r, s)


@pytest.mark.parametrize("name", ["upconv_c512_128x128", "upconv_c512_256x256", "upconv_c256_512x512"])
def test_decoder_shapes_sampled(name):
    """The FLUX.2 decoder up-sampler shapes at full size, in the launch the
    benchmark times: 4096 sampled outputs (image corners and edges, tile
    boundaries and random positions) against the oracle one by one."""
    wk = wl.UPCONV_BY_NAME[name]
    c = wl.make_upconv_inputs(wk)
    y = run_device(c)
    N, OH, OW, Cout = y.shape
    rng = np.random.default_rng(5)
    pts = [(0, 0), (0, OW - 1), (OH - 1, 0), (OH - 1, OW - 1), (1, 1), (OH - 2, OW - 2),
           (255, 255), (256, 256), (1, 254), (2, 257)]
    idx = []
    for (P, Q) in pts:
        if P < OH and Q < OW:
            for co in (0, 1, Cout // 2, Cout - 1):
                idx.append(((0 * OH + P) * OW + Q) * Cout + co)
    idx = np.array(idx + list(rng.integers(0, y.numel(), 4096 - len(idx))), np.int64)
    got = y.reshape(-1)[torch.from_numpy(idx).cuda()].float().cpu().numpy().astype(np.float64)
    ref, absum = oracle.upconv().at(c["x_bits"], c["w_bits"], c["bias_bits"], idx, with_abs=True)
    check(got, ref, absum, name)


def test_deterministic_and_on_a_side_stream():
    c = wl.make_upconv_case(2, 8, 16, 128, 256, 31)
    a = run(c)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run(c, stream=s)
    assert np.array_equal(a, b)


def test_empty_batch_is_a_no_op():
    x = torch.zeros(0, 64, 8, 8, dtype=torch.bfloat16, device="cuda").to(memory_format=torch.channels_last)
    wf = gs.upconv_fold(torch.zeros(128, 64, 3, 3, dtype=torch.bfloat16, device="cuda"))
    y = gs.upsample_conv_nhwc(x, wf)
    torch.cuda.synchronize()
    assert y is not None and tuple(y.shape) == (0, 128, 16, 16)


def test_unsupported_inputs_return_none():
    dev = "cuda"
    w = torch.zeros(128, 64, 3, 3, dtype=torch.bfloat16, device=dev)
    wf = gs.upconv_fold(w)
    x = torch.zeros(1, 64, 8, 8, dtype=torch.bfloat16, device=dev)
    assert gs.upsample_conv_nhwc(x, wf) is None                       # NCHW, not channels_last
    x96 = torch.zeros(1, 64, 8, 96, dtype=torch.bfloat16, device=dev).to(memory_format=torch.channels_last)
    with pytest.warns(UserWarning):
        assert gs.upsample_conv_nhwc(x96, wf) is None                 # W = 96 has no tiling
    with pytest.warns(UserWarning):
        assert gs.upconv_fold(torch.zeros(100, 64, 3, 3, dtype=torch.bfloat16, device=dev)) is None
    assert gs.upconv_fold(w.float()) is None


def test_single_sm_schedule_matches_oracle():
    """The single-CTA schedule (taken when the CTA-pair kernel is switched
    off with GN_UPCONV_PAIR=0, and always for Cout not a multiple of 256) on
    a 256-channel case, in a child process (the switch is read once)."""
    import os
    import subprocess
    import sys
    code = (
        "import numpy as np, torch, oracle\n"
        "from channels_last_groupnorm_gb300 import gnsilu as gs, workloads as wl\n"
        "c = wl.make_upconv_case(2, 8, 16, 128, 512, 41)\n"
        "d = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(torch.bfloat16)\n"
        "x = d(c['x_bits']).reshape(2, 8, 16, 128).permute(0, 3, 1, 2)\n"
        "wf = gs.upconv_fold(d(c['w_bits']).reshape(512, 128, 3, 3).contiguous())\n"
        "y = gs.upsample_conv_nhwc(x, wf, d(c['bias_bits']))\n"
        "torch.cuda.synchronize()\n"
        "assert gs.gn_device_status(False) == 0\n"
        "ref, ab = oracle.upconv().forward(c['x_bits'], c['w_bits'], c['bias_bits'], with_abs=True)\n"
        "err = np.abs(y.permute(0, 2, 3, 1).float().cpu().numpy().astype(np.float64) - ref)\n"
        "assert np.all(err <= 2.0 ** -8 * (ab + np.abs(ref))), err.max()\n"
        "print('ok')\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GN_UPCONV_PAIR="0", PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
