"""Single-head attention with the output projection folded into V on the
GPU (gn_attn_fold + gn_attn_folded, both schedules: the one-pass CTA-pair
kernel with the scores kept on chip, and the stored-weights GEMMs) against
the fp64 oracle of the UNFOLDED block (value projection, softmax
attention, output projection, residual; sglang PR #33451, "FLUX.2 VAE
decoder fast path behind quality=high", section "Modifications", item 2,
attention bullet).

Acceptance bound, per output, derived from the arithmetic (one bf16
rounding errs by at most u = 2^-8 relative): the folded weight, the folded
value rows and the softmax weights are each rounded to bf16 once (each
perturbs the output by at most 2^-8 of the magnitude M = |bo| + |residual| +
sum_c |wo| sum_j a_j (|bv| + sum_i |xn wv|) that the oracle returns), fp32
scores and accumulations add far less, and the output is rounded to bf16
(2^-8 |y|); together less than
    |y_gpu - y_ref| <= 2^-6 M + 2^-7 |y_ref|.
The rms check below (rms error < 2^-7 of the rms output) is what a dropped
bias or a mis-scaled softmax would fail first.
"""
import numpy as np
import pytest
import torch

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    gs.lib()
    yield
    gu.assert_clean_device()


def dev(bits):
    if bits is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


ONE_PASS, STORED = gs.ATTN_ONE_PASS, gs.ATTN_STORED_WEIGHTS
SCHEDULES = pytest.mark.parametrize("schedule", [ONE_PASS, STORED], ids=["one_pass", "stored_weights"])


def run(c, residual_in_place=False, schedule=gs.ATTN_AUTO):
    wf, bf = gs.attn_fold(dev(c["wv"]), dev(c["bv"]), dev(c["wo"]), dev(c["bo"]))
    res = dev(c["residual"])
    out = res if residual_in_place else None
    y = gs.attention_folded(dev(c["q"]), dev(c["k"]), dev(c["xn"]), wf, bf, residual=res, out=out,
                            schedule=schedule)
    assert y is not None, "the CUDA path rejected a supported input"
    torch.cuda.synchronize()
    assert gs.gn_device_status(False) == 0
    return y


def check(got, ref, mag, what):
    err = np.abs(got - ref)
    bound = 2.0 ** -6 * mag + 2.0 ** -7 * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the bound; worst err "
                           f"{err.max():.3e}")
    rel = np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    assert rel < 2.0 ** -7, f"{what}: rms error {rel:.3e} of the rms output"


def oracle_args(c):
    return (c["q"], c["k"], c["xn"], c["wv"], c["bv"], c["wo"], c["bo"], c["residual"])


@SCHEDULES
@pytest.mark.parametrize("S,D,residual", [(256, 512, True), (256, 512, False), (384, 128, True),
                                          (128, 256, True), (640, 384, False),
                                          (1024, 512, True),    # weighted sum on CTA pairs (K = S >= 1024)
                                          (256, 1024, False)])  # the widest D the entry takes
def test_matches_oracle(S, D, residual, schedule):
    c = wl.make_attn_case(S, D, S + D, residual)
    if schedule == ONE_PASS and D > 512:
        assert run_none(c, schedule), "the one-pass schedule takes D <= 512 only"
        return
    y = run(c, schedule=schedule).float().cpu().numpy().astype(np.float64)
    ref, mag = oracle.attn().forward(*oracle_args(c), with_mag=True)
    check(y, ref, mag, f"S={S} D={D} residual={residual}")


def run_none(c, schedule):
    wf, bf = gs.attn_fold(dev(c["wv"]), dev(c["bv"]), dev(c["wo"]), dev(c["bo"]))
    return gs.attention_folded(dev(c["q"]), dev(c["k"]), dev(c["xn"]), wf, bf, schedule=schedule) is None


@SCHEDULES
def test_in_place_on_the_residual(schedule):
    c = wl.make_attn_case(256, 512, 3)
    ref, mag = oracle.attn().forward(*oracle_args(c), with_mag=True)
    y = run(c, residual_in_place=True, schedule=schedule).float().cpu().numpy().astype(np.float64)
    check(y, ref, mag, "in place")


@pytest.mark.parametrize("S,one_pass", [(2048, False), (4096, True), (16384, True)])
def test_auto_schedule(S, one_pass):
    """ATTN_AUTO takes the one-pass kernel from 32 query tiles on and the
    stored-weights GEMMs below (five launches)."""
    D = 512
    q = torch.zeros(S, D, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(D, D, dtype=torch.bfloat16, device="cuda")
    wf, bf = gs.attn_fold(w, q[0], w.clone(), q[1])
    torch.cuda.synchronize()
    before = gs.gn_kernel_launch_count()
    assert gs.attention_folded(q, q, q, wf, bf) is not None
    torch.cuda.synchronize()
    # one pass: the value rows, the pair kernel and, when tiles are split
    # between CTA pairs, the merge of their pieces
    assert gs.gn_kernel_launch_count() - before in ((2, 3) if one_pass else (5,))


@pytest.mark.parametrize("S,D,residual,in_place", [(640, 512, True, False), (1024, 512, False, False),
                                                   (512, 256, True, False), (768, 384, True, False),
                                                   (640, 512, True, True)])
def test_one_pass_split_tiles_match_oracle(S, D, residual, in_place):
    """With a workspace larger than the minimum the one-pass schedule can
    give CTA pairs equal shares of (tile, key block) units; at these shapes
    its estimate prefers that, so the tiles are split into pieces (down to
    one key block each) that a third kernel merges by their row maxima and
    sums."""
    c = wl.make_attn_case(S, D, 3 * S + D, residual)
    wf, bf = gs.attn_fold(dev(c["wv"]), dev(c["bv"]), dev(c["wo"]), dev(c["bo"]))
    need = gs.gn_attn_workspace_bytes(S, D)
    ws = torch.zeros(need + 2 * 152 * (D * 128 + 256) * 4, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    before = gs.gn_kernel_launch_count()
    res = dev(c["residual"])
    y = gs.attention_folded(dev(c["q"]), dev(c["k"]), dev(c["xn"]), wf, bf, residual=res,
                            out=res if in_place else None, workspace=ws, schedule=ONE_PASS)
    torch.cuda.synchronize()
    assert y is not None and gs.gn_device_status(False) == 0
    assert gs.gn_kernel_launch_count() - before == 3, "expected the pieces to be merged"
    ref, mag = oracle.attn().forward(*oracle_args(c), with_mag=True)
    check(y.float().cpu().numpy().astype(np.float64), ref, mag, f"split S={S} D={D}")


def test_fold_matches_the_weight_product():
    D = 512
    c = wl.make_attn_case(128, D, 21)
    wf, bf = gs.attn_fold(dev(c["wv"]), dev(c["bv"]), dev(c["wo"]), dev(c["bo"]))
    torch.cuda.synchronize()
    v = lambda n: wl.bf16_bits_to_f32(c[n]).astype(np.float64).reshape(np.shape(c[n]))  # noqa: E731
    w_want = v("wo") @ v("wv")
    b_want = v("wo") @ v("bv") + v("bo")
    w_abs = np.abs(v("wo")) @ np.abs(v("wv"))
    b_abs = np.abs(v("wo")) @ np.abs(v("bv")) + np.abs(v("bo"))
    wg = wf.float().cpu().numpy().astype(np.float64)
    bg = bf.cpu().numpy().astype(np.float64)
    # one bf16 rounding (2^-8 relative) after an fp32 sum of D products
    # (at most D 2^-24 = 2^-15 of the sum of their magnitudes)
    assert np.all(np.abs(wg - w_want) <= 2.0 ** -8 * np.abs(w_want) + 2.0 ** -14 * w_abs)
    assert np.all(np.abs(bg - b_want) <= 2.0 ** -14 * b_abs)


@SCHEDULES
@pytest.mark.parametrize("name,rows", [("attn_s4096_d512", 48), ("attn_s16384_d512", 24)])
def test_decoder_shapes_sampled(name, rows, schedule):
    """The FLUX.2 mid-block shapes in full, sampled query rows (first, last,
    tile edges, random) against the oracle row by row."""
    w = wl.ATTN_BY_NAME[name]
    c = wl.make_attn_inputs(w)
    y = run(c, schedule=schedule)
    idx = np.unique(np.concatenate([[0, 1, 127, 128, w.S - 1],
                                    np.random.default_rng(7).integers(0, w.S, rows)]))
    got = y[torch.from_numpy(idx).cuda()].float().cpu().numpy().astype(np.float64)
    ref, mag = oracle.attn().rows(*oracle_args(c), idx, with_mag=True)
    check(got, ref, mag, name)


def test_longest_sequence_one_pass_sampled():
    """S = 32768, the longest the entry takes, on the one-pass schedule: every
    CTA pair takes ~6.7 tiles' worth of units, so its run crosses several
    tile boundaries (pieces at both ends); sampled rows, including the
    first and last rows of tiles, against the oracle."""
    S, D = 32768, 512
    c = wl.make_attn_case(S, D, 5, True)
    y = run(c, schedule=ONE_PASS)
    idx = np.unique(np.concatenate([[0, 127, 128, 255, S - 129, S - 128, S - 1],
                                    np.random.default_rng(11).integers(0, S, 12)]))
    got = y[torch.from_numpy(idx).cuda()].float().cpu().numpy().astype(np.float64)
    ref, mag = oracle.attn().rows(*oracle_args(c), idx, with_mag=True)
    check(got, ref, mag, "S=32768 one pass")


@SCHEDULES
def test_deterministic(schedule):
    c = wl.make_attn_case(512, 512, 5)
    a = run(c, schedule=schedule).cpu()
    b = run(c, schedule=schedule).cpu()
    assert torch.equal(a, b)


def test_unsupported_inputs_return_none():
    q = torch.zeros(256, 512, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(512, 512, dtype=torch.bfloat16, device="cuda")
    wf, bf = gs.attn_fold(w, q[0], w.clone(), q[1])
    assert gs.attention_folded(q.float(), q, q, wf, bf) is None                 # fp32
    q100 = torch.zeros(100, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.warns(UserWarning):
        assert gs.attention_folded(q100, q100, q100, wf, bf) is None           # S not a multiple of 128
    assert gs.attention_folded(q.t(), q, q, wf, bf) is None                    # not contiguous


def test_single_cta_gemm_schedule_matches_oracle():
    """The single-CTA GEMM schedule (taken for row counts that are not a
    multiple of 256, for fewer than 16 K steps, and for every GEMM with
    GN_GEMM_PAIR=0) on a shape whose weighted sum the CTA-pair schedule
    would otherwise take, in a child process."""
    import os
    import subprocess
    import sys
    code = (
        "import numpy as np, torch, oracle\n"
        "from channels_last_groupnorm_gb300 import gnsilu as gs, workloads as wl\n"
        "c = wl.make_attn_case(1024, 512, 77)\n"
        "d = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(torch.bfloat16)\n"
        "wf, bf = gs.attn_fold(d(c['wv']), d(c['bv']), d(c['wo']), d(c['bo']))\n"
        "y = gs.attention_folded(d(c['q']), d(c['k']), d(c['xn']), wf, bf, residual=d(c['residual']))\n"
        "torch.cuda.synchronize()\n"
        "assert gs.gn_device_status(False) == 0\n"
        "ref, mag = oracle.attn().forward(c['q'], c['k'], c['xn'], c['wv'], c['bv'], c['wo'], c['bo'],\n"
        "                                 c['residual'], with_mag=True)\n"
        "err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)\n"
        "assert np.all(err <= 2.0 ** -6 * mag + 2.0 ** -7 * np.abs(ref)), err.max()\n"
        "print('ok')\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GN_GEMM_PAIR="0", PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
