"""Generalised channel counts and 5D input (GPU): gn_silu_rows_any and
gn_silu_ndhwc against the fp64 oracle.

These entry points widen C from powers of two to any multiple of 8 up to
2048 with any G dividing C (any channels per group, e.g. C = 320 or 960),
and add 5D channels-last input: the range of the existing general kernel on
the sglang PR #33451 page ("FLUX.2 VAE decoder fast path behind
quality=high", section "Modifications", item 1, third bullet).  The oracle
needs no change for them: its definition never assumed a power of two."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

VARIANTS = [gs.VARIANT_FUSED, gs.VARIANT_TWO_PASS]
ALL_VARIANTS = VARIANTS + [gs.VARIANT_CLUSTER]
VNAME = {gs.VARIANT_FUSED: "fused", gs.VARIANT_TWO_PASS: "two_pass", gs.VARIANT_CLUSTER: "cluster"}


def skip_unless_cluster_fits(N, L, C, G, variant):
    """The explicit cluster variant is refused (GN_ERR_VARIANT) for shapes
    whose slices do not fit the clusters' shared memory."""
    if variant != gs.VARIANT_CLUSTER:
        return
    x = torch.zeros((N, L, C), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(C, device="cuda")
    rc = gs.raw_gn_silu_rows_any(x.data_ptr(), g.data_ptr(), g.data_ptr(), x.data_ptr(), N, L, C, G, 1e-6, 1,
                                 variant=gs.VARIANT_CLUSTER)
    torch.cuda.synchronize()
    assert rc in (gs.GN_OK, gs.GN_ERR_VARIANT), gs.status_string(rc)
    if rc != gs.GN_OK:
        pytest.skip("the cluster schedule does not fit this shape")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    gs.lib()
    yield
    gu.assert_clean_device()


def run_any(x, gamma, beta, G, eps, silu, variant=gs.VARIANT_AUTO, out=None):
    r = gs.gn_silu_rows_any(x, gamma, beta, G=G, eps=eps, apply_silu=silu, out=out,
                            variant=variant)
    assert r is not None, "gn_silu_rows_any rejected a supported input"
    torch.cuda.synchronize()
    return r


# N, L, C, G: channels per group 1, 3, 5, 10, 20, 30, 40, 60, 129, 255; C with
# V = C / 8 vector slots that do not divide the 512 consumer threads (and
# some that exceed a warp), ragged L, several batch entries
GENERAL = [
    (1, 4096, 320, 32), (2, 1000, 960, 32), (1, 777, 24, 8), (3, 513, 2040, 8),
    (1, 2049, 1032, 8), (2, 333, 96, 32), (1, 5000, 640, 32), (1, 300, 1280, 32),
    (1, 100, 1920, 32), (4, 77, 40, 8), (1, 1, 320, 32), (2, 3, 1920, 32), (5, 999, 480, 96),
    (1, 20000, 160, 32), (1, 3001, 1536, 1536), (160, 17, 320, 32), (1, 9999, 72, 72),
]


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("N,L,C,G", GENERAL)
def test_general_channel_counts_every_output(N, L, C, G, variant):
    skip_unless_cluster_fits(N, L, C, G, variant)
    case = wl.make_case(N, L, C, seed=N * 7919 + L * 13 + C * 3 + G, mean=0.4, std=1.6,
                        channel_offset=0.5)
    x, gamma, beta = gu.device_inputs(case)
    for silu in (True, False):
        y, mean, rstd = run_any(x, gamma, beta, G, 1e-6, silu, variant)
        y_ref, m_ref, r_ref = oracle.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6,
                                             silu)
        what = f"N={N} L={L} C={C} G={G} silu={silu} {VNAME[variant]}"
        gu.check_y(gu.bf16_to_f64(y), y_ref, what)
        gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, what)


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("N,L,C", [(1, 16384, 256), (2, 3001, 512), (1, 999, 2048), (3, 77, 8)])
def test_power_of_two_channels_match_the_pow2_entry_bitwise(N, L, C, variant):
    """For a power-of-two C both entry points run the same kernels with the
    same geometry, so every output and statistic is bitwise identical."""
    skip_unless_cluster_fits(N, L, C, 32 if C >= 32 else C, variant)
    case = wl.make_case(N, L, C, seed=L + C, mean=-0.3, std=1.2)
    x, gamma, beta = gu.device_inputs(case)
    a = run_any(x, gamma, beta, 32 if C >= 32 else C, 1e-6, True, variant)
    b = gu.run_rows_ex(x, gamma, beta, 32 if C >= 32 else C, 1e-6, True, variant)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("N,L,C", [(1, 100000, 960), (2, 30000, 320), (1, 200000, 960)])
def test_general_ring_reuse_is_race_free(N, L, C, variant):
    """Many more pieces per CTA than ring slots with a C whose slots leave
    consumer threads idle (at 366 MiB the fused kernel also deals pass 2 out
    at run time): repeated calls are bitwise identical and sampled outputs
    match the oracle."""
    case = wl.make_case(N, L, C, seed=L * 3 + C, mean=1.0, std=2.0)
    x, gamma, beta = gu.device_inputs(case)
    first = run_any(x, gamma, beta, 32, 1e-6, True, variant)
    for _ in range(6):
        again = run_any(x, gamma, beta, 32, 1e-6, True, variant)
        for u, v in zip(first, again):
            assert torch.equal(u, v), "outputs differ between identical calls"
    m_ref, _, r_ref = oracle.stats(case["x_bits"], 32, 1e-6)
    gu.check_stats(first[1].cpu().numpy(), first[2].cpu().numpy(), m_ref, r_ref, "general reuse")
    idx = np.random.default_rng(C).integers(0, N * L * C, 1 << 18)
    y_ref = oracle.apply_at(case["x_bits"], case["gamma"], case["beta"], 32, m_ref, r_ref, True, idx)
    gu.check_y(gu.bf16_to_f64(first[0].reshape(-1)[torch.from_numpy(idx).cuda()]), y_ref,
               "general reuse sampled")


def ndhwc_case(N, C, D, H, W, seed):
    """Seeded 5D input: the rows case (N, D*H*W, C) viewed as a channels_last_3d
    (N, C, D, H, W) tensor (same memory)."""
    case = wl.make_case(N, D * H * W, C, seed=seed, mean=0.2, std=1.3, channel_offset=0.3)
    x_rows, gamma, beta = gu.device_inputs(case)
    x = x_rows.view(N, D, H, W, C).permute(0, 4, 1, 2, 3)
    assert x.is_contiguous(memory_format=torch.channels_last_3d)
    return case, x, gamma, beta


@pytest.mark.parametrize("N,C,D,H,W,G", [(1, 320, 5, 16, 16, 32), (2, 128, 3, 9, 11, 32),
                                          (1, 960, 2, 8, 8, 32), (1, 24, 4, 4, 4, 8)])
def test_ndhwc_against_the_oracle(N, C, D, H, W, G):
    case, x, gamma, beta = ndhwc_case(N, C, D, H, W, seed=C + D * H * W)
    for silu in (True, False):
        y = gs.gn_silu_ndhwc(x, gamma, beta, G=G, eps=1e-6, apply_silu=silu)
        assert y is not None
        torch.cuda.synchronize()
        assert y.shape == x.shape and y.is_contiguous(memory_format=torch.channels_last_3d)
        y_ref, _, _ = oracle.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, silu)
        y_rows = y.permute(0, 2, 3, 4, 1).reshape(N, D * H * W, C)
        gu.check_y(gu.bf16_to_f64(y_rows), y_ref, f"ndhwc C={C} silu={silu}")


def test_ndhwc_against_torch_group_norm_in_float64():
    """The 5D entry against PyTorch's own GroupNorm on the same values in
    float64 on the CPU (NCDHW semantics), SiLU after it."""
    N, C, D, H, W, G = 2, 320, 3, 10, 12, 32
    _, x, gamma, beta = ndhwc_case(N, C, D, H, W, seed=77)
    y = gs.gn_silu_ndhwc(x, gamma, beta, G=G, eps=1e-6, apply_silu=True)
    torch.cuda.synchronize()
    xr = x.detach().cpu().double().contiguous()
    ref = F.silu(F.group_norm(xr, G, gamma.cpu().double(), beta.cpu().double(), eps=1e-6))
    gu.check_y(y.cpu().double().numpy(), ref.numpy(), "ndhwc vs torch")


def test_rows_any_returns_none_for_channels_not_a_multiple_of_8():
    x = torch.zeros((1, 8, 12), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(12, device="cuda")
    with pytest.warns(UserWarning):
        assert gs.gn_silu_rows_any(x, g, g, G=4) is None


def test_ndhwc_returns_none_for_non_channels_last_3d():
    x = torch.zeros((1, 320, 2, 2, 2), dtype=torch.bfloat16, device="cuda")   # NCDHW contiguous
    g = torch.ones(320, device="cuda")
    assert gs.gn_silu_ndhwc(x, g, g) is None


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("name", [w.name for w in wl.GENERAL_WORKLOADS])
def test_general_workloads_full_size(name, variant):
    """The general-channel benchmark shapes at full size, in the launch
    configuration the benchmark times: all group statistics, plus sampled
    outputs (and every channel of the first and last rows) against the
    oracle."""
    w = wl.BY_NAME[name]
    case = wl.make_inputs(w)
    x, gamma, beta = gu.device_inputs(case)
    y, mean, rstd = run_any(x, gamma, beta, w.G, w.eps, True, variant)
    m_ref, _, r_ref = oracle.stats(case["x_bits"], w.G, w.eps)
    gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, name)
    rows = w.N * w.L
    idx = np.unique(np.concatenate([np.random.default_rng(w.index).integers(0, w.elements, 1 << 20),
                                    np.arange(w.C), (rows - 1) * w.C + np.arange(w.C)]))
    y_ref = oracle.apply_at(case["x_bits"], case["gamma"], case["beta"], w.G, m_ref, r_ref, True,
                            idx)
    gu.check_y(gu.bf16_to_f64(y.reshape(-1)[torch.from_numpy(idx).cuda()]), y_ref,
               f"{name} {VNAME[variant]} sampled")
