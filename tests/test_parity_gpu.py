"""CUDA path vs the fp64 oracle on the same seeded inputs (GPU).

Elementwise on every output for the shapes the oracle finishes in seconds
(including ragged tails, odd batch counts and every supported C), and on
sampled outputs plus all group statistics at the full benchmark sizes, for
every kernel schedule (the cluster schedule wherever it fits the shape)."""
import numpy as np
import pytest
import torch

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

VARIANTS = [gs.VARIANT_FUSED, gs.VARIANT_TWO_PASS]
ALL_VARIANTS = VARIANTS + [gs.VARIANT_CLUSTER]
VNAME = {gs.VARIANT_FUSED: "fused", gs.VARIANT_TWO_PASS: "two_pass", gs.VARIANT_AUTO: "auto",
         gs.VARIANT_CLUSTER: "cluster"}


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    gs.lib()
    yield
    gu.assert_clean_device()


def fits_cluster(N, L, C, G):
    """The cluster schedule takes this shape (its slices fit the clusters'
    shared memory); the explicit variant is refused otherwise."""
    return gs.gn_silu_pick_variant(N, L, C, G) == gs.VARIANT_CLUSTER or _cluster_accepts(N, L, C, G)


def _cluster_accepts(N, L, C, G):
    x = torch.zeros((N, L, C), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(C, device="cuda")
    rc = gs.raw_gn_silu_rows_ex(x.data_ptr(), g.data_ptr(), g.data_ptr(), x.data_ptr(), N, L, C, G, 1e-6, 1,
                                variant=gs.VARIANT_CLUSTER)
    torch.cuda.synchronize()
    assert rc in (gs.GN_OK, gs.GN_ERR_VARIANT), gs.status_string(rc)
    return rc == gs.GN_OK


def full_check(case, G, eps, silu, variant, what):
    x, gamma, beta = gu.device_inputs(case)
    if variant == gs.VARIANT_CLUSTER and not fits_cluster(*x.shape, G):
        pytest.skip("the cluster schedule does not fit this shape")
    y, mean, rstd = gu.run_rows_ex(x, gamma, beta, G, eps, silu, variant)
    y_ref, m_ref, r_ref = oracle.forward(case["x_bits"], case["gamma"], case["beta"], G, eps, silu)
    gu.check_y(gu.bf16_to_f64(y), y_ref, what)
    gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, what)
    return y


# ---------------------------------------------------------------------------
# the benchmark workloads
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("index", [0, 1])
def test_small_workloads_every_output(index, variant):
    w = wl.WORKLOADS[index]
    case = wl.make_inputs(w)
    full_check(case, w.G, w.eps, True, variant, f"{w.name} {VNAME[variant]}")


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("silu", [True, False], ids=["silu", "nosilu"])
def test_offset_stress_every_output(silu, variant):
    # the cluster schedule takes this 64 MiB tensor in several rounds of clusters
    w = wl.WORKLOADS[2]
    case = wl.make_inputs(w)
    full_check(case, w.G, w.eps, silu, variant, f"{w.name} silu={silu} {VNAME[variant]}")


def sampled_indices(w, count, seed):
    rng = np.random.default_rng(seed)
    total = w.elements
    rows = w.N * w.L
    # random outputs, plus every channel of the first and last rows of the tensor
    head = np.arange(w.C)
    tail = (rows - 1) * w.C + np.arange(w.C)
    return np.unique(np.concatenate([rng.integers(0, total, count), head, tail]))


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("index", [3, 4, 5])
def test_large_workloads_sampled(index, variant):
    w = wl.WORKLOADS[index]
    case = wl.make_inputs(w)
    x, gamma, beta = gu.device_inputs(case)
    for silu in w.silu_modes:
        y, mean, rstd = gu.run_rows_ex(x, gamma, beta, w.G, w.eps, silu, variant)
        m_ref, _, r_ref = oracle.stats(case["x_bits"], w.G, w.eps)
        gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, w.name)
        idx = sampled_indices(w, 1 << 20, 7 + index)
        y_ref = oracle.apply_at(case["x_bits"], case["gamma"], case["beta"], w.G, m_ref, r_ref,
                                silu, idx)
        y_gpu = gu.bf16_to_f64(y.reshape(-1)[torch.from_numpy(idx).cuda()])
        gu.check_y(y_gpu, y_ref, f"{w.name} {VNAME[variant]} sampled")
        del y


@pytest.mark.parametrize("N,L,C,G", [(1, 262144, 512, 64), (1, 1048576, 256, 128)])
def test_dealt_out_pass2_with_the_grid_wide_finalize(N, L, C, G):
    """Large single-entry tensors with many groups: the fused kernel merges
    the records with its grid-wide finalize (a second barrier) and deals
    pass 2 out at run time; sampled outputs and every statistic against the
    oracle."""
    case = wl.make_case(N, L, C, seed=L + G, mean=0.5, std=1.5)
    x, gamma, beta = gu.device_inputs(case)
    y, mean, rstd = gu.run_rows_ex(x, gamma, beta, G, 1e-6, True, gs.VARIANT_FUSED)
    m_ref, _, r_ref = oracle.stats(case["x_bits"], G, 1e-6)
    gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, f"G={G}")
    idx = np.random.default_rng(G).integers(0, N * L * C, 1 << 20)
    y_ref = oracle.apply_at(case["x_bits"], case["gamma"], case["beta"], G, m_ref, r_ref, True, idx)
    gu.check_y(gu.bf16_to_f64(y.reshape(-1)[torch.from_numpy(idx).cuda()]), y_ref, f"G={G} sampled")


# ---------------------------------------------------------------------------
# edge cases: every C, ragged and tiny L, several batch entries, G extremes
# ---------------------------------------------------------------------------
EDGE = [
    # N, L, C, G
    (1, 1, 8, 8), (1, 1, 32, 32), (1, 2, 64, 32), (1, 3, 128, 32), (2, 7, 256, 32),
    (3, 5, 2048, 32), (1, 4099, 8, 1), (1, 4099, 16, 2), (2, 1000, 32, 32), (1, 777, 64, 4),
    (1, 12345, 128, 32), (3, 3001, 256, 16), (2, 2049, 512, 32), (1, 999, 1024, 32),
    (1, 1025, 2048, 32), (2, 513, 2048, 2048), (1, 10000, 512, 1), (5, 300, 512, 512),
    (4, 1, 1024, 32), (1, 65537, 64, 32), (7, 97, 128, 8), (160, 33, 64, 32), (400, 9, 32, 32),
]


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("N,L,C,G", EDGE)
def test_edge_shapes(N, L, C, G, variant):
    case = wl.make_case(N, L, C, seed=N * 1000003 + L * 31 + C + G, mean=0.5, std=1.7)
    for silu in (True, False):
        full_check(case, G, 1e-6, silu, variant, f"N={N} L={L} C={C} G={G} {VNAME[variant]}")


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
def test_constant_input(variant):
    """var = 0: the mean is the constant exactly, rstd = 1/sqrt(eps) and
    y = beta (SiLU off)."""
    case = wl.make_case(2, 3000, 256, 5, mean=4.0, kind="constant")
    x, gamma, beta = gu.device_inputs(case)
    y, mean, rstd = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, False, variant)
    assert torch.all(mean == 4.0)
    np.testing.assert_allclose(rstd.cpu().numpy(), 1000.0, rtol=1e-5)
    gu.check_y(gu.bf16_to_f64(y), np.broadcast_to(case["beta"].astype(np.float64), y.shape),
               "constant")


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
def test_in_place(variant):
    case = wl.make_case(2, 5000, 512, 11, std=2.0)
    x, gamma, beta = gu.device_inputs(case)
    y_ref, _, _ = oracle.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True)
    gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant, out=x)
    gu.check_y(gu.bf16_to_f64(x), y_ref, "in place")


@pytest.mark.parametrize("variant", ALL_VARIANTS, ids=lambda v: VNAME[v])
def test_no_writes_outside_y(variant):
    """y sits inside a larger poisoned buffer; only its own bytes change."""
    N, L, C = 1, 3333, 256
    case = wl.make_case(N, L, C, 13)
    x, gamma, beta = gu.device_inputs(case)
    pad = 4096
    buf = torch.full((pad + N * L * C + pad,), -12345.0, dtype=torch.bfloat16, device="cuda")
    y = buf[pad:pad + N * L * C].view(N, L, C)
    gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant, out=y)
    assert torch.all(buf[:pad] == -12345.0) and torch.all(buf[pad + N * L * C:] == -12345.0)
    y_ref, _, _ = oracle.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True)
    gu.check_y(gu.bf16_to_f64(y), y_ref, "guarded")


def test_variants_agree_closely():
    case = wl.make_case(1, 20000, 512, 17, mean=-1.0, std=3.0)
    x, gamma, beta = gu.device_inputs(case)
    a = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, gs.VARIANT_FUSED)
    b = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, gs.VARIANT_TWO_PASS)
    np.testing.assert_allclose(a[1].cpu().numpy(), b[1].cpu().numpy(), rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(a[2].cpu().numpy(), b[2].cpu().numpy(), rtol=2e-6)
    diff = (a[0].float() - b[0].float()).abs().max().item()
    assert diff <= 0.02


def test_repeated_calls_are_deterministic():
    case = wl.make_case(1, 50000, 256, 19)
    x, gamma, beta = gu.device_inputs(case)
    for variant in ALL_VARIANTS:
        first = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant)
        for _ in range(3):
            again = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant)
            assert torch.equal(first[0], again[0])
            assert torch.equal(first[1], again[1]) and torch.equal(first[2], again[2])


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAME[v])
@pytest.mark.parametrize("N,L,C", [(1, 131072, 512), (2, 40000, 256), (1, 300000, 64)])
def test_ring_reuse_is_race_free(N, L, C, variant):
    """Shapes with many more pieces per CTA than ring slots, so every slot is
    refilled many times in both passes.  The result is a deterministic
    function of the input: every repetition must be bitwise identical, and
    sampled outputs must match the oracle."""
    case = wl.make_case(N, L, C, seed=L + C, mean=1.0, std=2.0)
    x, gamma, beta = gu.device_inputs(case)
    first = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant)
    for _ in range(12):
        again = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant)
        assert torch.equal(first[0], again[0]), "outputs differ between identical calls"
        assert torch.equal(first[1], again[1]) and torch.equal(first[2], again[2])
    m_ref, _, r_ref = oracle.stats(case["x_bits"], 32, 1e-6)
    gu.check_stats(first[1].cpu().numpy(), first[2].cpu().numpy(), m_ref, r_ref, "ring reuse")
    idx = np.random.default_rng(L).integers(0, N * L * C, 1 << 18)
    y_ref = oracle.apply_at(case["x_bits"], case["gamma"], case["beta"], 32, m_ref, r_ref, True, idx)
    gu.check_y(gu.bf16_to_f64(first[0].reshape(-1)[torch.from_numpy(idx).cuda()]), y_ref,
               "ring reuse sampled")


_STATIC_PASS2_CHILD = """
import sys
import numpy as np
import torch
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu
N, L, C = (int(v) for v in sys.argv[1:4])
case = wl.make_case(N, L, C, seed=L + C, mean=1.0, std=2.0)
x, gamma, beta = gu.device_inputs(case)
y, mean, rstd = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, gs.VARIANT_FUSED)
np.save(sys.argv[4], y.view(torch.int16).cpu().numpy())
np.save(sys.argv[5], torch.stack([mean, rstd]).cpu().numpy())
"""


@pytest.mark.parametrize("N,L,C", [(1, 262144, 512), (1, 524288, 256)])
def test_dynamic_pass2_matches_the_static_assignment_bitwise(N, L, C, tmp_path):
    """For large single-entry tensors the fused kernel deals the pieces of
    pass 2 out at run time.  Which CTA applies a piece must not change a bit
    of the output: compare with the static assignment (GN_DYNAMIC_PASS2=0,
    read once per process, so in a child process)."""
    import os
    import subprocess
    import sys
    case = wl.make_case(N, L, C, seed=L + C, mean=1.0, std=2.0)
    x, gamma, beta = gu.device_inputs(case)
    y, mean, rstd = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, gs.VARIANT_FUSED)
    env = dict(os.environ, GN_DYNAMIC_PASS2="0")
    yf, sf = tmp_path / "y.npy", tmp_path / "s.npy"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([sys.executable, "-c", _STATIC_PASS2_CHILD, str(N), str(L), str(C), str(yf), str(sf)],
                   env=env, cwd=root, check=True, timeout=600)
    assert np.array_equal(np.load(yf), y.view(torch.int16).cpu().numpy()), "outputs differ from the static assignment"
    assert np.array_equal(np.load(sf), torch.stack([mean, rstd]).cpu().numpy())


# ---------------------------------------------------------------------------
# the cluster schedule: where the automatic choice takes it, and where not
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,L,C", [(1, 4096, 128), (1, 1024, 512), (1, 4096, 512), (4, 1024, 512),
                                   (1, 16384, 512), (1, 16384, 128), (1, 16384, 256)])
def test_small_tensors_take_the_cluster_schedule(N, L, C):
    assert gs.gn_silu_pick_variant(N, L, C, 32) == gs.VARIANT_CLUSTER


@pytest.mark.parametrize("N,L,C", [(1, 65536, 128)])
def test_automatic_choice_leaves_narrow_slices_of_larger_tensors_to_the_fused_schedule(N, L, C):
    assert gs.gn_silu_pick_variant(N, L, C, 32) == gs.VARIANT_FUSED
    assert fits_cluster(N, L, C, 32)


def test_automatic_choice_leaves_the_offset_stress_shape_to_the_fused_schedule():
    w = wl.WORKLOADS[2]
    assert gs.gn_silu_pick_variant(w.N, w.L, w.C, w.G) == gs.VARIANT_FUSED
    assert fits_cluster(w.N, w.L, w.C, w.G)


@pytest.mark.parametrize("index", [3, 4, 5])
def test_large_workloads_do_not_fit_the_cluster_schedule(index):
    w = wl.WORKLOADS[index]
    assert gs.gn_silu_pick_variant(w.N, w.L, w.C, w.G) != gs.VARIANT_CLUSTER
    x = torch.empty((w.N, w.L, w.C), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(w.C, device="cuda")
    before = gs.gn_kernel_launch_count()
    rc = gs.raw_gn_silu_rows_ex(x.data_ptr(), g.data_ptr(), g.data_ptr(), x.data_ptr(), w.N, w.L, w.C, w.G,
                                w.eps, 1, variant=gs.VARIANT_CLUSTER)
    assert rc == gs.GN_ERR_VARIANT
    assert gs.gn_kernel_launch_count() == before


@pytest.mark.parametrize("N,L,C,G", [(1, 4096, 128, 32), (1, 16384, 512, 32), (3, 777, 2048, 32),
                                     (160, 33, 64, 32), (2, 513, 2048, 2048)])
def test_cluster_schedule_matches_two_pass_closely(N, L, C, G):
    """Same statistics as the two-pass schedule to fp32 rounding, outputs
    within one bf16 rounding step."""
    case = wl.make_case(N, L, C, seed=N + L + C + G, mean=-0.7, std=2.5)
    x, gamma, beta = gu.device_inputs(case)
    a = gu.run_rows_ex(x, gamma, beta, G, 1e-6, True, gs.VARIANT_CLUSTER)
    b = gu.run_rows_ex(x, gamma, beta, G, 1e-6, True, gs.VARIANT_TWO_PASS)
    np.testing.assert_allclose(a[1].cpu().numpy(), b[1].cpu().numpy(), rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(a[2].cpu().numpy(), b[2].cpu().numpy(), rtol=2e-6)
    assert (a[0].float() - b[0].float()).abs().max().item() <= 0.02
