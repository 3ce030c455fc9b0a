"""Caller-given buffers and the library's own workspaces (GPU).

Unsupported input gives None, the contract of the sglang PR #33451 page
("FLUX.2 VAE decoder fast path behind quality=high", section
"Modifications", item 1, second bullet).  A caller-given ``out`` or
``workspace`` of the wrong shape, dtype, device or layout is unsupported
input: the binding refuses it before anything is launched, so it can never
become an out-of-bounds write.  A zero-filled caller workspace serves any
number of calls in a row.  The library keeps at most eight workspaces per
device however many streams call it."""
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


def small_case(C=256, L=1000, seed=3):
    case = wl.make_case(2, L, C, seed=seed)
    return case, gu.device_inputs(case)


BAD_OUTS = {
    "short": lambda x: torch.empty((x.shape[0], x.shape[1] - 1, x.shape[2]), dtype=x.dtype, device=x.device),
    "fp32": lambda x: torch.empty(x.shape, dtype=torch.float32, device=x.device),
    "cpu": lambda x: torch.empty(x.shape, dtype=x.dtype),
    "strided": lambda x: torch.empty((x.shape[0], x.shape[2], x.shape[1]), dtype=x.dtype,
                                     device=x.device).transpose(1, 2),
}

BAD_WORKSPACES = {
    "cpu": lambda n, dev: torch.zeros(n, dtype=torch.uint8),
    "fp32": lambda n, dev: torch.zeros((n + 3) // 4, dtype=torch.float32, device=dev),
    "strided": lambda n, dev: torch.zeros(2 * n, dtype=torch.uint8, device=dev)[::2],
    "2d": lambda n, dev: torch.zeros((2, n), dtype=torch.uint8, device=dev),
}


@pytest.mark.parametrize("entry", ["gn_silu_rows_ex", "gn_silu_rows_any"])
@pytest.mark.parametrize("bad", sorted(BAD_OUTS))
def test_wrong_out_is_refused_before_launch(entry, bad):
    _, (x, gamma, beta) = small_case()
    out = BAD_OUTS[bad](x)
    torch.cuda.synchronize()
    before = gs.gn_kernel_launch_count()
    assert getattr(gs, entry)(x, gamma, beta, G=32, out=out) is None
    assert gs.gn_kernel_launch_count() == before


@pytest.mark.parametrize("entry", ["gn_silu_rows_ex", "gn_silu_rows_any"])
@pytest.mark.parametrize("bad", sorted(BAD_WORKSPACES))
def test_wrong_workspace_is_refused_before_launch(entry, bad):
    _, (x, gamma, beta) = small_case()
    N, L, C = x.shape
    ws = BAD_WORKSPACES[bad](gs.gn_silu_workspace_bytes(N, L, C, 32), x.device)
    torch.cuda.synchronize()
    before = gs.gn_kernel_launch_count()
    assert getattr(gs, entry)(x, gamma, beta, G=32, workspace=ws) is None
    assert gs.gn_kernel_launch_count() == before


def test_attention_refuses_a_host_workspace():
    S, D = 256, 512
    q = torch.zeros((S, D), dtype=torch.bfloat16, device="cuda")
    wf = torch.zeros((D, D), dtype=torch.bfloat16, device="cuda")
    bf = torch.zeros(D, dtype=torch.float32, device="cuda")
    ws = torch.zeros(gs.gn_attn_workspace_bytes(S, D), dtype=torch.uint8)
    torch.cuda.synchronize()
    before = gs.gn_kernel_launch_count()
    assert gs.attention_folded(q, q, q, wf, bf, workspace=ws) is None
    assert gs.gn_kernel_launch_count() == before


@pytest.mark.parametrize("variant", [gs.VARIANT_FUSED, gs.VARIANT_TWO_PASS], ids=["fused", "two_pass"])
@pytest.mark.parametrize("C,L", [(256, 1000), (512, 4099), (2048, 77)])
def test_caller_workspace_serves_calls_in_a_row(variant, C, L):
    case, (x, gamma, beta) = small_case(C, L, seed=C + L)
    ws = gs.new_workspace(x, 32)
    assert ws is not None and ws.numel() == gs.gn_silu_workspace_bytes(*x.shape, 32)
    y_ref, m_ref, r_ref = oracle.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True)
    for call in range(3):
        y, mean, rstd = gu.run_rows_ex(x, gamma, beta, 32, 1e-6, True, variant=variant, workspace=ws)
        gu.check_y(gu.bf16_to_f64(y), y_ref, f"caller workspace, call {call}")
        gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, f"caller workspace, call {call}")
    # the barrier words are left zero for the next call
    assert int(ws[:256].count_nonzero()) == 0


def test_library_workspaces_stay_bounded_over_many_streams():
    # scale/shift of 64 x 2048 channels: each library workspace is over 1 MiB
    N, L, C, G = 64, 8, 2048, 32
    case = wl.make_case(N, L, C, seed=17)
    x, gamma, beta = gu.device_inputs(case)
    y = torch.empty_like(x)
    need = gs.gn_silu_workspace_bytes(N, L, C, G)
    assert need > (1 << 20)

    def calls_on_new_streams(count):
        for _ in range(count):
            s = torch.cuda.Stream()
            assert gs.gn_silu_rows(x, gamma, beta, G=G, out=y, stream=s) is not None
            s.synchronize()
            del s
        assert 1 <= gs.gn_library_workspaces() <= 8

    # a first round lets the driver set up whatever per-stream state it
    # keeps for the streams PyTorch hands out (its pool is finite)
    calls_on_new_streams(100)
    assert gs.gn_release_workspaces() == gs.GN_OK
    assert gs.gn_library_workspaces() == 0
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    calls_on_new_streams(100)
    torch.cuda.synchronize()
    grown = free_before - torch.cuda.mem_get_info()[0]
    assert grown <= 8 * (need + need // 4) + (16 << 20), grown
    y_ref, _, _ = oracle.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, True)
    gu.check_y(gu.bf16_to_f64(y), y_ref, "last of 100 streams")
    assert gs.gn_release_workspaces() == gs.GN_OK
    assert gs.gn_library_workspaces() == 0
    assert torch.cuda.mem_get_info()[0] >= free_before - (16 << 20)
    # and calls allocate again afterwards
    assert gs.gn_silu_rows(x, gamma, beta, G=G, out=y) is not None
    torch.cuda.synchronize()
    assert gs.gn_library_workspaces() == 1
    assert np.isfinite(gu.bf16_to_f64(y)).all()
