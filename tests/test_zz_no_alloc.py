"""gn_silu_rows_static: the entry point for callers that cannot allocate
device memory -- a plug-in whose host framework owns all device memory and
forbids allocations behind its back, a latency-critical path that cannot
afford an allocation's device-wide synchronisation, a process under a fixed
device-memory budget.

It takes its scratch from a fixed array inside the library instead of a
workspace.  Here it is called through the C ABI and its outputs are compared
with the fp64 oracle and with those of the ordinary entry point
(gn_silu_rows_ex), on two calls in a row so that the second call sees the
scratch the first one left behind; and a call on a stream the library has
not seen before is checked to allocate nothing.

This file is collected last on purpose; it passes alone in a fresh process
and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20   # GN_STATIC_SCRATCH_BYTES in include/gnsilu.h


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    return gs.lib()


def call_static(x, gamma, beta, y, mean, rstd, G, eps, silu, stream):
    N, L, C = x.shape
    return gs.lib().gn_silu_rows_static(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(gamma.data_ptr()),
        ctypes.c_void_p(beta.data_ptr()), ctypes.c_void_p(y.data_ptr()), N, L, C, G,
        ctypes.c_float(eps), int(silu), ctypes.c_void_p(mean.data_ptr()),
        ctypes.c_void_p(rstd.data_ptr()), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("shape,silu", [((1, 16384, 512, 32), True), ((2, 3001, 256, 32), False),
                                        ((3, 777, 2048, 32), True)])
def test_static_matches_oracle_and_ordinary_entry_point_twice(shape, silu):
    N, L, C, G = shape
    case = wl.make_case(N, L, C, seed=N * 7 + L + C, mean=0.3, std=1.4)
    x, gamma, beta = gu.device_inputs(case)
    stream = torch.cuda.current_stream()
    y_orc, m_orc, r_orc = oracle.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, silu)
    y_ex, m_ex, r_ex = gu.run_rows_ex(x, gamma, beta, G, 1e-6, silu)
    y_ex = gu.bf16_to_f64(y_ex)
    m_ex = m_ex.cpu().numpy().astype(np.float64)
    r_ex = r_ex.cpu().numpy().astype(np.float64)
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        mean = torch.full((N, G), float("nan"), device=x.device)
        rstd = torch.full((N, G), float("nan"), device=x.device)
        rc = call_static(x, gamma, beta, y, mean, rstd, G, 1e-6, silu, stream)
        assert rc == gs.GN_OK, gs.status_string(rc)
        torch.cuda.synchronize()
        y_np = gu.bf16_to_f64(y)
        m_np, r_np = mean.cpu().numpy(), rstd.cpu().numpy()
        gu.check_y(y_np, y_orc, f"static call {call} against the oracle")
        gu.check_stats(m_np, r_np, m_orc, r_orc, f"static call {call} against the oracle")
        gu.check_y(y_np, y_ex, f"static call {call} against gn_silu_rows_ex")
        gu.check_stats(m_np, r_np, m_ex, r_ex, f"static call {call} against gn_silu_rows_ex")
    assert gs.gn_device_status(False) == gs.GN_OK


def test_static_call_on_a_new_stream_allocates_nothing():
    # scale/shift of 128 x 2048 channels: a library workspace for this shape
    # would take more than 2 MiB of device memory
    N, L, C, G = 128, 8, 2048, 32
    need = gs.gn_silu_workspace_bytes(N, L, C, G)
    assert 2 << 20 < need <= STATIC_SCRATCH_BYTES
    case = wl.make_case(N, L, C, seed=41)
    x, gamma, beta = gu.device_inputs(case)
    y = torch.empty_like(x)
    mean = torch.empty((N, G), device=x.device)
    rstd = torch.empty((N, G), device=x.device)
    # first call of the library on this device from this test: sets the device up
    assert call_static(x, gamma, beta, y, mean, rstd, G, 1e-6, True, torch.cuda.current_stream()) == gs.GN_OK
    torch.cuda.synchronize()
    fresh = torch.cuda.Stream()
    workspaces = gs.gn_library_workspaces()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        assert call_static(x, gamma, beta, y, mean, rstd, G, 1e-6, True, fresh) == gs.GN_OK
    fresh.synchronize()
    assert gs.gn_library_workspaces() == workspaces
    assert abs(torch.cuda.mem_get_info()[0] - free_before) < (1 << 20)
    y_ref, m_ref, r_ref = oracle.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, True)
    gu.check_y(gu.bf16_to_f64(y), y_ref, "static call on a new stream")
    gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref, "static call on a new stream")


def test_static_refuses_shapes_beyond_its_scratch():
    N, L, C, G = 1024, 16, 2048, 32       # 64 MiB of x; scale/shift alone need 16 MiB
    assert gs.gn_silu_workspace_bytes(N, L, C, G) > STATIC_SCRATCH_BYTES
    x = torch.zeros((N, L, C), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(C, device="cuda")
    y = torch.empty_like(x)
    mean = torch.empty((N, G), device="cuda")
    rstd = torch.empty((N, G), device="cuda")
    before = gs.gn_kernel_launch_count()
    rc = call_static(x, g, g, y, mean, rstd, G, 1e-6, True, torch.cuda.current_stream())
    assert rc == gs.GN_ERR_WORKSPACE
    assert gs.gn_kernel_launch_count() == before


def test_static_rejects_unsupported_input_like_the_ordinary_entry_point():
    x = torch.zeros((1, 8, 24), dtype=torch.bfloat16, device="cuda")   # C = 24: not a power of two
    g = torch.ones(24, device="cuda")
    y = torch.empty_like(x)
    m = torch.empty((1, 8), device="cuda")
    rc = call_static(x, g, g, y, m, m.clone(), 8, 1e-6, True, torch.cuda.current_stream())
    assert rc == gs.GN_ERR_CHANNELS
