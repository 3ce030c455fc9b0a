"""gn_silu_rows_static: the entry point for callers that cannot allocate
device memory (code inside a CUDA graph capture, plug-ins whose host owns all
device memory, paths that cannot risk an allocator's synchronisation).

It takes its scratch from a fixed array inside the library instead of a
workspace.  Here it is called through the C ABI and its outputs are compared
with those of the ordinary entry point (gn_silu_rows_ex), on two calls in a
row so that the second call sees the scratch the first one left behind.

This file is collected last on purpose; it passes alone in a fresh process
and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

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
def test_static_matches_ordinary_entry_point_twice(shape, silu):
    N, L, C, G = shape
    case = wl.make_case(N, L, C, seed=N * 7 + L + C, mean=0.3, std=1.4)
    x, gamma, beta = gu.device_inputs(case)
    stream = torch.cuda.current_stream()
    y_ref, m_ref, r_ref = gu.run_rows_ex(x, gamma, beta, G, 1e-6, silu)
    y_ref = gu.bf16_to_f64(y_ref)
    m_ref = m_ref.cpu().numpy().astype(np.float64)
    r_ref = r_ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        mean = torch.full((N, G), float("nan"), device=x.device)
        rstd = torch.full((N, G), float("nan"), device=x.device)
        rc = call_static(x, gamma, beta, y, mean, rstd, G, 1e-6, silu, stream)
        assert rc == gs.GN_OK, gs.status_string(rc)
        torch.cuda.synchronize()
        gu.check_y(gu.bf16_to_f64(y), y_ref, f"static call {call}")
        gu.check_stats(mean.cpu().numpy(), rstd.cpu().numpy(), m_ref, r_ref,
                       f"static call {call}")
    assert gs.gn_device_status(False) == gs.GN_OK


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
