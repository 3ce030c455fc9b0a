"""Failure handling on the GPU, without a fault: kernels that wait for
something nothing will ever do must give up after their bound, report
GN_ERR_KERNEL through gn_device_status and through every later call of the
C ABI (which then launches nothing), and leave the context usable (the next
ordinary call after clearing the status is correct)."""
import ctypes
import time

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
    assert gs.gn_device_status(False) == gs.GN_OK


def raw_rows(x, gamma, beta, y, stream=None):
    N, L, C = x.shape
    return gs.raw_gn_silu_rows(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), y.data_ptr(), N, L, C, 32,
                               1e-6, 1, stream=stream or 0)


@pytest.mark.parametrize("mode", [0, 1], ids=["mbarrier_phase", "barrier_count"])
def test_unsatisfiable_wait_expires_and_reports(mode):
    blocks = 4
    case = wl.make_case(1, 4096, 128, 3)
    x, gamma, beta = gu.device_inputs(case)
    torch.cuda.synchronize()
    done = torch.zeros(blocks, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    y_early = torch.full_like(x, 7.0)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = gs.lib().gn_selftest_bounded_wait(mode, 300, ctypes.c_void_p(done.data_ptr()), blocks,
                                           ctypes.c_void_p(stream))
    assert rc == gs.GN_OK
    # enqueued behind the expiring wait, before it has expired: the call is
    # accepted, and its kernels find the status set and return without writing
    assert raw_rows(x, gamma, beta, y_early, stream) == gs.GN_OK
    assert gs.gn_device_status(False) == gs.GN_ERR_KERNEL
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0
    assert done.tolist() == [1] * blocks          # every CTA gave up and returned
    assert torch.all(y_early == 7.0)
    # now that the host sees the status, every entry point refuses to launch
    y = torch.full_like(x, 7.0)
    before = gs.gn_kernel_launch_count()
    assert raw_rows(x, gamma, beta, y) == gs.GN_ERR_KERNEL
    N, L, C = x.shape
    assert gs.raw_gn_silu_rows_ex(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), y.data_ptr(), N, L, C, 32,
                                  1e-6, 1, variant=gs.VARIANT_TWO_PASS) == gs.GN_ERR_KERNEL
    r = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(256, dtype=torch.bfloat16, device="cuda")
    assert gs.raw_gn_residual_gate_add(r.data_ptr(), r.data_ptr(), g.data_ptr(), r.data_ptr(), 8, 256,
                                       0) == gs.GN_ERR_KERNEL
    with pytest.raises(gs.GnError) as err:        # the tensor binding raises: not an unsupported input
        gs.gn_silu_rows(x, gamma, beta, G=32, out=y)
    assert err.value.status == gs.GN_ERR_KERNEL
    torch.cuda.synchronize()
    assert gs.gn_kernel_launch_count() == before
    assert torch.all(y == 7.0)
    # clearing restores normal operation in the same context
    assert gs.gn_device_status(True) == gs.GN_ERR_KERNEL
    assert gs.gn_device_status(False) == gs.GN_OK
    y2 = torch.full_like(x, 7.0)
    assert raw_rows(x, gamma, beta, y2) == gs.GN_OK
    torch.cuda.synchronize()
    y_ref, _, _ = oracle.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True)
    gu.check_y(gu.bf16_to_f64(y2), y_ref, "after clearing")
    assert gs.gn_device_status(False) == gs.GN_OK


def test_selftest_rejects_bad_arguments():
    assert gs.lib().gn_selftest_bounded_wait(2, 10, None, 1, None) == gs.GN_ERR_SHAPE
    assert gs.lib().gn_selftest_bounded_wait(0, 10, None, 1, None) == gs.GN_ERR_NULL
