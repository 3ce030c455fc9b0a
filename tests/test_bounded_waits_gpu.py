"""Failure handling on the GPU, without a fault: kernels that wait for
something nothing will ever do must give up after their bound, report
GN_ERR_KERNEL through gn_device_status, and leave the context usable (the
next ordinary call after clearing the status is correct)."""
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


@pytest.mark.parametrize("mode", [0, 1], ids=["mbarrier_phase", "barrier_count"])
def test_unsatisfiable_wait_expires_and_reports(mode):
    blocks = 4
    done = torch.zeros(blocks, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    rc = gs.lib().gn_selftest_bounded_wait(mode, 50, ctypes.c_void_p(done.data_ptr()), blocks, None)
    assert rc == gs.GN_OK
    assert gs.gn_device_status(False) == gs.GN_ERR_KERNEL
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0
    assert done.tolist() == [1] * blocks          # every CTA gave up and returned
    # while the status is set, launched kernels return without writing
    case = wl.make_case(1, 4096, 128, 3)
    x, gamma, beta = gu.device_inputs(case)
    y = torch.full_like(x, 7.0)
    r = gs.gn_silu_rows(x, gamma, beta, G=32, out=y)
    torch.cuda.synchronize()
    assert r is not None and torch.all(y == 7.0)
    # clearing restores normal operation in the same context
    assert gs.gn_device_status(True) == gs.GN_ERR_KERNEL
    assert gs.gn_device_status(False) == gs.GN_OK
    y2 = gs.gn_silu_rows(x, gamma, beta, G=32)
    torch.cuda.synchronize()
    y_ref, _, _ = oracle.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, True)
    gu.check_y(gu.bf16_to_f64(y2), y_ref, "after clearing")
    assert gs.gn_device_status(False) == gs.GN_OK


def test_selftest_rejects_bad_arguments():
    assert gs.lib().gn_selftest_bounded_wait(2, 10, None, 1, None) == gs.GN_ERR_SHAPE
    assert gs.lib().gn_selftest_bounded_wait(0, 10, None, 1, None) == gs.GN_ERR_NULL
