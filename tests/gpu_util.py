"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

from channels_last_groupnorm_gb300 import gnsilu as gs

# Acceptance bounds (bf16 output; fp32 statistics):
#   |y_gpu - y_ref| <= Y_ATOL + Y_RTOL * |y_ref|   elementwise
#   |rstd_gpu - rstd_ref| <= STAT_RTOL * rstd_ref
#   |mean_gpu - mean_ref| <= STAT_RTOL * max(|mean_ref|, sigma_ref), sigma_ref = 1 / rstd_ref
Y_ATOL = 1e-2
Y_RTOL = 8e-3
STAT_RTOL = 1e-5


def device_inputs(case: dict, device: str = "cuda"):
    x = torch.from_numpy(case["x_bits"].view(np.int16)).to(device).view(torch.bfloat16)
    gamma = torch.from_numpy(case["gamma"]).to(device)
    beta = torch.from_numpy(case["beta"]).to(device)
    return x.contiguous(), gamma.contiguous(), beta.contiguous()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_rows_ex(x, gamma, beta, G, eps, silu, variant=gs.VARIANT_AUTO, out=None, workspace=None,
                stream=None):
    r = gs.gn_silu_rows_ex(x, gamma, beta, G=G, eps=eps, apply_silu=silu, out=out,
                           variant=variant, workspace=workspace, stream=stream)
    assert r is not None, "the CUDA path rejected a supported input"
    torch.cuda.synchronize()
    return r


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    err = np.abs(y_gpu - y_ref)
    bound = Y_ATOL + Y_RTOL * np.abs(y_ref)
    bad = ~(err <= bound)
    if bad.any():
        k = int(np.flatnonzero(bad.reshape(-1))[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs out of tolerance; first at flat {k}: "
            f"gpu {y_gpu.reshape(-1)[k]!r} ref {y_ref.reshape(-1)[k]!r}; "
            f"max err {float(err.max()):.3e}")


def check_stats(mean_gpu, rstd_gpu, mean_ref, rstd_ref, what: str = ""):
    mean_gpu = np.asarray(mean_gpu, np.float64)
    rstd_gpu = np.asarray(rstd_gpu, np.float64)
    rel_r = np.abs(rstd_gpu - rstd_ref) / rstd_ref
    assert np.all(rel_r <= STAT_RTOL), f"{what}: rstd rel err {rel_r.max():.3e}"
    scale = np.maximum(np.abs(mean_ref), 1.0 / rstd_ref)
    rel_m = np.abs(mean_gpu - mean_ref) / scale
    assert np.all(rel_m <= STAT_RTOL), f"{what}: mean rel err {rel_m.max():.3e}"


def assert_clean_device():
    assert gs.gn_device_status(False) == gs.GN_OK, "a kernel gave up a bounded wait"
