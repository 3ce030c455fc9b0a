"""Residual-gate update on the GPU (gn_residual_gate_add) against the
oracle, bit for bit: y = residual + gate * update in bf16 / fp16 with the
two roundings of the eager evaluation (the prhub digest of sglang PR #33823,
FLUX.2 bit-exact residual-gate fusion, section "Implementation breakdown",
items 3-4: half dtypes only, atol = 0, rtol = 0)."""
import numpy as np
import pytest
import torch

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from channels_last_groupnorm_gb300 import workloads as wl
from tests import gpu_util as gu
from tests import rga_pins as rp

pytestmark = pytest.mark.gpu

FMTS = ["bf16", "fp16"]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    gs.lib()
    yield
    gu.assert_clean_device()


def run(r, u, g, out=None):
    y = gs.residual_gate_add(r, u, g, out=out)
    assert y is not None, "the CUDA path rejected a supported input"
    torch.cuda.synchronize()
    return y


def check_against_oracle(r, u, g, y, fmt, what):
    D = r.shape[-1]
    want = oracle.rga().forward(rp.bits(r.cpu().reshape(-1, D)), rp.bits(u.cpu().reshape(-1, D)),
                                rp.bits(g.cpu().reshape(-1)), fmt)
    got = rp.bits(y.cpu().reshape(-1, D))
    ok = rp.same(got, want, fmt)
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outputs differ from the oracle"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 512, 3072), (3, 77, 264), (1, 1, 8), (2, 1000, 3072), (5, 4099, 16)])
def test_matches_oracle_bit_for_bit(shape, fmt):
    r = rp.wide_values(shape, fmt, sum(shape)).cuda()
    u = rp.wide_values(shape, fmt, sum(shape) + 1).cuda()
    g = rp.wide_values((shape[-1],), fmt, sum(shape) + 2).cuda()
    y = run(r, u, g)
    check_against_oracle(r, u, g, y, fmt, f"{shape} {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_flux2_dev_shape_matches_eager_and_oracle(fmt):
    """The FLUX.2-dev 1024^2 shape (1, 4608, 6144) the page adds to its
    bit-exactness cases, at full size, in the configuration the benchmark
    times, against PyTorch's own eager kernels and the oracle."""
    w = wl.RGA_BY_NAME["rga_flux2_dev_4608x6144"]
    r, u, g = (t.to(rp.DT[fmt]).cuda() for t in wl.make_rga_inputs(w))
    y = run(r, u, g)
    eager = r + g * u
    torch.cuda.synchronize()
    ok = rp.same(rp.bits(y.cpu()).reshape(-1), rp.bits(eager.cpu()).reshape(-1), fmt)
    assert ok.all(), f"{int((~ok).sum())} outputs differ from eager"
    check_against_oracle(r, u, g, y, fmt, f"flux2 dev {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bit_pattern_as_update(fmt):
    u = torch.from_numpy(np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.int16)).view(
        rp.DT[fmt]).reshape(256, 256).cuda()
    for rv, gv in ((0.75, 1.5), (-3.0, 0.1), (1e-3, -7.0), (0.0, 1.0)):
        r = torch.full((256, 256), rv, dtype=rp.DT[fmt], device="cuda")
        g = torch.full((256,), gv, dtype=rp.DT[fmt], device="cuda")
        y = run(r, u, g)
        check_against_oracle(r, u, g, y, fmt, f"exhaustive r={rv} g={gv} {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_in_place_on_residual_and_on_update(fmt):
    shape = (4, 333, 192)
    r = rp.wide_values(shape, fmt, 1).cuda()
    u = rp.wide_values(shape, fmt, 2).cuda()
    g = rp.wide_values((192,), fmt, 3).cuda()
    want = run(r, u, g).clone()
    r2 = r.clone()
    assert run(r2, u, g, out=r2) is r2
    u2 = u.clone()
    assert run(r, u2, g, out=u2) is u2
    for t in (r2, u2):
        ok = rp.same(rp.bits(t.cpu()).reshape(-1), rp.bits(want.cpu()).reshape(-1), fmt)
        assert ok.all()


def test_no_writes_outside_out():
    shape = (3, 50, 64)
    r = rp.wide_values(shape, "bf16", 4).cuda()
    u = rp.wide_values(shape, "bf16", 5).cuda()
    g = rp.wide_values((64,), "bf16", 6).cuda()
    n = r.numel()
    buf = torch.full((4096 + n + 4096,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[4096:4096 + n].view(shape)
    run(r, u, g, out=out)
    assert torch.all(buf[:4096] == -7.0) and torch.all(buf[4096 + n:] == -7.0)
    check_against_oracle(r, u, g, out, "bf16", "guarded")


def test_unsupported_inputs_return_none():
    r = torch.randn(2, 8, 64, device="cuda")
    g = torch.randn(64, device="cuda")
    assert gs.residual_gate_add(r, r.clone(), g) is None                       # fp32: eager rounds differently
    rb, gb = r.bfloat16(), g.bfloat16()
    assert gs.residual_gate_add(rb, rb.clone(), gb.reshape(1, 1, 64)) is not None   # [1, 1, D] gate is fine
    assert gs.residual_gate_add(rb, rb.clone(), torch.randn(2, 1, 64, device="cuda").bfloat16()) is None
    assert gs.residual_gate_add(rb, rb.clone().half(), gb) is None             # mixed dtypes
    assert gs.residual_gate_add(rb.transpose(0, 1), rb.transpose(0, 1).clone(), gb) is None   # not contiguous
    with pytest.warns(UserWarning):
        r12 = torch.zeros(2, 12, dtype=torch.bfloat16, device="cuda")
        assert gs.residual_gate_add(r12, r12.clone(), torch.ones(12, dtype=torch.bfloat16, device="cuda")) is None
    torch.cuda.synchronize()
