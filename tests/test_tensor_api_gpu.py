"""The PyTorch-facing entry points on CUDA tensors (GPU).

A channels_last tensor is a pure permutation of the NCHW one, so the 4D
entry on a channels_last input must agree with PyTorch's own GroupNorm (+
SiLU) on the NCHW tensor in float64 (the layout swap of the sglang PR #33451
page, "FLUX.2 VAE decoder fast path behind quality=high", section
"Modifications", item 2, is "pure permutations").  Unsupported inputs give
None (same section, item 1, second bullet): not channels_last, grad
enabled, wrong dtype, non-power-of-two C, C > 2048."""
import pytest
import torch
import torch.nn.functional as F

from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
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


def nchw_case(N, C, H, W, seed):
    gen = torch.Generator().manual_seed(seed)
    x = (torch.randn(N, C, H, W, generator=gen) * 1.5 + 0.3).to(torch.bfloat16)
    gamma = torch.rand(C, generator=gen) + 0.5
    beta = torch.randn(C, generator=gen) * 0.1
    return x, gamma, beta


def torch_ref(x_nchw, gamma, beta, G, eps, silu):
    z = F.group_norm(x_nchw.double(), G, gamma.double(), beta.double(), eps=eps)
    return F.silu(z) if silu else z


@pytest.mark.parametrize("N,C,H,W,G", [(1, 128, 64, 64, 32), (2, 256, 17, 23, 32), (1, 512, 32, 32, 16),
                                        (3, 64, 9, 5, 4)])
@pytest.mark.parametrize("silu", [True, False], ids=["silu", "nosilu"])
def test_channels_last_entry_matches_torch_group_norm_on_nchw(N, C, H, W, G, silu):
    x, gamma, beta = nchw_case(N, C, H, W, seed=N + C + H + W)
    x_cl = x.cuda().contiguous(memory_format=torch.channels_last)   # pure permutation of memory
    y = gs.gn_silu_nhwc(x_cl, gamma.cuda(), beta.cuda(), G=G, eps=1e-6, apply_silu=silu)
    assert y is not None
    torch.cuda.synchronize()
    assert y.shape == x.shape and y.is_contiguous(memory_format=torch.channels_last)
    ref = torch_ref(x, gamma, beta, G, 1e-6, silu)
    gu.check_y(y.cpu().double().numpy(), ref.numpy(), f"nhwc N={N} C={C} {H}x{W} G={G}")


def test_out_argument_and_side_stream():
    x, gamma, beta = nchw_case(1, 256, 32, 32, seed=5)
    x_cl = x.cuda().contiguous(memory_format=torch.channels_last)
    out = torch.empty_like(x_cl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = gs.gn_silu_nhwc(x_cl, gamma.cuda(), beta.cuda(), G=32, out=out, stream=s)
    s.synchronize()
    assert y is out
    gu.check_y(out.cpu().double().numpy(), torch_ref(x, gamma, beta, 32, 1e-6, True).numpy(), "out=")


def test_rows_entry_on_a_permute_view_equals_the_4d_entry():
    x, gamma, beta = nchw_case(2, 128, 16, 16, seed=9)
    x_cl = x.cuda().contiguous(memory_format=torch.channels_last)
    rows = x_cl.permute(0, 2, 3, 1).reshape(2, 256, 128)       # free view of the same memory
    y4 = gs.gn_silu_nhwc(x_cl, gamma.cuda(), beta.cuda(), G=32)
    yr = gs.gn_silu_rows(rows, gamma.cuda(), beta.cuda(), G=32)
    torch.cuda.synchronize()
    assert torch.equal(y4.permute(0, 2, 3, 1).reshape(2, 256, 128), yr)


def test_unsupported_inputs_return_none():
    x, gamma, beta = nchw_case(1, 64, 8, 8, seed=1)
    g, b = gamma.cuda(), beta.cuda()
    x_nchw = x.cuda()                                           # contiguous NCHW, not channels_last
    assert gs.gn_silu_nhwc(x_nchw, g, b, G=32) is None
    x_cl = x_nchw.contiguous(memory_format=torch.channels_last)
    assert gs.gn_silu_nhwc(x_cl.float(), g, b, G=32) is None   # not bf16
    xg = x_cl.clone().requires_grad_(True)
    assert gs.gn_silu_nhwc(xg, g, b, G=32) is None             # grad enabled
    with torch.no_grad():
        assert gs.gn_silu_nhwc(xg, g, b, G=32) is not None     # fine under no_grad
    with pytest.warns(UserWarning):                             # C not a power of two
        x24 = torch.zeros(1, 24, 4, 4, dtype=torch.bfloat16, device="cuda").contiguous(
            memory_format=torch.channels_last)
        assert gs.gn_silu_nhwc(x24, torch.ones(24, device="cuda"), torch.zeros(24, device="cuda"),
                               G=8) is None
    with pytest.warns(UserWarning):                             # C > 2048
        x4k = torch.zeros(1, 4096, 2, 2, dtype=torch.bfloat16, device="cuda").contiguous(
            memory_format=torch.channels_last)
        assert gs.gn_silu_nhwc(x4k, torch.ones(4096, device="cuda"), torch.zeros(4096, device="cuda"),
                               G=32) is None
    with pytest.warns(UserWarning):                             # G does not divide C
        assert gs.gn_silu_nhwc(x_cl, g, b, G=3) is None
    assert gs.gn_silu_nhwc(x_cl, g[:32], b, G=32) is None      # gamma of the wrong length
    torch.cuda.synchronize()
