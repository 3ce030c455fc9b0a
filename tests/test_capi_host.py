"""The C-ABI library on the host, without a GPU: it loads, exports every
symbol the header declares, and rejects each kind of unsupported input with
its status code before any CUDA call."""
import math
import os
import re

import pytest
import torch

from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gnsilu.h")

X = 0x10000000          # stand-in device addresses (never dereferenced: every call
Y = 0x20000000          # below is rejected before the library touches the device)
GAM = 0x30000000
BET = 0x30001000
no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="valid stand-in pointers must never reach a real GPU")


@pytest.fixture(scope="module", autouse=True)
def built():
    gnbuild.build()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gn_[a-z_0-9]+)\s*\(", text, re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"gn_silu_nhwc", "gn_silu_rows", "gn_silu_rows_ex", "gn_silu_workspace_bytes",
            "gn_status_string", "gn_device_status", "gn_kernel_launch_count"} <= names


def test_library_exports_every_declared_symbol():
    lib = gs.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(gs.EXPORTS)


def test_abi_version_and_status_strings():
    assert gs.gn_abi_version() == 7
    for code in range(13):
        s = gs.status_string(code)
        assert s.startswith("GN_"), (code, s)
    assert "unknown" in gs.status_string(99)


def rows(**kw):
    a = dict(x=X, gamma=GAM, beta=BET, y=Y, N=1, L=4, C=32, G=32, eps=1e-6, apply_silu=1)
    a.update(kw)
    return gs.raw_gn_silu_rows(a["x"], a["gamma"], a["beta"], a["y"], a["N"], a["L"], a["C"],
                               a["G"], a["eps"], a["apply_silu"])


def rows_ex(**kw):
    a = dict(x=X, gamma=GAM, beta=BET, y=Y, N=1, L=4, C=32, G=32, eps=1e-6, apply_silu=1,
             mean_out=0, rstd_out=0, workspace=0, workspace_bytes=0, variant=0)
    a.update(kw)
    return gs.raw_gn_silu_rows_ex(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), gs.GN_ERR_NULL),
    (dict(y=0), gs.GN_ERR_NULL),
    (dict(gamma=0), gs.GN_ERR_NULL),
    (dict(beta=0), gs.GN_ERR_NULL),
    (dict(N=0), gs.GN_ERR_SHAPE),
    (dict(L=0), gs.GN_ERR_SHAPE),
    (dict(N=-3), gs.GN_ERR_SHAPE),
    (dict(N=1 << 40, L=1 << 40), gs.GN_ERR_SHAPE),
    (dict(C=7, G=7), gs.GN_ERR_CHANNELS),
    (dict(C=12, G=4), gs.GN_ERR_CHANNELS),
    (dict(C=4, G=4), gs.GN_ERR_CHANNELS),
    (dict(C=4096, G=32), gs.GN_ERR_CHANNELS),
    (dict(C=64, G=0), gs.GN_ERR_CHANNELS),
    (dict(C=64, G=3), gs.GN_ERR_CHANNELS),
    (dict(C=64, G=128), gs.GN_ERR_CHANNELS),
    (dict(x=X + 8), gs.GN_ERR_ALIGN),
    (dict(y=Y + 2), gs.GN_ERR_ALIGN),
    (dict(gamma=GAM + 2), gs.GN_ERR_ALIGN),
    (dict(beta=BET + 1), gs.GN_ERR_ALIGN),
    (dict(eps=math.nan), gs.GN_ERR_EPS),
    (dict(eps=math.inf), gs.GN_ERR_EPS),
    (dict(eps=-1e-6), gs.GN_ERR_EPS),
    (dict(y=X + 16), gs.GN_ERR_ALIAS),
    (dict(y=X - 16), gs.GN_ERR_ALIAS),
    (dict(gamma=Y + 64), gs.GN_ERR_ALIAS),
    (dict(beta=Y), gs.GN_ERR_ALIAS),
])
def test_rows_rejects(kw, code):
    assert rows(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(variant=4), gs.GN_ERR_VARIANT),
    (dict(variant=-1), gs.GN_ERR_VARIANT),
    (dict(workspace=0x40000010, workspace_bytes=1 << 20), gs.GN_ERR_ALIGN),
    (dict(mean_out=0x50000002), gs.GN_ERR_ALIGN),
    (dict(mean_out=Y + 32), gs.GN_ERR_ALIAS),
    (dict(mean_out=0x50000000, rstd_out=0x50000000 + 64), gs.GN_ERR_ALIAS),
])
def test_rows_ex_rejects(kw, code):
    assert rows_ex(**kw) == code


@pytest.mark.parametrize("H,W,code", [(0, 4, gs.GN_ERR_SHAPE), (4, -1, gs.GN_ERR_SHAPE),
                                      (1 << 40, 1 << 40, gs.GN_ERR_SHAPE)])
def test_nhwc_rejects_bad_spatial_shape(H, W, code):
    assert gs.raw_gn_silu_nhwc(X, GAM, BET, Y, 1, H, W, 32, 32, 1e-6, 1) == code


def test_nhwc_null_before_shape():
    assert gs.raw_gn_silu_nhwc(0, GAM, BET, Y, 1, 0, 4, 32, 32, 1e-6, 1) == gs.GN_ERR_NULL


@no_gpu
def test_valid_arguments_without_a_device_report_no_device():
    assert rows() == gs.GN_ERR_DEVICE
    assert rows(y=X) == gs.GN_ERR_DEVICE          # in place is allowed
    assert gs.gn_silu_workspace_bytes(1, 4, 32, 32) == 0
    assert gs.gn_silu_pick_variant(1, 4, 32, 32) == -gs.GN_ERR_DEVICE


@no_gpu
def test_workspace_management_without_a_device():
    assert gs.gn_release_workspaces() == gs.GN_ERR_DEVICE
    assert gs.gn_library_workspaces() == -gs.GN_ERR_DEVICE


def static(**kw):
    a = dict(x=X, gamma=GAM, beta=BET, y=Y, N=1, L=4, C=32, G=32, eps=1e-6, apply_silu=1,
             mean_out=None, rstd_out=None, stream=None)
    a.update(kw)
    return gs.lib().gn_silu_rows_static(a["x"], a["gamma"], a["beta"], a["y"], a["N"], a["L"], a["C"],
                                        a["G"], a["eps"], a["apply_silu"], a["mean_out"], a["rstd_out"],
                                        a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), gs.GN_ERR_NULL),
    (dict(L=0), gs.GN_ERR_SHAPE),
    (dict(C=24, G=8), gs.GN_ERR_CHANNELS),        # a general C: only the power-of-two contract here
    (dict(y=Y + 2), gs.GN_ERR_ALIGN),
    (dict(eps=-1.0), gs.GN_ERR_EPS),
    (dict(y=X + 16), gs.GN_ERR_ALIAS),
])
def test_static_entry_checks_arguments_before_anything_else(kw, code):
    # the same statuses, in the same order, as gn_silu_rows_ex; no device is touched
    assert static(**kw) == code


@no_gpu
def test_static_entry_without_a_device():
    assert static() == gs.GN_ERR_DEVICE


def test_workspace_query_rejects_bad_shapes():
    assert gs.gn_silu_workspace_bytes(1, 4, 12, 4) == 0
    assert gs.gn_silu_workspace_bytes(0, 4, 32, 32) == 0
    assert gs.gn_silu_pick_variant(1, 4, 12, 4) == -gs.GN_ERR_CHANNELS


def test_tensor_binding_returns_none_for_cpu_tensors():
    x = torch.zeros(1, 32, 2, 2, dtype=torch.bfloat16).to(memory_format=torch.channels_last)
    g = torch.ones(32)
    assert gs.gn_silu_nhwc(x, g, g) is None
    assert gs.gn_silu_rows(x.reshape(1, 4, 32), g, g) is None
    assert gs.gn_silu_rows_ex(x.reshape(1, 4, 32), g, g) is None


def test_launch_counter_starts_readable():
    assert gs.gn_kernel_launch_count() >= 0


def rows_any(**kw):
    a = dict(x=X, gamma=GAM, beta=BET, y=Y, N=1, L=4, C=320, G=32, eps=1e-6, apply_silu=1,
             mean_out=0, rstd_out=0, workspace=0, workspace_bytes=0, variant=0)
    a.update(kw)
    return gs.raw_gn_silu_rows_any(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), gs.GN_ERR_NULL),
    (dict(L=0), gs.GN_ERR_SHAPE),
    (dict(C=12, G=4), gs.GN_ERR_CHANNELS),        # a row is not whole 16-byte vectors
    (dict(C=4, G=4), gs.GN_ERR_CHANNELS),
    (dict(C=2056, G=8), gs.GN_ERR_CHANNELS),      # above 2048
    (dict(C=320, G=3), gs.GN_ERR_CHANNELS),       # G does not divide C
    (dict(C=320, G=0), gs.GN_ERR_CHANNELS),
    (dict(x=X + 8), gs.GN_ERR_ALIGN),
    (dict(y=X + 16), gs.GN_ERR_ALIAS),
    (dict(eps=-1.0), gs.GN_ERR_EPS),
    (dict(variant=5), gs.GN_ERR_VARIANT),
])
def test_rows_any_rejects(kw, code):
    assert rows_any(**kw) == code


@pytest.mark.parametrize("C,G", [(320, 32), (24, 8), (960, 32), (2040, 8)])
def test_power_of_two_entries_still_reject_general_channel_counts(C, G):
    assert rows(C=C, G=G) == gs.GN_ERR_CHANNELS
    assert rows_ex(C=C, G=G) == gs.GN_ERR_CHANNELS
    assert gs.raw_gn_silu_nhwc(X, GAM, BET, Y, 1, 2, 2, C, G, 1e-6, 1) == gs.GN_ERR_CHANNELS


@no_gpu
@pytest.mark.parametrize("C,G", [(320, 32), (24, 8), (960, 32), (2040, 8), (256, 32), (8, 1)])
def test_rows_any_accepts_general_channel_counts(C, G):
    # accepted by validation; without a GPU the next check reports no device
    assert rows_any(C=C, G=G) == gs.GN_ERR_DEVICE
    assert gs.raw_gn_silu_ndhwc(X, GAM, BET, Y, 1, 2, 2, 2, C, G, 1e-6, 1) == gs.GN_ERR_DEVICE


@pytest.mark.parametrize("D,H,W,code", [(0, 2, 2, gs.GN_ERR_SHAPE), (2, 0, 2, gs.GN_ERR_SHAPE),
                                        (2, 2, -1, gs.GN_ERR_SHAPE),
                                        (1 << 30, 1 << 20, 1 << 20, gs.GN_ERR_SHAPE)])
def test_ndhwc_rejects_bad_spatial_shape(D, H, W, code):
    assert gs.raw_gn_silu_ndhwc(X, GAM, BET, Y, 1, D, H, W, 320, 32, 1e-6, 1) == code
    assert gs.raw_gn_silu_ndhwc(0, GAM, BET, Y, 1, D, H, W, 320, 32, 1e-6, 1) == gs.GN_ERR_NULL


def test_ndhwc_rejects_channels_like_rows_any():
    assert gs.raw_gn_silu_ndhwc(X, GAM, BET, Y, 1, 2, 2, 2, 12, 4, 1e-6, 1) == gs.GN_ERR_CHANNELS


def test_general_tensor_bindings_return_none_for_cpu_tensors():
    x = torch.zeros(1, 320, 2, 2, 2, dtype=torch.bfloat16).to(memory_format=torch.channels_last_3d)
    g = torch.ones(320)
    assert gs.gn_silu_ndhwc(x, g, g) is None
    assert gs.gn_silu_rows_any(torch.zeros(1, 8, 320, dtype=torch.bfloat16), g, g) is None


def rga(**kw):
    a = dict(residual=X, update=Y, gate=GAM, out=0x40000000, rows=4, D=64, fmt=0)
    a.update(kw)
    return gs.raw_gn_residual_gate_add(a["residual"], a["update"], a["gate"], a["out"], a["rows"], a["D"],
                                       a["fmt"])


@pytest.mark.parametrize("kw,code", [
    (dict(residual=0), gs.GN_ERR_NULL),
    (dict(update=0), gs.GN_ERR_NULL),
    (dict(gate=0), gs.GN_ERR_NULL),
    (dict(out=0), gs.GN_ERR_NULL),
    (dict(rows=-1), gs.GN_ERR_SHAPE),
    (dict(rows=1 << 60, D=1 << 20), gs.GN_ERR_SHAPE),
    (dict(D=0), gs.GN_ERR_CHANNELS),
    (dict(D=4), gs.GN_ERR_CHANNELS),
    (dict(D=12), gs.GN_ERR_CHANNELS),
    (dict(residual=X + 2), gs.GN_ERR_ALIGN),
    (dict(gate=GAM + 8), gs.GN_ERR_ALIGN),
    (dict(out=0x40000008), gs.GN_ERR_ALIGN),
    (dict(fmt=2), gs.GN_ERR_FORMAT),
    (dict(fmt=-1), gs.GN_ERR_FORMAT),
    (dict(out=X + 16), gs.GN_ERR_ALIAS),
    (dict(out=Y - 16), gs.GN_ERR_ALIAS),
    (dict(out=GAM - 64), gs.GN_ERR_ALIAS),
])
def test_residual_gate_rejects(kw, code):
    assert rga(**kw) == code


@no_gpu
def test_residual_gate_valid_arguments_without_a_device():
    assert rga() == gs.GN_ERR_DEVICE
    assert rga(out=X) == gs.GN_ERR_DEVICE          # in place on the residual
    assert rga(out=Y, fmt=1) == gs.GN_ERR_DEVICE   # in place on the update, fp16
    assert rga(rows=0) == gs.GN_ERR_DEVICE


def test_residual_gate_binding_returns_none_for_cpu_tensors():
    r = torch.zeros(2, 16, dtype=torch.bfloat16)
    assert gs.residual_gate_add(r, r.clone(), torch.ones(16, dtype=torch.bfloat16)) is None


WF = 0x50000000
BIAS = 0x60000000


def upconv(**kw):
    a = dict(x=X, wf=WF, bias=BIAS, y=Y, N=1, H=16, W=16, Cin=64, Cout=128)
    a.update(kw)
    return gs.raw_gn_upconv_nhwc(a["x"], a["wf"], a["bias"], a["y"], a["N"], a["H"], a["W"], a["Cin"],
                                 a["Cout"])


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), gs.GN_ERR_NULL),
    (dict(wf=0), gs.GN_ERR_NULL),
    (dict(y=0), gs.GN_ERR_NULL),
    (dict(N=-1), gs.GN_ERR_SHAPE),
    (dict(H=0), gs.GN_ERR_SHAPE),
    (dict(W=0), gs.GN_ERR_SHAPE),
    (dict(W=96), gs.GN_ERR_SHAPE),            # below 128 and not a power of two
    (dict(W=192), gs.GN_ERR_SHAPE),           # above 128, not a multiple of it
    (dict(W=16, H=12), gs.GN_ERR_SHAPE),      # H not a multiple of 128 / W = 8
    (dict(W=32, H=3), gs.GN_ERR_SHAPE),       # H below 128 / W and not a power of two
    (dict(Cin=32), gs.GN_ERR_CHANNELS),
    (dict(Cin=96), gs.GN_ERR_CHANNELS),
    (dict(Cout=64), gs.GN_ERR_CHANNELS),
    (dict(Cout=320), gs.GN_ERR_CHANNELS),
    (dict(Cin=16384), gs.GN_ERR_CHANNELS),
    (dict(x=X + 8), gs.GN_ERR_ALIGN),
    (dict(wf=WF + 8), gs.GN_ERR_ALIGN),
    (dict(y=Y + 8), gs.GN_ERR_ALIGN),
    (dict(bias=BIAS + 2), gs.GN_ERR_ALIGN),
    (dict(y=X + 1024), gs.GN_ERR_ALIAS),
    (dict(y=WF - 4096), gs.GN_ERR_ALIAS),
    (dict(y=BIAS - 4096), gs.GN_ERR_ALIAS),
])
def test_upconv_rejects(kw, code):
    assert upconv(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(w=0), gs.GN_ERR_NULL),
    (dict(wf=0), gs.GN_ERR_NULL),
    (dict(Cin=0), gs.GN_ERR_CHANNELS),
    (dict(Cout=100), gs.GN_ERR_CHANNELS),
    (dict(w=X + 1), gs.GN_ERR_ALIGN),
    (dict(wf=WF + 4), gs.GN_ERR_ALIGN),
    (dict(wf=X + 64), gs.GN_ERR_ALIAS),
])
def test_upconv_fold_rejects(kw, code):
    a = dict(w=X, wf=WF, Cin=64, Cout=128)
    a.update(kw)
    assert gs.raw_gn_upconv_fold(a["w"], a["wf"], a["Cin"], a["Cout"]) == code


def test_upconv_folded_bytes():
    assert gs.gn_upconv_folded_bytes(512, 512) == 16 * 512 * 512 * 2
    assert gs.gn_upconv_folded_bytes(0, 128) == -1


@no_gpu
def test_upconv_valid_arguments_without_a_device():
    assert upconv() == gs.GN_ERR_DEVICE
    assert upconv(bias=0) == gs.GN_ERR_DEVICE
    assert upconv(N=3, H=8, W=8) == gs.GN_ERR_DEVICE       # images grouped in one tile
    assert upconv(N=1, H=4, W=256, Cout=256) == gs.GN_ERR_DEVICE
    assert upconv(N=0) == gs.GN_ERR_DEVICE
    assert gs.raw_gn_upconv_fold(X, WF, 64, 128) == gs.GN_ERR_DEVICE


def test_upconv_bindings_return_none_for_cpu_tensors():
    x = torch.zeros(1, 64, 8, 8, dtype=torch.bfloat16).to(memory_format=torch.channels_last)
    w = torch.zeros(128, 64, 3, 3, dtype=torch.bfloat16)
    assert gs.upconv_fold(w) is None
    assert gs.upsample_conv_nhwc(x, torch.zeros(4, 128, 256, dtype=torch.bfloat16)) is None


AQ, AK, AX, AW, AB, AR, AO, AWS = (0x70000000 + i * 0x02000000 for i in range(8))


def attn(**kw):
    a = dict(q=AQ, k=AK, xn=AX, wf=AW, bf=AB, residual=AR, out=AO, S=256, D=512, ws=AWS,
             ws_bytes=gs.gn_attn_workspace_bytes(256, 512))
    a.update(kw)
    return gs.raw_gn_attn_folded(a["q"], a["k"], a["xn"], a["wf"], a["bf"], a["residual"], a["out"], a["S"],
                                 a["D"], a["ws"], a["ws_bytes"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), gs.GN_ERR_NULL),
    (dict(k=0), gs.GN_ERR_NULL),
    (dict(xn=0), gs.GN_ERR_NULL),
    (dict(wf=0), gs.GN_ERR_NULL),
    (dict(bf=0), gs.GN_ERR_NULL),
    (dict(out=0), gs.GN_ERR_NULL),
    (dict(ws=0), gs.GN_ERR_NULL),
    (dict(S=0), gs.GN_ERR_SHAPE),
    (dict(S=100), gs.GN_ERR_SHAPE),
    (dict(S=65536), gs.GN_ERR_SHAPE),
    (dict(D=64), gs.GN_ERR_CHANNELS),
    (dict(D=320), gs.GN_ERR_CHANNELS),
    (dict(D=2048), gs.GN_ERR_CHANNELS),
    (dict(q=AQ + 8), gs.GN_ERR_ALIGN),
    (dict(residual=AR + 8), gs.GN_ERR_ALIGN),
    (dict(ws=AWS + 16), gs.GN_ERR_ALIGN),
    (dict(ws_bytes=1024), gs.GN_ERR_WORKSPACE),
    (dict(out=AQ + 256), gs.GN_ERR_ALIAS),
    (dict(out=AWS + 1024), gs.GN_ERR_ALIAS),
    (dict(residual=AO + 256), gs.GN_ERR_ALIAS),
    (dict(ws=AX), gs.GN_ERR_ALIAS),
    (dict(ws=AO - 0x100000, ws_bytes=0x200000), gs.GN_ERR_ALIAS),   # the whole declared workspace counts
])
def test_attn_rejects(kw, code):
    assert attn(**kw) == code


def test_attn_workspace_bytes():
    def up(v):
        return (v + 255) // 256 * 256
    S, D = 256, 512
    # folded value rows, per-row-segment softmax records (room for 128-wide tiles), row stats, P
    want = up(2 * D * S) + up(8 * S * 2 * (S // 128)) + up(8 * S) + up(2 * S * S)
    assert gs.gn_attn_workspace_bytes(S, D) == want
    assert gs.gn_attn_workspace_bytes(100, 512) == 0
    assert gs.gn_attn_workspace_bytes(256, 96) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(wv=0), gs.GN_ERR_NULL),
    (dict(bf=0), gs.GN_ERR_NULL),
    (dict(D=100), gs.GN_ERR_CHANNELS),
    (dict(wf=AW + 8), gs.GN_ERR_ALIGN),
    (dict(wv=AQ + 1), gs.GN_ERR_ALIGN),
    (dict(wf=AQ), gs.GN_ERR_ALIAS),
])
def test_attn_fold_rejects(kw, code):
    a = dict(wv=AQ, bv=AK, wo=AX, bo=AR, wf=AW, bf=AB, D=512)
    a.update(kw)
    assert gs.raw_gn_attn_fold(a["wv"], a["bv"], a["wo"], a["bo"], a["wf"], a["bf"], a["D"]) == code


def attn_ex(schedule, **kw):
    a = dict(q=AQ, k=AK, xn=AX, wf=AW, bf=AB, residual=AR, out=AO, S=256, D=512, ws=AWS,
             ws_bytes=gs.gn_attn_workspace_bytes(256, 512))
    a.update(kw)
    return gs.raw_gn_attn_folded_ex(a["q"], a["k"], a["xn"], a["wf"], a["bf"], a["residual"], a["out"], a["S"],
                                    a["D"], a["ws"], a["ws_bytes"], schedule)


@pytest.mark.parametrize("schedule,kw,code", [
    (3, {}, gs.GN_ERR_VARIANT),
    (-1, {}, gs.GN_ERR_VARIANT),
    (gs.ATTN_ONE_PASS, dict(D=1024, ws_bytes=gs.gn_attn_workspace_bytes(256, 1024)), gs.GN_ERR_VARIANT),
    (gs.ATTN_ONE_PASS, dict(q=0), gs.GN_ERR_NULL),
    (gs.ATTN_STORED_WEIGHTS, dict(S=100), gs.GN_ERR_SHAPE),
    (gs.ATTN_ONE_PASS, dict(ws_bytes=1024), gs.GN_ERR_WORKSPACE),
])
def test_attn_ex_rejects(schedule, kw, code):
    assert attn_ex(schedule, **kw) == code


def test_attention_binding_refuses_a_bad_schedule():
    t = torch.zeros(256, 512, dtype=torch.bfloat16)
    w = torch.zeros(512, 512, dtype=torch.bfloat16)
    assert gs.attention_folded(t, t, t, w, torch.zeros(512), schedule=7) is None


@no_gpu
def test_attn_valid_arguments_without_a_device():
    for schedule in (gs.ATTN_AUTO, gs.ATTN_ONE_PASS, gs.ATTN_STORED_WEIGHTS):
        assert attn_ex(schedule) == gs.GN_ERR_DEVICE
    assert attn() == gs.GN_ERR_DEVICE
    assert attn(residual=0) == gs.GN_ERR_DEVICE
    assert attn(residual=AO) == gs.GN_ERR_DEVICE        # in place on the residual
    assert gs.raw_gn_attn_fold(AQ, AK, AX, AR, AW, AB, 512) == gs.GN_ERR_DEVICE


def test_attn_bindings_return_none_for_cpu_tensors():
    t = torch.zeros(256, 512, dtype=torch.bfloat16)
    assert gs.attn_fold(torch.zeros(512, 512, dtype=torch.bfloat16), t[0], t[:512].clone(), t[1]) is None
    assert gs.attention_folded(t, t, t, torch.zeros(512, 512, dtype=torch.bfloat16), torch.zeros(512)) is None
