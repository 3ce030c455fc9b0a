"""Python binding of libgnsilu (``include/gnsilu.h``): argument marshalling only.

Every step of the computation runs in the CUDA kernels of ``libgnsilu.so``;
this module checks tensor metadata, takes device pointers and the current
stream from PyTorch, and calls the C entry point of the same name.  There is
no CPU or PyTorch fallback: if the library is missing, every entry point
raises.

Unsupported inputs give ``None``, the contract of the sglang PR #33451 page
("FLUX.2 VAE decoder fast path behind quality=high", section
"Modifications", item 1, second bullet: non-CUDA, grad enabled,
non-power-of-two C, C > 2048, not channels_last), so callers can fall back
to their own path.  A caller-given ``out`` or ``workspace`` of the wrong
shape, dtype, device or layout is unsupported input too.
``gn_silu_rows_any`` and ``gn_silu_ndhwc`` take any C that is a multiple of 8
up to 2048 (any channels per group) and 5D channels-last input, the range of
the page's existing general kernel (same section, item 1, third bullet).
``residual_gate_add``, ``upconv_fold`` / ``upsample_conv_nhwc`` and
``attn_fold`` / ``attention_folded`` bind the residual-gate update, the
fused nearest-2x upsample + 3x3 conv and the folded single-head attention
the same way.
"""
from __future__ import annotations

import ctypes
import os
import threading
import warnings

LIB_NAME = "libgnsilu.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

GN_OK = 0
GN_ERR_NULL = 1
GN_ERR_SHAPE = 2
GN_ERR_CHANNELS = 3
GN_ERR_ALIGN = 4
GN_ERR_EPS = 5
GN_ERR_ALIAS = 6
GN_ERR_WORKSPACE = 7
GN_ERR_CUDA = 8
GN_ERR_DEVICE = 9
GN_ERR_VARIANT = 10
GN_ERR_KERNEL = 11
GN_ERR_FORMAT = 12

VARIANT_AUTO = 0
VARIANT_TWO_PASS = 1
VARIANT_FUSED = 2
VARIANT_CLUSTER = 3

# schedules of gn_attn_folded_ex (GN_ATTN_* in gnsilu.h)
ATTN_AUTO = 0
ATTN_ONE_PASS = 1
ATTN_STORED_WEIGHTS = 2

# statuses that mean "this input is not supported" (the caller falls back)
UNSUPPORTED = {GN_ERR_SHAPE, GN_ERR_CHANNELS, GN_ERR_ALIGN, GN_ERR_EPS, GN_ERR_ALIAS, GN_ERR_FORMAT}

EXPORTS = {
    # name: (restype, argtypes)
    "gn_silu_nhwc": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 5
                     + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "gn_silu_rows": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 4
                     + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "gn_silu_rows_ex": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 4
                        + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]),
    "gn_silu_rows_any": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 4
                         + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]),
    "gn_silu_ndhwc": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 6
                      + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "gn_silu_rows_static": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 4
                            + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p]),
    "gn_residual_gate_add": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 2
                             + [ctypes.c_int, ctypes.c_void_p]),
    "gn_upconv_folded_bytes": (ctypes.c_int64, [ctypes.c_int64] * 2),
    "gn_upconv_fold": (ctypes.c_int, [ctypes.c_void_p] * 2 + [ctypes.c_int64] * 2 + [ctypes.c_void_p]),
    "gn_upconv_nhwc": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 5 + [ctypes.c_void_p]),
    "gn_attn_fold": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int64, ctypes.c_void_p]),
    "gn_attn_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64] * 2),
    "gn_attn_folded": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int64] * 2
                       + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gn_attn_folded_ex": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int64] * 2
                          + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]),
    "gn_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_int, ctypes.c_void_p]),
    "gn_silu_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64] * 4),
    "gn_silu_pick_variant": (ctypes.c_int, [ctypes.c_int64] * 4),
    "gn_kernel_launch_count": (ctypes.c_uint64, []),
    "gn_device_status": (ctypes.c_int, [ctypes.c_int]),
    "gn_release_workspaces": (ctypes.c_int, []),
    "gn_library_workspaces": (ctypes.c_int, []),
    "gn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gn_abi_version": (ctypes.c_int, []),
}


class GnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded ``libgnsilu.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m channels_last_groupnorm_gb300.build` (nvcc, sm_103a)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().gn_status_string(int(status)).decode()


# ---------------------------------------------------------------------------
# raw C entry points (integer device pointers)
# ---------------------------------------------------------------------------
def raw_gn_silu_rows_ex(x, gamma, beta, y, N, L, C, G, eps, apply_silu, mean_out=0, rstd_out=0,
                        workspace=0, workspace_bytes=0, variant=VARIANT_AUTO, stream=0) -> int:
    return lib().gn_silu_rows_ex(x, gamma, beta, y, N, L, C, G, float(eps), int(apply_silu),
                                 mean_out or None, rstd_out or None, workspace or None,
                                 workspace_bytes, variant, stream or None)


def raw_gn_silu_rows_any(x, gamma, beta, y, N, L, C, G, eps, apply_silu, mean_out=0, rstd_out=0,
                         workspace=0, workspace_bytes=0, variant=VARIANT_AUTO, stream=0) -> int:
    return lib().gn_silu_rows_any(x, gamma, beta, y, N, L, C, G, float(eps), int(apply_silu),
                                  mean_out or None, rstd_out or None, workspace or None,
                                  workspace_bytes, variant, stream or None)


def raw_gn_silu_ndhwc(x, gamma, beta, y, N, D, H, W, C, G, eps, apply_silu, stream=0) -> int:
    return lib().gn_silu_ndhwc(x, gamma, beta, y, N, D, H, W, C, G, float(eps), int(apply_silu),
                               stream or None)


def raw_gn_silu_rows(x, gamma, beta, y, N, L, C, G, eps, apply_silu, stream=0) -> int:
    return lib().gn_silu_rows(x, gamma, beta, y, N, L, C, G, float(eps), int(apply_silu),
                              stream or None)


def raw_gn_silu_nhwc(x, gamma, beta, y, N, H, W, C, G, eps, apply_silu, stream=0) -> int:
    return lib().gn_silu_nhwc(x, gamma, beta, y, N, H, W, C, G, float(eps), int(apply_silu),
                              stream or None)


def gn_silu_workspace_bytes(N: int, L: int, C: int, G: int) -> int:
    return int(lib().gn_silu_workspace_bytes(N, L, C, G))


def gn_silu_pick_variant(N: int, L: int, C: int, G: int) -> int:
    return int(lib().gn_silu_pick_variant(N, L, C, G))


def gn_kernel_launch_count() -> int:
    return int(lib().gn_kernel_launch_count())


def gn_device_status(clear: bool = False) -> int:
    return int(lib().gn_device_status(int(bool(clear))))


def gn_abi_version() -> int:
    return int(lib().gn_abi_version())


def gn_release_workspaces() -> int:
    """Free the workspaces the library allocated on the current device."""
    return int(lib().gn_release_workspaces())


def gn_library_workspaces() -> int:
    return int(lib().gn_library_workspaces())


# ---------------------------------------------------------------------------
# tensor entry points
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _affine_ok(t, C, device) -> bool:
    torch = _torch()
    return (t is not None and t.is_cuda and t.device == device and t.dtype == torch.float32
            and t.dim() == 1 and t.numel() == C and t.is_contiguous())


def _workspace_ok(ws, device) -> bool:
    torch = _torch()
    return (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.device == device and ws.dtype == torch.uint8
            and ws.dim() == 1 and ws.is_contiguous())


def _grad_blocked(*ts) -> bool:
    torch = _torch()
    return torch.is_grad_enabled() and any(t is not None and t.requires_grad for t in ts)


def _stream_handle(device, stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _finish(rc: int, what: str):
    if rc == GN_OK:
        return True
    if rc in UNSUPPORTED:
        warnings.warn(f"{what}: unsupported input ({status_string(rc)})", stacklevel=3)
        return False
    raise GnError(rc, what)


def gn_silu_nhwc(x, gamma, beta, G: int = 32, eps: float = 1e-6, apply_silu: bool = True,
                 out=None, stream=None):
    """GroupNorm(+SiLU) of a channels_last bf16 CUDA tensor (N, C, H, W).

    Returns y with x's shape and memory format, or None when the input is
    not supported (the caller then falls back)."""
    lib()
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16
            and x.dim() == 4):
        return None
    if not x.is_contiguous(memory_format=torch.channels_last) or _grad_blocked(x, gamma, beta):
        return None
    N, C, H, W = x.shape
    if not (_affine_ok(gamma, C, x.device) and _affine_ok(beta, C, x.device)):
        return None
    if out is None:
        out = torch.empty_like(x, memory_format=torch.channels_last)
    elif not (out.shape == x.shape and out.dtype == x.dtype and out.device == x.device
              and out.is_contiguous(memory_format=torch.channels_last)):
        return None
    with torch.cuda.device(x.device):
        rc = raw_gn_silu_nhwc(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), out.data_ptr(),
                              N, H, W, C, G, eps, apply_silu, _stream_handle(x.device, stream))
    return out if _finish(rc, "gn_silu_nhwc") else None


def gn_silu_rows(x, gamma, beta, G: int = 32, eps: float = 1e-6, apply_silu: bool = True,
                 out=None, stream=None):
    """GroupNorm(+SiLU) of contiguous bf16 CUDA rows (N, L, C).  Returns y or
    None when the input is not supported."""
    lib()
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16
            and x.dim() == 3 and x.is_contiguous()) or _grad_blocked(x, gamma, beta):
        return None
    N, L, C = x.shape
    if not (_affine_ok(gamma, C, x.device) and _affine_ok(beta, C, x.device)):
        return None
    if out is None:
        out = torch.empty_like(x)
    elif not (out.shape == x.shape and out.dtype == x.dtype and out.device == x.device
              and out.is_contiguous()):
        return None
    with torch.cuda.device(x.device):
        rc = raw_gn_silu_rows(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), out.data_ptr(),
                              N, L, C, G, eps, apply_silu, _stream_handle(x.device, stream))
    return out if _finish(rc, "gn_silu_rows") else None


def new_workspace(x, G: int = 32):
    """A zero-filled workspace for ``gn_silu_rows_ex`` / ``gn_silu_rows_any``
    on rows shaped like ``x`` (N, L, C): a uint8 tensor on x's device of
    ``gn_silu_workspace_bytes`` bytes, or None if the shape is unsupported."""
    torch = _torch()
    N, L, C = x.shape
    with torch.cuda.device(x.device):
        need = gn_silu_workspace_bytes(N, L, C, G)
    if need == 0:
        return None
    return torch.zeros(need, dtype=torch.uint8, device=x.device)


def gn_silu_rows_ex(x, gamma, beta, G: int = 32, eps: float = 1e-6, apply_silu: bool = True,
                    out=None, variant: int = VARIANT_AUTO, workspace=None, stream=None):
    """``gn_silu_rows`` that also returns the fp32 statistics:
    (y, mean [N, G], rstd [N, G]), or None when unsupported.

    ``workspace``: None (the library's own), or a contiguous uint8 tensor on
    x's device of at least ``gn_silu_workspace_bytes`` bytes whose first 256
    bytes are zero before its first use -- ``new_workspace(x, G)`` makes one.
    The kernels leave those bytes zero after every successful call, so the
    same workspace serves any number of calls that do not overlap on the
    GPU; after ``gn_device_status(True)`` clears a failure it must be zeroed
    again."""
    return _rows_with_stats(raw_gn_silu_rows_ex, "gn_silu_rows_ex", x, gamma, beta, G, eps,
                            apply_silu, out, variant, workspace, stream)


def gn_silu_rows_any(x, gamma, beta, G: int = 32, eps: float = 1e-6, apply_silu: bool = True,
                     out=None, variant: int = VARIANT_AUTO, workspace=None, stream=None):
    """``gn_silu_rows_ex`` for any C that is a multiple of 8 up to 2048 and
    any G dividing C: (y, mean [N, G], rstd [N, G]), or None when
    unsupported."""
    return _rows_with_stats(raw_gn_silu_rows_any, "gn_silu_rows_any", x, gamma, beta, G, eps,
                            apply_silu, out, variant, workspace, stream)


def gn_silu_ndhwc(x, gamma, beta, G: int = 32, eps: float = 1e-6, apply_silu: bool = True,
                  out=None, stream=None):
    """GroupNorm(+SiLU) of a channels_last_3d bf16 CUDA tensor (N, C, D, H, W),
    any C that is a multiple of 8 up to 2048.  Returns y with x's shape and
    memory format, or None when the input is not supported."""
    lib()
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16
            and x.dim() == 5):
        return None
    if not x.is_contiguous(memory_format=torch.channels_last_3d) or _grad_blocked(x, gamma, beta):
        return None
    N, C, D, H, W = x.shape
    if not (_affine_ok(gamma, C, x.device) and _affine_ok(beta, C, x.device)):
        return None
    if out is None:
        out = torch.empty_like(x, memory_format=torch.channels_last_3d)
    elif not (out.shape == x.shape and out.dtype == x.dtype and out.device == x.device
              and out.is_contiguous(memory_format=torch.channels_last_3d)):
        return None
    with torch.cuda.device(x.device):
        rc = raw_gn_silu_ndhwc(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), out.data_ptr(),
                               N, D, H, W, C, G, eps, apply_silu, _stream_handle(x.device, stream))
    return out if _finish(rc, "gn_silu_ndhwc") else None


def _rows_with_stats(raw, what, x, gamma, beta, G, eps, apply_silu, out, variant, workspace,
                     stream):
    lib()
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16
            and x.dim() == 3 and x.is_contiguous()) or _grad_blocked(x, gamma, beta):
        return None
    N, L, C = x.shape
    if not (_affine_ok(gamma, C, x.device) and _affine_ok(beta, C, x.device)):
        return None
    if out is None:
        out = torch.empty_like(x)
    elif not (isinstance(out, torch.Tensor) and out.shape == x.shape and out.dtype == x.dtype
              and out.device == x.device and out.is_contiguous()):
        return None
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        if not _workspace_ok(workspace, x.device):
            return None
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    mean = torch.empty((N, G), dtype=torch.float32, device=x.device)
    rstd = torch.empty((N, G), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = raw(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), out.data_ptr(),
                 N, L, C, G, eps, apply_silu, mean.data_ptr(), rstd.data_ptr(),
                 ws_ptr, ws_bytes, variant, _stream_handle(x.device, stream))
    return (out, mean, rstd) if _finish(rc, what) else None


# ---------------------------------------------------------------------------
# residual-gate update (the prhub digest of sglang PR #33823, FLUX.2
# bit-exact residual-gate fusion): residual + gate * update in half
# precision, bit for bit equal to the eager two-kernel evaluation
# ---------------------------------------------------------------------------
FORMAT = {"bfloat16": 0, "float16": 1}


def raw_gn_residual_gate_add(residual, update, gate, out, rows, D, fmt, stream=0) -> int:
    return lib().gn_residual_gate_add(residual, update, gate, out, rows, D, int(fmt), stream or None)


def residual_gate_add(residual, update, gate, out=None, stream=None):
    """``residual + gate * update`` for contiguous bf16 / fp16 CUDA tensors
    of the same shape [..., D] and a gate broadcast along every dimension
    but the last (shape [D] or [1, ..., 1, D]).  Returns the result (``out``
    if given; ``out`` may be ``residual`` or ``update``) or None when the
    input is not supported (not CUDA, fp32 or another dtype -- whose eager
    evaluation rounds differently --, a gate that varies along another
    dimension, D not a multiple of 8, non-contiguous), so the caller can
    fall back to the eager expression."""
    lib()
    torch = _torch()
    ts = (residual, update, gate)
    if not all(isinstance(t, torch.Tensor) and t.is_cuda for t in ts):
        return None
    dt = residual.dtype
    if str(dt).replace("torch.", "") not in FORMAT or update.dtype != dt or gate.dtype != dt:
        return None
    if residual.shape != update.shape or residual.dim() < 1 or _grad_blocked(*ts):
        return None
    D = residual.shape[-1]
    if gate.shape[-1] != D or gate.numel() != D:
        return None
    if not (residual.is_contiguous() and update.is_contiguous() and gate.is_contiguous()):
        return None
    if not (residual.device == update.device == gate.device):
        return None
    if out is None:
        out = torch.empty_like(residual)
    elif not (out.shape == residual.shape and out.dtype == dt and out.device == residual.device
              and out.is_contiguous()):
        return None
    rows = residual.numel() // D if D else 0
    with torch.cuda.device(residual.device):
        rc = raw_gn_residual_gate_add(residual.data_ptr(), update.data_ptr(), gate.data_ptr(), out.data_ptr(),
                                      rows, D, FORMAT[str(dt).replace("torch.", "")],
                                      _stream_handle(residual.device, stream))
    return out if _finish(rc, "gn_residual_gate_add") else None


# ---------------------------------------------------------------------------
# fused nearest-2x upsample + 3x3 convolution
# ---------------------------------------------------------------------------
def raw_gn_upconv_fold(w, wf, Cin, Cout, stream=0) -> int:
    return lib().gn_upconv_fold(w, wf, Cin, Cout, stream or None)


def raw_gn_upconv_nhwc(x, wf, bias, y, N, H, W, Cin, Cout, stream=0) -> int:
    return lib().gn_upconv_nhwc(x, wf, bias or None, y, N, H, W, Cin, Cout, stream or None)


def gn_upconv_folded_bytes(Cin: int, Cout: int) -> int:
    return int(lib().gn_upconv_folded_bytes(Cin, Cout))


def upconv_fold(weight, stream=None):
    """Summed 2x2-window taps of a Conv2d(Cin, Cout, 3, padding=1) weight
    (bf16 CUDA tensor [Cout, Cin, 3, 3]) for ``upsample_conv_nhwc``: a bf16
    tensor [4, Cout, 4 * Cin].  None when the weight is not supported (not a
    contiguous bf16 CUDA tensor of that shape, Cin not a multiple of 64,
    Cout not a multiple of 128)."""
    lib()
    torch = _torch()
    if not (isinstance(weight, torch.Tensor) and weight.is_cuda and weight.dtype == torch.bfloat16
            and weight.dim() == 4 and tuple(weight.shape[2:]) == (3, 3) and weight.is_contiguous()):
        return None
    if _grad_blocked(weight):
        return None
    Cout, Cin = weight.shape[:2]
    if gn_upconv_folded_bytes(Cin, Cout) < 0:
        return None
    wf = torch.empty((4, Cout, 4 * Cin), dtype=torch.bfloat16, device=weight.device)
    with torch.cuda.device(weight.device):
        rc = raw_gn_upconv_fold(weight.data_ptr(), wf.data_ptr(), Cin, Cout,
                                _stream_handle(weight.device, stream))
    return wf if _finish(rc, "gn_upconv_fold") else None


def upsample_conv_nhwc(x, folded, bias=None, out=None, stream=None):
    """``conv2d(interpolate(x, scale_factor=2, mode="nearest"), w, bias,
    padding=1)`` for a channels_last bf16 CUDA tensor x (N, Cin, H, W) and
    the folded weight from ``upconv_fold(w)``.  Returns y (N, Cout, 2H, 2W)
    in channels_last, or None when the input is not supported (layout,
    dtype, channel counts, or an (H, W) the kernel's tiles do not cover)."""
    lib()
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 4):
        return None
    if not x.is_contiguous(memory_format=torch.channels_last):
        return None
    N, Cin, H, W = x.shape
    if not (isinstance(folded, torch.Tensor) and folded.is_cuda and folded.dtype == torch.bfloat16
            and folded.dim() == 3 and folded.shape[0] == 4 and folded.shape[2] == 4 * Cin
            and folded.is_contiguous() and folded.device == x.device):
        return None
    Cout = folded.shape[1]
    if bias is not None and not (isinstance(bias, torch.Tensor) and bias.is_cuda and bias.dtype == torch.bfloat16
                                 and bias.numel() == Cout and bias.is_contiguous()
                                 and bias.device == x.device):
        return None
    if _grad_blocked(x, folded, bias):
        return None
    shape = (N, Cout, 2 * H, 2 * W)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=x.device, memory_format=torch.channels_last)
    elif not (tuple(out.shape) == shape and out.dtype == torch.bfloat16 and out.device == x.device
              and out.is_contiguous(memory_format=torch.channels_last)):
        return None
    if N == 0:
        return out
    with torch.cuda.device(x.device):
        rc = raw_gn_upconv_nhwc(x.data_ptr(), folded.data_ptr(), 0 if bias is None else bias.data_ptr(),
                                out.data_ptr(), N, H, W, Cin, Cout, _stream_handle(x.device, stream))
    return out if _finish(rc, "gn_upconv_nhwc") else None


# ---------------------------------------------------------------------------
# single-head attention with the output projection folded into V
# ---------------------------------------------------------------------------
def raw_gn_attn_fold(wv, bv, wo, bo, wf, bf, D, stream=0) -> int:
    return lib().gn_attn_fold(wv, bv, wo, bo, wf, bf, D, stream or None)


def raw_gn_attn_folded(q, k, xn, wf, bf, residual, out, S, D, workspace, workspace_bytes, stream=0) -> int:
    return lib().gn_attn_folded(q, k, xn, wf, bf, residual or None, out, S, D, workspace, workspace_bytes,
                                stream or None)


def raw_gn_attn_folded_ex(q, k, xn, wf, bf, residual, out, S, D, workspace, workspace_bytes, schedule,
                          stream=0) -> int:
    return lib().gn_attn_folded_ex(q, k, xn, wf, bf, residual or None, out, S, D, workspace, workspace_bytes,
                                   schedule, stream or None)


def gn_attn_workspace_bytes(S: int, D: int) -> int:
    return int(lib().gn_attn_workspace_bytes(S, D))


def attn_fold(wv, bv, wo, bo, stream=None):
    """Fold an attention block's value projection (wv [D, D], bv [D]) and
    output projection (wo, bo) -- bf16 CUDA tensors, Linear layout -- into
    (W' bf16 [D, D], b' fp32 [D]).  None when not supported."""
    lib()
    torch = _torch()
    ts = (wv, bv, wo, bo)
    if not all(isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
               for t in ts):
        return None
    if _grad_blocked(*ts) or wv.dim() != 2 or wv.shape[0] != wv.shape[1]:
        return None
    D = wv.shape[0]
    if wo.shape != wv.shape or bv.numel() != D or bo.numel() != D or not all(t.device == wv.device for t in ts):
        return None
    wf = torch.empty((D, D), dtype=torch.bfloat16, device=wv.device)
    bf = torch.empty((D,), dtype=torch.float32, device=wv.device)
    with torch.cuda.device(wv.device):
        rc = raw_gn_attn_fold(wv.data_ptr(), bv.data_ptr(), wo.data_ptr(), bo.data_ptr(), wf.data_ptr(),
                              bf.data_ptr(), D, _stream_handle(wv.device, stream))
    return (wf, bf) if _finish(rc, "gn_attn_fold") else None


def attention_folded(q, k, xn, wf, bf, residual=None, out=None, workspace=None, stream=None,
                     schedule=ATTN_AUTO):
    """``softmax(q k^T / sqrt(D)) (xn W'^T + b') + residual`` for bf16 CUDA
    tensors q, k, xn (and residual) of shape [S, D] and the folded weight
    from ``attn_fold``; equal to the unfolded single-head attention block
    (value projection, attention, output projection, residual).  Returns
    out [S, D] bf16, or None when not supported (S not a multiple of 128 in
    [128, 32768], D not a multiple of 128 in [128, 1024], layouts, dtypes,
    a ``workspace`` that is not a contiguous 1-D uint8 tensor on q's
    device -- a smaller one is replaced by a fresh one --, ATTN_ONE_PASS
    with D > 512).  ``schedule``: ATTN_AUTO, ATTN_ONE_PASS (scores kept on
    chip) or ATTN_STORED_WEIGHTS (softmax weights through the workspace).
    All of a given ``workspace`` may be used: the one-pass schedule keeps
    there the pieces of query tiles it splits between CTA pairs."""
    lib()
    torch = _torch()
    ts = (q, k, xn)
    if not all(isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 2
               and t.is_contiguous() for t in ts):
        return None
    S, D = q.shape
    if k.shape != q.shape or xn.shape != q.shape or not all(t.device == q.device for t in ts):
        return None
    if not (isinstance(wf, torch.Tensor) and wf.is_cuda and wf.dtype == torch.bfloat16 and wf.shape == (D, D)
            and wf.is_contiguous() and isinstance(bf, torch.Tensor) and bf.dtype == torch.float32
            and bf.numel() == D and bf.is_contiguous() and wf.device == q.device and bf.device == q.device):
        return None
    if residual is not None and not (isinstance(residual, torch.Tensor) and residual.shape == q.shape
                                     and residual.dtype == torch.bfloat16 and residual.is_contiguous()
                                     and residual.device == q.device):
        return None
    if _grad_blocked(q, k, xn, wf, bf, residual):
        return None
    if schedule not in (ATTN_AUTO, ATTN_ONE_PASS, ATTN_STORED_WEIGHTS) or (schedule == ATTN_ONE_PASS and D > 512):
        return None
    need = gn_attn_workspace_bytes(S, D)
    if need == 0:
        warnings.warn("attention_folded: unsupported S or D", stacklevel=2)
        return None
    if out is None:
        out = torch.empty_like(q)
    elif not (out.shape == q.shape and out.dtype == torch.bfloat16 and out.is_contiguous()
              and out.device == q.device):
        return None
    if workspace is not None and not _workspace_ok(workspace, q.device):
        return None
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = raw_gn_attn_folded_ex(q.data_ptr(), k.data_ptr(), xn.data_ptr(), wf.data_ptr(), bf.data_ptr(),
                                   0 if residual is None else residual.data_ptr(), out.data_ptr(), S, D,
                                   workspace.data_ptr(), workspace.numel(), schedule,
                                   _stream_handle(q.device, stream))
    return out if _finish(rc, "gn_attn_folded") else None
