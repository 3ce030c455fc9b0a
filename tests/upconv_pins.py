"""Pins of the fused nearest-2x upsample + 3x3 conv oracle, shared by the pin
tests and the mutation tests: each function takes an oracle object and
returns a list of failure messages (empty = pass).

Independent references:
  * PyTorch's CPU float64 `interpolate(mode="nearest")` followed by
    `conv2d(padding=1)` -- the two library routines of the definition;
  * the page's identity (sglang PR #33451, "FLUX.2 VAE decoder fast path
    behind quality=high", section "Modifications", item 2): a transposed
    convolution with kernel 4, stride 2, padding 1 whose 4x4 taps are sums
    of the 3x3 taps, evaluated by PyTorch's `conv_transpose2d` in float64;
  * closed forms (constant input, a single nonzero input pixel), a mirror
    invariant and brute force with explicit numpy pixel replication on tiny
    tensors.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

from channels_last_groupnorm_gb300 import workloads as wl


def _values(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _case(N, H, W, Cin, Cout, seed, bias=True):
    return wl.make_upconv_case(N, H, W, Cin, Cout, seed, bias)


def _torch_reference(c):
    """F.conv2d(F.interpolate(x, 2, 'nearest'), w, b, padding=1) in float64,
    returned channels-last [N, 2H, 2W, Cout]."""
    x = torch.from_numpy(_values(c["x_bits"])).permute(0, 3, 1, 2)
    w = torch.from_numpy(_values(c["w_bits"]))
    b = None if c["bias_bits"] is None else torch.from_numpy(_values(c["bias_bits"]))
    u = F.interpolate(x, scale_factor=2, mode="nearest")
    return F.conv2d(u, w, b, padding=1).permute(0, 2, 3, 1).numpy()


# For kernel index k of the 4-tap transposed convolution (output row
# P = 2 i - 1 + k from input row i), the 3x3 kernel rows whose taps it sums.
# k = 0: odd output rows, input one row below -> kernel row 2
# k = 1: even output rows, same input row     -> kernel rows 1, 2
# k = 2: odd output rows, same input row      -> kernel rows 0, 1
# k = 3: even output rows, input one row above -> kernel row 0
_SUMMED_ROWS = ((2,), (1, 2), (0, 1), (0,))


def _transposed_reference(c):
    x = torch.from_numpy(_values(c["x_bits"])).permute(0, 3, 1, 2)
    w = _values(c["w_bits"])                       # [Cout, Cin, 3, 3]
    Cout, Cin = w.shape[:2]
    w4 = np.zeros((Cin, Cout, 4, 4))               # conv_transpose2d weight layout
    for k1, rows in enumerate(_SUMMED_ROWS):
        for k2, cols in enumerate(_SUMMED_ROWS):
            for ky in rows:
                for kx in cols:
                    w4[:, :, k1, k2] += w[:, :, ky, kx].T
    b = None if c["bias_bits"] is None else torch.from_numpy(_values(c["bias_bits"]))
    y = F.conv_transpose2d(x, torch.from_numpy(w4), b, stride=2, padding=1)
    return y.permute(0, 2, 3, 1).numpy()


def _close(got, want, what, rtol=1e-12, atol=1e-12):
    if got.shape != want.shape:
        return [f"{what}: shape {got.shape} != {want.shape}"]
    err = np.abs(got - want)
    bad = err > atol + rtol * np.abs(want)
    if bad.any():
        at = np.unravel_index(int(np.argmax(err)), err.shape)
        return [f"{what}: {int(bad.sum())} of {bad.size} differ, worst at {at}: "
                f"{got[at]!r} vs {want[at]!r}"]
    return []


def pin_library_conv(o):
    """Agrees with PyTorch's float64 interpolate + conv2d (several shapes,
    with and without bias, odd H and W, N > 1)."""
    out = []
    for shp, seed, bias in (((1, 5, 7, 3, 4), 1, True), ((2, 4, 3, 8, 5), 2, False),
                            ((1, 8, 8, 16, 8), 3, True), ((3, 1, 1, 2, 3), 4, True)):
        c = _case(*shp, seed, bias)
        out += _close(o.forward(c["x_bits"], c["w_bits"], c["bias_bits"]), _torch_reference(c),
                      f"conv2d(interpolate) {shp}")
    return out


def pin_transposed_identity(o):
    """Agrees with the transposed convolution (kernel 4, stride 2, padding 1)
    whose taps are sums of the 3x3 taps."""
    out = []
    for shp, seed, bias in (((1, 6, 5, 4, 3), 5, True), ((2, 3, 4, 8, 8), 6, False)):
        c = _case(*shp, seed, bias)
        out += _close(o.forward(c["x_bits"], c["w_bits"], c["bias_bits"]), _transposed_reference(c),
                      f"conv_transpose2d identity {shp}")
    return out


def pin_constant_input(o):
    """x = 1 everywhere, no bias: each output is the sum of the weight taps
    that land inside the upsampled image (all 9 in the interior, 6 on an
    edge row or column, 4 at a corner)."""
    N, H, W, Cin, Cout = 1, 4, 3, 3, 2
    c = _case(N, H, W, Cin, Cout, 7, bias=False)
    c["x_bits"] = np.full((N, H, W, Cin), 0x3F80, np.uint16)        # bf16 1.0
    w = _values(c["w_bits"])
    y = o.forward(c["x_bits"], c["w_bits"], None)
    want = np.zeros_like(y)
    for P in range(2 * H):
        for Q in range(2 * W):
            ky = [k for k in range(3) if 0 <= P + k - 1 < 2 * H]
            kx = [k for k in range(3) if 0 <= Q + k - 1 < 2 * W]
            want[0, P, Q, :] = w[:, :, ky][:, :, :, kx].sum(axis=(1, 2, 3))
    return _close(y, want, "constant input", rtol=1e-13, atol=1e-13)


def pin_single_pixel(o):
    """One nonzero input pixel (value 1 in channel ci0): the output is
    nonzero only in the 4x4 window of the replicated 2x2 block grown by the
    3x3 kernel, where it is the sum of the taps that reach the block."""
    N, H, W, Cin, Cout = 1, 5, 6, 3, 2
    i0, j0, ci0 = 2, 4, 1
    c = _case(N, H, W, Cin, Cout, 8, bias=False)
    x = np.zeros((N, H, W, Cin), np.uint16)
    x[0, i0, j0, ci0] = 0x3F80
    c["x_bits"] = x
    w = _values(c["w_bits"])
    y = o.forward(c["x_bits"], c["w_bits"], None)
    want = np.zeros_like(y)
    for P in range(2 * H):
        for Q in range(2 * W):
            for ky in range(3):
                for kx in range(3):
                    p, q = P + ky - 1, Q + kx - 1
                    if p in (2 * i0, 2 * i0 + 1) and q in (2 * j0, 2 * j0 + 1):
                        want[0, P, Q, :] += w[:, ci0, ky, kx]
    out = _close(y, want, "single pixel", rtol=1e-13, atol=1e-13)
    nz = np.argwhere(np.abs(y[0]).sum(axis=2) > 0)
    if nz.size and (nz[:, 0].min() < 2 * i0 - 1 or nz[:, 0].max() > 2 * i0 + 2
                    or nz[:, 1].min() < 2 * j0 - 1 or nz[:, 1].max() > 2 * j0 + 2):
        out.append("single pixel: output outside the 4x4 window")
    return out


def pin_brute_force(o):
    """Explicit np.repeat pixel replication, zero padding by np.pad and a
    direct sum over the 3x3 window, on a tiny tensor."""
    N, H, W, Cin, Cout = 2, 3, 2, 2, 3
    c = _case(N, H, W, Cin, Cout, 9, bias=True)
    x = _values(c["x_bits"])
    w = _values(c["w_bits"])
    b = _values(c["bias_bits"])
    u = np.repeat(np.repeat(x, 2, axis=1), 2, axis=2)         # [N, 2H, 2W, Cin]
    up = np.pad(u, ((0, 0), (1, 1), (1, 1), (0, 0)))
    want = np.zeros((N, 2 * H, 2 * W, Cout))
    for n in range(N):
        for P in range(2 * H):
            for Q in range(2 * W):
                win = up[n, P:P + 3, Q:Q + 3, :]                   # [3, 3, Cin]
                for co in range(Cout):
                    want[n, P, Q, co] = b[co] + float(np.sum(win * w[co].transpose(1, 2, 0)))
    return _close(o.forward(c["x_bits"], c["w_bits"], c["bias_bits"]), want, "brute force",
                  rtol=1e-12, atol=1e-12)


def pin_mirror(o):
    """Mirroring the input left-right and the kernel's columns mirrors the
    output left-right (nearest upsampling and zero padding are symmetric)."""
    c = _case(1, 4, 5, 4, 3, 10, bias=True)
    y = o.forward(c["x_bits"], c["w_bits"], c["bias_bits"])
    xm = np.ascontiguousarray(c["x_bits"][:, :, ::-1, :])
    wm = np.ascontiguousarray(c["w_bits"][:, :, :, ::-1])
    ym = o.forward(xm, wm, c["bias_bits"])
    out = _close(ym, y[:, :, ::-1, :], "left-right mirror", rtol=1e-12, atol=1e-12)
    xv = np.ascontiguousarray(c["x_bits"][:, ::-1, :, :])
    wv = np.ascontiguousarray(c["w_bits"][:, :, ::-1, :])
    yv = o.forward(xv, wv, c["bias_bits"])
    out += _close(yv, y[:, ::-1, :, :], "top-bottom mirror", rtol=1e-12, atol=1e-12)
    return out


def pin_at_and_abs(o):
    """The sampled entry point equals the full output at random indices, the
    absolute-term sums bound |y|, equal y for all-positive operands, and an
    index outside the output is rejected."""
    out = []
    c = _case(2, 3, 4, 5, 6, 11, bias=True)
    y, a = o.forward(c["x_bits"], c["w_bits"], c["bias_bits"], with_abs=True)
    idx = np.random.default_rng(0).integers(0, y.size, 200)
    ys, as_ = o.at(c["x_bits"], c["w_bits"], c["bias_bits"], idx, with_abs=True)
    out += _close(ys, y.reshape(-1)[idx], "at() vs forward()", rtol=0, atol=0)
    out += _close(as_, a.reshape(-1)[idx], "at() abs vs forward() abs", rtol=0, atol=0)
    if np.any(a < np.abs(y) * (1 - 1e-12)):
        out.append("abs sums below |y|")
    pos = dict(c)
    pos["x_bits"] = wl.f32_to_bf16_bits(np.abs(_values(c["x_bits"])).astype(np.float32)).reshape(c["x_bits"].shape)
    pos["w_bits"] = wl.f32_to_bf16_bits(np.abs(_values(c["w_bits"])).astype(np.float32)).reshape(c["w_bits"].shape)
    pos["bias_bits"] = wl.f32_to_bf16_bits(np.abs(_values(c["bias_bits"])).astype(np.float32))
    yp, ap = o.forward(pos["x_bits"], pos["w_bits"], pos["bias_bits"], with_abs=True)
    out += _close(ap, yp, "abs sums of positive operands", rtol=1e-12, atol=0)
    try:
        o.at(c["x_bits"], c["w_bits"], c["bias_bits"], np.array([y.size]))
        out.append("out-of-range index accepted")
    except ValueError:
        pass
    return out


ALL_PINS = [pin_library_conv, pin_transposed_identity, pin_constant_input, pin_single_pixel,
            pin_brute_force, pin_mirror, pin_at_and_abs]


def failing_pins(o):
    failed = []
    for pin in ALL_PINS:
        try:
            msgs = pin(o)
        except Exception as e:  # a mutant may also crash a pin
            msgs = [f"raised {type(e).__name__}: {e}"]
        if msgs:
            failed.append((pin.__name__, msgs))
    return failed
