"""Pins of the residual-gate oracle (y = residual + gate * update, half
precision, eager two-step rounding), shared by the pin tests and the
mutation tests: each function returns a list of failure messages.

Independent references: PyTorch's own CPU elementwise kernels (eager
`r + g * u` on bf16 / fp16 tensors), numpy's float16 arithmetic, and closed
forms (gate = 1, gate = 0, exhaustive sweeps over every bit pattern)."""
from __future__ import annotations

import numpy as np
import torch

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, fmt: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(DT[fmt])


def same(a: np.ndarray, b: np.ndarray, fmt: str) -> np.ndarray:
    """Elementwise bit equality, with every NaN equal to every NaN."""
    ta, tb = from_bits(a, fmt).float(), from_bits(b, fmt).float()
    return (a == b) | (torch.isnan(ta) & torch.isnan(tb)).numpy()


def wide_values(shape, fmt, seed):
    """Random half values over a wide exponent range, with specials mixed in."""
    rng = np.random.default_rng(seed)
    mant = rng.standard_normal(shape).astype(np.float32)
    lim = 30 if fmt == "bf16" else 6
    scale = np.exp2(rng.integers(-lim, lim, shape)).astype(np.float32)
    t = torch.from_numpy(mant * scale).to(DT[fmt])
    flat = t.view(-1)
    k = flat.numel()
    specials = torch.tensor([float("inf"), float("-inf"), float("nan"), 0.0, -0.0], dtype=DT[fmt])
    pos = rng.choice(k, size=min(k, 25), replace=False)
    flat[torch.from_numpy(pos)] = specials[torch.from_numpy(rng.integers(0, 5, pos.size))]
    tiny = torch.finfo(DT[fmt]).tiny
    pos2 = rng.choice(k, size=min(k, 25), replace=False)
    flat[torch.from_numpy(pos2)] = (torch.from_numpy(rng.standard_normal(pos2.size).astype(np.float32)) * tiny
                                    * 0.3).to(DT[fmt])   # subnormals
    return t


def pin_torch_eager(orc):
    fails = []
    for fmt in ("bf16", "fp16"):
        for rows, D, seed in ((7, 40, 1), (64, 128, 2), (3, 1000, 3)):
            r = wide_values((rows, D), fmt, seed)
            u = wide_values((rows, D), fmt, seed + 10)
            g = wide_values((D,), fmt, seed + 20)
            ref = bits(r + g * u)
            got = orc.forward(bits(r), bits(u), bits(g), fmt)
            ok = same(got, ref, fmt)
            if not ok.all():
                fails.append(f"torch eager {fmt} {rows}x{D}: {int((~ok).sum())} mismatches")
    return fails


def pin_numpy_float16(orc):
    rng = np.random.default_rng(11)
    r = (rng.standard_normal((50, 64)) * 30).astype(np.float16)
    u = (rng.standard_normal((50, 64)) * 3).astype(np.float16)
    g = (rng.standard_normal(64) * 0.2).astype(np.float16)
    ref = (r + g * u).view(np.uint16)          # numpy: fp32 arithmetic, one rounding per op
    got = orc.forward(r.view(np.uint16), u.view(np.uint16), g.view(np.uint16), "fp16")
    return [] if np.array_equal(got, ref) else [f"numpy float16: {(got != ref).sum()} mismatches"]


def pin_closed_forms(orc):
    fails = []
    for fmt in ("bf16", "fp16"):
        r = wide_values((9, 33), fmt, 5)
        u = wide_values((9, 33), fmt, 6)
        one = torch.ones(33, dtype=DT[fmt])
        zero = torch.zeros(33, dtype=DT[fmt])
        if not same(orc.forward(bits(r), bits(u), bits(one), fmt), bits(r + u), fmt).all():
            fails.append(f"gate = 1 is not the single rounded sum ({fmt})")
        got0 = orc.forward(bits(r), bits(u), bits(zero), fmt)
        finite = torch.isfinite(u).numpy()
        exp0 = bits(r + zero * u)          # r, with -0 + +0 = +0 and NaN/inf * 0 = NaN
        if not same(got0[finite], exp0[finite], fmt).all():
            fails.append(f"gate = 0 does not give the residual ({fmt})")
        if not np.array_equal(got0[finite & (bits(r) != 0x8000)], bits(r)[finite & (bits(r) != 0x8000)]):
            fails.append(f"gate = 0 changed a residual ({fmt})")
    return fails


def pin_exhaustive(orc):
    """Every bf16 and fp16 bit pattern as `update`, against torch eager."""
    fails = []
    for fmt in ("bf16", "fp16"):
        allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        u = allbits.reshape(256, 256)
        for rv, gv in ((0.75, 1.5), (-3.0, 0.1), (1e-3, -7.0)):
            r = torch.full((256, 256), rv, dtype=DT[fmt])
            g = torch.full((256,), gv, dtype=DT[fmt])
            ref = bits(r + g * from_bits(u, fmt))
            got = orc.forward(bits(r), u, bits(g), fmt)
            ok = same(got, ref, fmt)
            if not ok.all():
                fails.append(f"exhaustive {fmt} r={rv} g={gv}: {int((~ok).sum())} mismatches")
    return fails


def pin_at_consistent(orc):
    r = wide_values((40, 24), "bf16", 8)
    u = wide_values((40, 24), "bf16", 9)
    g = wide_values((24,), "bf16", 10)
    full = orc.forward(bits(r), bits(u), bits(g), "bf16")
    idx = np.random.default_rng(1).integers(0, 40 * 24, 300)
    at = orc.at(bits(r), bits(u), bits(g), "bf16", idx)
    return [] if np.array_equal(at, full.reshape(-1)[idx]) else ["rga_oracle_at disagrees with forward"]


ALL_PINS = [pin_torch_eager, pin_numpy_float16, pin_closed_forms, pin_exhaustive, pin_at_consistent]


def failing_pins(orc):
    out = []
    for pin in ALL_PINS:
        try:
            out += pin(orc)
        except Exception as exc:  # noqa: BLE001 -- a crash in a mutant counts as a failed pin
            out.append(f"{pin.__name__}: {exc!r}")
    return out
