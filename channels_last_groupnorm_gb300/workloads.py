"""Seeded synthetic inputs for the GroupNorm(+SiLU) workloads.

This module holds no GroupNorm arithmetic: it draws numbers and rounds them
to bf16 bit patterns.  It is the one piece of code that both the CUDA path's
callers and the fp64 oracle's callers share, so that both sides see the very
same input bytes.

The shapes are the FLUX.2 VAE decoder GroupNorm shapes of the kernel
micro-benchmark on the sglang PR #33451 page ("FLUX.2 VAE decoder fast path
behind quality=high", section "Speedup", first table), written as (N, C, H, W)
of a channels_last tensor, plus the small 64x64 case.  GENERAL_WORKLOADS
are shapes for the generalised entry points (non-power-of-two C, 5D
channels-last input with D frames), which the pages name but do not
measure; they use the same distributions.  The value
distributions stand in for decoder activations (the pages print none):

  x     ~ N(mean, std) fp32, rounded to bf16 (round to nearest even)
  gamma ~ U(0.5, 1.5) fp32,   beta ~ N(0, 0.1) fp32
  cfg3  adds a per-channel offset U(-1, 1) to x ~ N(4, 0.25): a
        cancellation stress for the statistics.

Seeds: x = 1000 + index, gamma = 2000 + index, beta = 3000 + index, channel
offsets = 4000; numpy PCG64 (``numpy.random.default_rng``).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Values are drawn in fixed-size chunks so that the stream of numbers (and so
# every byte of the tensor) does not depend on how much memory is at hand.
_CHUNK = 1 << 24


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (round to nearest, ties to even) and
    return the 16-bit patterns.  Inputs must be finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to binary32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int          # seed index
    N: int
    C: int
    H: int
    W: int
    G: int = 32
    D: int = 1                    # frames of a 5D (N, C, D, H, W) input; 1 = 4D
    eps: float = 1e-6
    x_mean: float = 0.0
    x_std: float = 1.0
    channel_offset: float = 0.0   # half-width a of per-channel offsets U(-a, a); 0 = none
    silu_modes: tuple = (True,)
    note: str = ""
    pages_us_h200: float | None = None   # the pages' two-pass time for this shape (context)

    @property
    def L(self) -> int:
        return self.D * self.H * self.W

    @property
    def general(self) -> bool:
        """C is not a power of two: only the general entry points take it."""
        return self.C & (self.C - 1) != 0

    @property
    def elements(self) -> int:
        return self.N * self.L * self.C

    @property
    def nchw(self) -> tuple:
        return (self.N, self.C, self.H, self.W)

    def describe(self) -> dict:
        spatial = {"D": self.D} if self.D > 1 else {}
        return {"workload": self.name, "N": self.N, "C": self.C, **spatial, "H": self.H,
                "W": self.W, "G": self.G, "eps": self.eps,
                "layout": "NDHWC (channels_last_3d)" if self.D > 1 else "NHWC (channels_last)",
                "x": (f"N({self.x_mean},{self.x_std})"
                      + (f"+U(-{self.channel_offset},{self.channel_offset})[c]"
                         if self.channel_offset else "")),
                "gamma": "U(0.5,1.5)", "beta": "N(0,0.1)"}


WORKLOADS = [
    Workload("gn_silu_c128_64x64", 0, 1, 128, 64, 64,
             note="small case the oracle finishes in well under a second"),
    Workload("gn_silu_c512_128x128", 1, 1, 512, 128, 128,
             note="VAE mid-block shape", pages_us_h200=76.0),
    Workload("gn_c512_256x256_offset_stress", 2, 1, 512, 256, 256, x_mean=4.0, x_std=0.25,
             channel_offset=1.0, silu_modes=(True, False),
             note="mean 4, sigma 0.25, per-channel offsets: cancellation stress",
             pages_us_h200=121.0),
    Workload("gn_silu_c512_512x512", 3, 1, 512, 512, 512,
             note="256 MiB activation", pages_us_h200=311.1),
    Workload("gn_silu_c256_1024x1024", 4, 1, 256, 1024, 1024, x_std=2.0,
             note="512 MiB up-block shape", pages_us_h200=913.8),
    Workload("gn_silu_c128_1024x1024", 5, 1, 128, 1024, 1024, x_std=2.0,
             note="256 MiB up-block shape", pages_us_h200=307.9),
]

GENERAL_WORKLOADS = [
    Workload("gn_silu_c960_128x128", 10, 1, 960, 128, 128, note="C = 960, Cg = 30"),
    Workload("gn_silu_c320_256x256", 11, 1, 320, 256, 256, note="C = 320, Cg = 10"),
    Workload("gn_silu_c384_d8_128x128", 12, 1, 384, 128, 128, D=8,
             note="5D channels-last video latent, C = 384, Cg = 12"),
]

BY_NAME = {w.name: w for w in WORKLOADS + GENERAL_WORKLOADS}


def _normal_bits(rng: np.random.Generator, count: int, C: int, mean: float, std: float,
                 offsets: np.ndarray | None) -> np.ndarray:
    out = np.empty(count, np.uint16)
    done = 0
    while done < count:
        k = min(_CHUNK // C * C, count - done)   # whole rows; _CHUNK itself for a power-of-two C
        v = rng.standard_normal(k, dtype=np.float32)
        v *= np.float32(std)
        v += np.float32(mean)
        if offsets is not None:
            v = v.reshape(-1, C)
            v += offsets[None, :]
            v = v.reshape(-1)
        out[done:done + k] = f32_to_bf16_bits(v)
        done += k
    return out


def affine_params(index: int, C: int) -> tuple[np.ndarray, np.ndarray]:
    gamma = np.random.default_rng(2000 + index).uniform(0.5, 1.5, C).astype(np.float32)
    beta = (np.random.default_rng(3000 + index).standard_normal(C, dtype=np.float32)
            * np.float32(0.1))
    return gamma, beta


def make_inputs(w: Workload) -> dict:
    """x_bits uint16 [N, L, C] (bf16 patterns, channels innermost), gamma and
    beta float32 [C]."""
    offsets = None
    if w.channel_offset:
        offsets = np.random.default_rng(4000).uniform(
            -w.channel_offset, w.channel_offset, w.C).astype(np.float32)
    rng = np.random.default_rng(1000 + w.index)
    x = _normal_bits(rng, w.elements, w.C, w.x_mean, w.x_std, offsets)
    gamma, beta = affine_params(w.index, w.C)
    return {"x_bits": x.reshape(w.N, w.L, w.C), "gamma": gamma, "beta": beta}


def make_case(N: int, L: int, C: int, seed: int, *, mean: float = 0.0, std: float = 1.0,
              channel_offset: float = 0.0, kind: str = "normal") -> dict:
    """A seeded test case of any shape.

    kind: "normal"   x ~ N(mean, std) (+ per-channel offsets U(-a, a))
          "constant" every x equals bf16(mean)
          "grid"     x = k/8 for integers k in [-64, 64]: values whose
                     affine images 2x+1 are also exact bf16 numbers
    """
    rng = np.random.default_rng(seed)
    count = N * L * C
    if kind == "normal":
        offsets = None
        if channel_offset:
            offsets = rng.uniform(-channel_offset, channel_offset, C).astype(np.float32)
        v = rng.standard_normal(count, dtype=np.float32) * np.float32(std) + np.float32(mean)
        if offsets is not None:
            v = (v.reshape(-1, C) + offsets[None, :]).reshape(-1)
        x = f32_to_bf16_bits(v)
    elif kind == "constant":
        x = f32_to_bf16_bits(np.full(count, mean, np.float32))
    elif kind == "grid":
        k = rng.integers(-64, 65, count)
        x = f32_to_bf16_bits((k / 8.0).astype(np.float32))
    else:
        raise ValueError(f"unknown kind {kind!r}")
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = (rng.standard_normal(C, dtype=np.float32) * np.float32(0.1))
    return {"x_bits": x.reshape(N, L, C), "gamma": gamma, "beta": beta}



# ---------------------------------------------------------------------------
# residual-gate update y = residual + gate * update: the shapes the prhub
# digest of sglang PR #33823 (FLUX.2 bit-exact residual-gate fusion) names,
# (1, 512, 3072) with its H200 micro-benchmark times and the FLUX.2-dev
# 1024^2 shape (1, 4608, 6144), plus the FLUX.2-klein (D = 3072) stream at
# the same token count.  Values: residual ~ N(0, 2), update ~ N(0, 1), gate
# ~ U(-0.5, 0.5), drawn in fp32 (the caller rounds them to bf16 / fp16).
# Seeds: 5000 + index (residual), 6000 + index (update), 7000 + index (gate).
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class RgaWorkload:
    name: str
    index: int
    B: int
    S: int
    D: int
    pages_us_h200: float | None = None        # fused kernel on H200 (context)
    pages_eager_us_h200: float | None = None  # the eager pair on H200 (context)
    note: str = ""

    @property
    def rows(self) -> int:
        return self.B * self.S

    @property
    def elements(self) -> int:
        return self.rows * self.D

    def describe(self) -> dict:
        return {"workload": self.name, "shape": [self.B, self.S, self.D], "gate": [1, 1, self.D],
                "residual": "N(0,2)", "update": "N(0,1)", "gate_values": "U(-0.5,0.5)"}


RGA_WORKLOADS = [
    RgaWorkload("rga_flux2_klein_512x3072", 0, 1, 512, 3072, pages_us_h200=13.0, pages_eager_us_h200=12.1,
                note="the page's micro-benchmark shape"),
    RgaWorkload("rga_flux2_dev_4608x6144", 1, 1, 4608, 6144, note="FLUX.2-dev 1024^2 (the page's test case)"),
    RgaWorkload("rga_flux2_klein_4608x3072", 2, 1, 4608, 3072, note="FLUX.2-klein stream at 1024^2"),
]

RGA_BY_NAME = {w.name: w for w in RGA_WORKLOADS}


def make_rga_inputs(w: RgaWorkload):
    """(residual, update, gate) as float32 torch tensors, shapes [B, S, D],
    [B, S, D] and [D]."""
    import torch
    res = np.random.default_rng(5000 + w.index).standard_normal((w.B, w.S, w.D), dtype=np.float32) * np.float32(2.0)
    upd = np.random.default_rng(6000 + w.index).standard_normal((w.B, w.S, w.D), dtype=np.float32)
    gate = np.random.default_rng(7000 + w.index).uniform(-0.5, 0.5, w.D).astype(np.float32)
    return torch.from_numpy(res), torch.from_numpy(upd), torch.from_numpy(gate)


# ---------------------------------------------------------------------------
# Fused nearest-2x upsample + 3x3 conv (the decoder's up-sampler).  The pages
# name the fusion (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
# quality=high", section "Modifications", item 2) but print no shapes; these
# are the up-samplers of the FLUX.2 VAE decoder (block widths 512, 512, 256)
# for a 1024^2 decode from a 128^2 latent, plus small shapes for exhaustive
# checks.  Values: x ~ N(0, 1) (a resnet-block output), weight and bias ~
# U(-b, b) with b = 1/sqrt(9 Cin) (PyTorch's default Conv2d initialisation),
# drawn in fp32 and rounded to bf16.
# Seeds: 8000 + index (x), 9000 + index (weight), 9500 + index (bias).
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class UpconvWorkload:
    name: str
    index: int
    N: int
    H: int          # input height (the output is 2H x 2W)
    W: int
    Cin: int
    Cout: int
    bias: bool = True
    note: str = ""

    @property
    def out_pixels(self) -> int:
        return self.N * 4 * self.H * self.W

    @property
    def flops(self) -> int:
        """Multiply-adds x 2 of the folded evaluation: 4 taps per output."""
        return 2 * self.out_pixels * self.Cout * 4 * self.Cin

    def describe(self) -> dict:
        return {"workload": self.name, "x": [self.N, self.H, self.W, self.Cin],
                "y": [self.N, 2 * self.H, 2 * self.W, self.Cout], "bias": self.bias,
                "x_values": "N(0,1)", "weight_values": "U(-1/sqrt(9Cin), 1/sqrt(9Cin))"}


UPCONV_WORKLOADS = [
    UpconvWorkload("upconv_c64_co128_16x16", 0, 1, 16, 16, 64, 128, note="small, full oracle"),
    UpconvWorkload("upconv_c512_128x128", 1, 1, 128, 128, 512, 512,
                   note="FLUX.2 decoder up-block 0 at 1024^2 (128^2 -> 256^2)"),
    UpconvWorkload("upconv_c512_256x256", 2, 1, 256, 256, 512, 512,
                   note="FLUX.2 decoder up-block 1 at 1024^2 (256^2 -> 512^2)"),
    UpconvWorkload("upconv_c256_512x512", 3, 1, 512, 512, 256, 256,
                   note="FLUX.2 decoder up-block 2 at 1024^2 (512^2 -> 1024^2)"),
]

UPCONV_BY_NAME = {w.name: w for w in UPCONV_WORKLOADS}


def make_upconv_case(N: int, H: int, W: int, Cin: int, Cout: int, index: int,
                     bias: bool = True) -> dict:
    """bf16 bit patterns: x [N, H, W, Cin], weight [Cout, Cin, 3, 3] and
    bias [Cout] (None without bias)."""
    b = 1.0 / np.sqrt(9.0 * Cin)
    x = np.random.default_rng(8000 + index).standard_normal((N, H, W, Cin), dtype=np.float32)
    w = np.random.default_rng(9000 + index).uniform(-b, b, (Cout, Cin, 3, 3)).astype(np.float32)
    out = {"x_bits": f32_to_bf16_bits(x).reshape(N, H, W, Cin),
           "w_bits": f32_to_bf16_bits(w).reshape(Cout, Cin, 3, 3), "bias_bits": None}
    if bias:
        bb = np.random.default_rng(9500 + index).uniform(-b, b, Cout).astype(np.float32)
        out["bias_bits"] = f32_to_bf16_bits(bb)
    return out


def make_upconv_inputs(w: UpconvWorkload) -> dict:
    return make_upconv_case(w.N, w.H, w.W, w.Cin, w.Cout, w.index, w.bias)


# ---------------------------------------------------------------------------
# Single-head attention of the VAE mid-block with the output projection
# folded into the value projection (sglang PR #33451, "FLUX.2 VAE decoder
# fast path behind quality=high", section "Modifications", item 2, attention
# bullet).  Width D = 512 (one head of the decoder's 512 channels); S = the
# latent's pixel count: 64^2 = 4096 for a 512^2 decode, 128^2 = 16384 for
# 1024^2, plus a small full-oracle case.  Values: q, k, xn (the GroupNorm
# output) and residual ~ N(0, 1); the value / output projection weights and
# biases ~ U(-b, b), b = 1/sqrt(D) (PyTorch's default Linear initialisation),
# drawn in fp32 and rounded to bf16.
# Seeds: 10000 + index (q), 11000 (k), 12000 (xn), 13000 (residual),
# 14000 (wv), 14500 (bv), 15000 (wo), 15500 (bo).
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class AttnWorkload:
    name: str
    index: int
    S: int
    D: int = 512
    residual: bool = True
    note: str = ""

    @property
    def flops(self) -> int:
        """Multiply-adds x 2 of the folded evaluation: the value projection,
        the scores, and the attention-weighted sum."""
        return 2 * self.S * self.D * self.D + 4 * self.S * self.S * self.D

    def describe(self) -> dict:
        return {"workload": self.name, "S": self.S, "D": self.D, "heads": 1, "residual": self.residual,
                "values": "q, k, xn, residual ~ N(0,1); W, b ~ U(-1/sqrt(D), 1/sqrt(D))"}


ATTN_WORKLOADS = [
    AttnWorkload("attn_s256_d512", 0, 256, note="small, full oracle"),
    AttnWorkload("attn_s4096_d512", 1, 4096, note="FLUX.2 VAE mid-block at a 512^2 decode (64^2 latent)"),
    AttnWorkload("attn_s16384_d512", 2, 16384, note="FLUX.2 VAE mid-block at a 1024^2 decode (128^2 latent)"),
]

ATTN_BY_NAME = {w.name: w for w in ATTN_WORKLOADS}


def make_attn_case(S: int, D: int, index: int, residual: bool = True) -> dict:
    """bf16 bit patterns: q, k, xn, residual [S, D]; wv, wo [D, D] (Linear
    layout [out][in]); bv, bo [D].  residual is None when not asked for."""
    b = 1.0 / np.sqrt(D)

    def normal(seed, shape):
        return f32_to_bf16_bits(np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)).reshape(shape)

    def uniform(seed, shape):
        v = np.random.default_rng(seed).uniform(-b, b, shape).astype(np.float32)
        return f32_to_bf16_bits(v).reshape(shape)
    out = {"q": normal(10000 + index, (S, D)), "k": normal(11000 + index, (S, D)),
           "xn": normal(12000 + index, (S, D)),
           "residual": normal(13000 + index, (S, D)) if residual else None,
           "wv": uniform(14000 + index, (D, D)), "bv": uniform(14500 + index, (D,)),
           "wo": uniform(15000 + index, (D, D)), "bo": uniform(15500 + index, (D,))}
    return out


def make_attn_inputs(w: AttnWorkload) -> dict:
    return make_attn_case(w.S, w.D, w.index, w.residual)
