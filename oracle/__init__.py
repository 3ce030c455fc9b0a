"""fp64 CPU oracle for channels-last GroupNorm (+SiLU) -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this package.  The CUDA library and its
Python binding never import it; the two share no code.

The arithmetic lives in ``gn_oracle.c`` (plain C, fp64, OpenMP over the
(n, g) groups), which writes out the definition given by the sglang PR
#33451 page ("FLUX.2 VAE decoder fast path behind quality=high", section
"Modifications", item 1): per-(batch, group) mean and biased variance over
(N, L, C) rows with C innermost, rstd = 1/sqrt(var + eps), the per-channel
affine, then SiLU if requested.  This module only compiles that file with
gcc and marshals numpy arrays through ctypes.

The package also holds the oracle of the residual-gate update
``y = residual + gate * update`` in half precision (``rga_oracle.c``; the
prhub digest of sglang PR #33823, FLUX.2 bit-exact residual-gate fusion),
which writes out the two roundings of the eager evaluation; ``rga()``
returns it.  ``upconv()`` returns the oracle of the decoder's fused
nearest-2x upsample + 3x3 convolution (``upconv_oracle.c``; the sglang PR
#33451 page, section "Modifications", item 2), which evaluates the upsample
and the convolution as defined, in fp64.  ``attn()`` returns the oracle of
the decoder's single-head attention block with its value and output
projections (``attn_oracle.c``; same page, item 2, attention bullet),
evaluated unfolded, in fp64.

Parity pins: the oracle is checked against brute force on tiny tensors, a
library special case (``torch.nn.functional.group_norm`` in float64), closed
forms and invariants in ``tests/test_oracle_pins.py``; every exported
function is pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gn_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libgn_oracle.so")

# -ffp-contract=off keeps gcc from fusing a*b+c into an FMA (it does so by
# default on aarch64), so x86 and Arm hosts round identically.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math"]

_lock = threading.Lock()
_default = None


def build(source: str = SOURCE, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile ``source`` into the shared library ``out`` (gcc + OpenMP)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(source)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, source, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


_i64 = ctypes.c_int64
_p = ctypes.c_void_p


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a
    deliberately broken copy built by the mutation tests)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.gn_oracle_stats.argtypes = [_p, _i64, _i64, _i64, _i64, ctypes.c_double,
                                        _p, _p, _p, ctypes.c_int]
        lib.gn_oracle_stats.restype = ctypes.c_int
        lib.gn_oracle_forward.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, ctypes.c_double,
                                          ctypes.c_int, _p, _p, _p, ctypes.c_int]
        lib.gn_oracle_forward.restype = ctypes.c_int
        lib.gn_oracle_apply_at.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _p, _p,
                                           ctypes.c_int, _p, _i64, _p, ctypes.c_int]
        lib.gn_oracle_apply_at.restype = ctypes.c_int
        lib.gn_oracle_max_threads.argtypes = []
        lib.gn_oracle_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _prep(x_bits, gamma=None, beta=None):
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        if x_bits.ndim != 3:
            raise ValueError("x_bits must be [N, L, C] bf16 bit patterns (uint16)")
        out = [x_bits]
        for v in (gamma, beta):
            if v is not None:
                out.append(np.ascontiguousarray(v, dtype=np.float32))
        return out

    def max_threads(self) -> int:
        return int(self.lib.gn_oracle_max_threads())

    # -- entry points ------------------------------------------------------
    def stats(self, x_bits, G: int, eps: float, nthreads: int = 0):
        """Return (mean, var, rstd), each float64 [N, G]."""
        (x_bits,) = self._prep(x_bits)
        N, L, C = x_bits.shape
        mean = np.empty((N, G), np.float64)
        var = np.empty((N, G), np.float64)
        rstd = np.empty((N, G), np.float64)
        rc = self.lib.gn_oracle_stats(x_bits.ctypes.data, N, L, C, G, float(eps),
                                      mean.ctypes.data, var.ctypes.data, rstd.ctypes.data,
                                      int(nthreads))
        if rc != 0:
            raise ValueError(f"gn_oracle_stats rejected its arguments (rc={rc})")
        return mean, var, rstd

    def forward(self, x_bits, gamma, beta, G: int, eps: float, apply_silu: bool,
                nthreads: int = 0):
        """Return (y float64 [N, L, C], mean float64 [N, G], rstd float64 [N, G])."""
        x_bits, gamma, beta = self._prep(x_bits, gamma, beta)
        N, L, C = x_bits.shape
        if gamma.shape != (C,) or beta.shape != (C,):
            raise ValueError("gamma and beta must have shape [C]")
        y = np.empty((N, L, C), np.float64)
        mean = np.empty((N, G), np.float64)
        rstd = np.empty((N, G), np.float64)
        rc = self.lib.gn_oracle_forward(x_bits.ctypes.data, gamma.ctypes.data,
                                        beta.ctypes.data, N, L, C, G, float(eps),
                                        int(bool(apply_silu)), y.ctypes.data,
                                        mean.ctypes.data, rstd.ctypes.data, int(nthreads))
        if rc != 0:
            raise ValueError(f"gn_oracle_forward rejected its arguments (rc={rc})")
        return y, mean, rstd

    def apply_at(self, x_bits, gamma, beta, G: int, mean, rstd, apply_silu: bool,
                 flat_index, nthreads: int = 0):
        """y (float64) at the given flat indices of the [N, L, C] tensor."""
        x_bits, gamma, beta = self._prep(x_bits, gamma, beta)
        N, L, C = x_bits.shape
        mean = np.ascontiguousarray(mean, np.float64)
        rstd = np.ascontiguousarray(rstd, np.float64)
        idx = np.ascontiguousarray(flat_index, np.int64)
        y = np.empty(idx.shape, np.float64)
        rc = self.lib.gn_oracle_apply_at(x_bits.ctypes.data, gamma.ctypes.data,
                                         beta.ctypes.data, N, L, C, G, mean.ctypes.data,
                                         rstd.ctypes.data, int(bool(apply_silu)),
                                         idx.ctypes.data, idx.size, y.ctypes.data,
                                         int(nthreads))
        if rc != 0:
            raise ValueError(f"gn_oracle_apply_at rejected its arguments (rc={rc})")
        return y


def get() -> Oracle:
    """The oracle built from ``gn_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def stats(*a, **k):
    return get().stats(*a, **k)


def forward(*a, **k):
    return get().forward(*a, **k)


def apply_at(*a, **k):
    return get().apply_at(*a, **k)


# ---------------------------------------------------------------------------
# residual-gate update oracle (rga_oracle.c): y = residual + gate * update in
# half precision with the two roundings of the eager evaluation
# ---------------------------------------------------------------------------
RGA_SOURCE = os.path.join(_HERE, "rga_oracle.c")
RGA_LIB_PATH = os.path.join(BUILD_DIR, "librga_oracle.so")
FMT = {"bf16": 0, "fp16": 1}
_rga_default = None


class RgaOracle:
    """ctypes view of one compiled residual-gate oracle library."""

    def __init__(self, lib_path: str):
        self.lib = ctypes.CDLL(lib_path)
        f = self.lib.rga_oracle_forward
        f.restype = ctypes.c_int
        f.argtypes = [_p, _p, _p, _p, _i64, _i64, ctypes.c_int]
        f = self.lib.rga_oracle_at
        f.restype = ctypes.c_int
        f.argtypes = [_p, _p, _p, _i64, _i64, ctypes.c_int, _p, _i64, _p]

    @staticmethod
    def _bits(a):
        return np.ascontiguousarray(a).view(np.uint16)

    def forward(self, residual_bits, update_bits, gate_bits, fmt: str):
        """uint16 [rows, D] output bits for uint16 [rows, D] residual / update
        bits and a uint16 [D] gate row."""
        r = self._bits(residual_bits)
        u = self._bits(update_bits)
        g = self._bits(gate_bits).reshape(-1)
        rows, D = r.shape
        if u.shape != (rows, D) or g.shape != (D,):
            raise ValueError("residual/update must be [rows, D] and gate [D]")
        out = np.empty((rows, D), np.uint16)
        rc = self.lib.rga_oracle_forward(r.ctypes.data, u.ctypes.data, g.ctypes.data, out.ctypes.data,
                                         rows, D, FMT[fmt])
        if rc != 0:
            raise ValueError(f"rga_oracle_forward rejected its arguments (rc={rc})")
        return out

    def at(self, residual_bits, update_bits, gate_bits, fmt: str, flat_index):
        """Output bits at the given flat indices of the [rows, D] tensors."""
        r = self._bits(residual_bits)
        u = self._bits(update_bits)
        g = self._bits(gate_bits).reshape(-1)
        rows, D = r.shape
        idx = np.ascontiguousarray(flat_index, np.int64)
        out = np.empty(idx.shape, np.uint16)
        rc = self.lib.rga_oracle_at(r.ctypes.data, u.ctypes.data, g.ctypes.data, rows, D, FMT[fmt],
                                    idx.ctypes.data, idx.size, out.ctypes.data)
        if rc != 0:
            raise ValueError(f"rga_oracle_at rejected its arguments (rc={rc})")
        return out


def build_rga(source: str = RGA_SOURCE, out: str = RGA_LIB_PATH, force: bool = False) -> str:
    return build(source=source, out=out, force=force)


def rga() -> RgaOracle:
    """The residual-gate oracle built from ``rga_oracle.c``."""
    global _rga_default
    with _lock:
        if _rga_default is None:
            _rga_default = RgaOracle(build_rga())
        return _rga_default


# ---------------------------------------------------------------------------
# fused nearest-2x upsample + 3x3 conv oracle (upconv_oracle.c): the two
# steps written out as defined, fp64, unrounded output
# ---------------------------------------------------------------------------
UPCONV_SOURCE = os.path.join(_HERE, "upconv_oracle.c")
UPCONV_LIB_PATH = os.path.join(BUILD_DIR, "libupconv_oracle.so")
_upconv_default = None


class UpconvOracle:
    """ctypes view of one compiled upsample+conv oracle library."""

    def __init__(self, lib_path: str):
        self.lib = ctypes.CDLL(lib_path)
        f = self.lib.upconv_oracle_forward
        f.restype = ctypes.c_int
        f.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _p, _p]
        f = self.lib.upconv_oracle_at
        f.restype = ctypes.c_int
        f.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _p, _i64, _p, _p]

    @staticmethod
    def _args(x_bits, w_bits, bias_bits):
        x = np.ascontiguousarray(x_bits).view(np.uint16)
        w = np.ascontiguousarray(w_bits).view(np.uint16)
        if x.ndim != 4 or w.ndim != 4 or w.shape[2:] != (3, 3) or w.shape[1] != x.shape[3]:
            raise ValueError("x must be [N, H, W, Cin] and w [Cout, Cin, 3, 3] bf16 bits")
        b = None
        if bias_bits is not None:
            b = np.ascontiguousarray(bias_bits).view(np.uint16).reshape(-1)
            if b.shape != (w.shape[0],):
                raise ValueError("bias must be [Cout] bf16 bits")
        return x, w, b

    def forward(self, x_bits, w_bits, bias_bits=None, with_abs: bool = False):
        """y float64 [N, 2H, 2W, Cout] (and the absolute-term sums if asked)."""
        x, w, b = self._args(x_bits, w_bits, bias_bits)
        N, H, W, Cin = x.shape
        Cout = w.shape[0]
        y = np.empty((N, 2 * H, 2 * W, Cout), np.float64)
        a = np.empty_like(y) if with_abs else None
        rc = self.lib.upconv_oracle_forward(x.ctypes.data, w.ctypes.data,
                                            None if b is None else b.ctypes.data,
                                            N, H, W, Cin, Cout, y.ctypes.data,
                                            None if a is None else a.ctypes.data)
        if rc != 0:
            raise ValueError(f"upconv_oracle_forward rejected its arguments (rc={rc})")
        return (y, a) if with_abs else y

    def at(self, x_bits, w_bits, bias_bits, flat_index, with_abs: bool = False):
        """y (and the absolute-term sums) at flat indices of [N, 2H, 2W, Cout]."""
        x, w, b = self._args(x_bits, w_bits, bias_bits)
        N, H, W, Cin = x.shape
        Cout = w.shape[0]
        idx = np.ascontiguousarray(flat_index, np.int64)
        y = np.empty(idx.shape, np.float64)
        a = np.empty_like(y) if with_abs else None
        rc = self.lib.upconv_oracle_at(x.ctypes.data, w.ctypes.data,
                                       None if b is None else b.ctypes.data,
                                       N, H, W, Cin, Cout, idx.ctypes.data, idx.size,
                                       y.ctypes.data, None if a is None else a.ctypes.data)
        if rc != 0:
            raise ValueError(f"upconv_oracle_at rejected its arguments (rc={rc})")
        return (y, a) if with_abs else y


def build_upconv(source: str = UPCONV_SOURCE, out: str = UPCONV_LIB_PATH,
                 force: bool = False) -> str:
    return build(source=source, out=out, force=force)


def upconv() -> UpconvOracle:
    """The upsample+conv oracle built from ``upconv_oracle.c``."""
    global _upconv_default
    with _lock:
        if _upconv_default is None:
            _upconv_default = UpconvOracle(build_upconv())
        return _upconv_default


# ---------------------------------------------------------------------------
# single-head attention block oracle (attn_oracle.c): value projection,
# softmax attention, output projection (+ residual), unfolded, fp64
# ---------------------------------------------------------------------------
ATTN_SOURCE = os.path.join(_HERE, "attn_oracle.c")
ATTN_LIB_PATH = os.path.join(BUILD_DIR, "libattn_oracle.so")
_attn_default = None


class AttnOracle:
    """ctypes view of one compiled attention oracle library."""

    def __init__(self, lib_path: str):
        self.lib = ctypes.CDLL(lib_path)
        f = self.lib.attn_oracle_forward
        f.restype = ctypes.c_int
        f.argtypes = [_p] * 8 + [_i64, _i64, _p, _p]
        f = self.lib.attn_oracle_rows
        f.restype = ctypes.c_int
        f.argtypes = [_p] * 8 + [_i64, _i64, _p, _i64, _p, _p]

    @staticmethod
    def _args(q, k, xn, wv, bv, wo, bo, residual):
        u = lambda a: np.ascontiguousarray(a).view(np.uint16)  # noqa: E731
        q, k, xn, wv, bv, wo, bo = (u(a) for a in (q, k, xn, wv, bv, wo, bo))
        S, D = q.shape
        if k.shape != (S, D) or xn.shape != (S, D) or wv.shape != (D, D) or wo.shape != (D, D):
            raise ValueError("q, k, xn must be [S, D] and wv, wo [D, D] bf16 bits")
        bv, bo = bv.reshape(-1), bo.reshape(-1)
        if bv.shape != (D,) or bo.shape != (D,):
            raise ValueError("bv, bo must be [D] bf16 bits")
        r = None
        if residual is not None:
            r = u(residual)
            if r.shape != (S, D):
                raise ValueError("residual must be [S, D] bf16 bits")
        return q, k, xn, wv, bv, wo, bo, r, S, D

    def forward(self, q, k, xn, wv, bv, wo, bo, residual=None, with_mag: bool = False):
        """out float64 [S, D] (and the magnitudes if asked)."""
        q, k, xn, wv, bv, wo, bo, r, S, D = self._args(q, k, xn, wv, bv, wo, bo, residual)
        out = np.empty((S, D), np.float64)
        mag = np.empty_like(out) if with_mag else None
        rc = self.lib.attn_oracle_forward(q.ctypes.data, k.ctypes.data, xn.ctypes.data, wv.ctypes.data,
                                          bv.ctypes.data, wo.ctypes.data, bo.ctypes.data,
                                          None if r is None else r.ctypes.data, S, D, out.ctypes.data,
                                          None if mag is None else mag.ctypes.data)
        if rc != 0:
            raise ValueError(f"attn_oracle_forward rejected its arguments (rc={rc})")
        return (out, mag) if with_mag else out

    def rows(self, q, k, xn, wv, bv, wo, bo, residual, rows, with_mag: bool = False):
        """out (and magnitudes) for the given query rows, float64 [len(rows), D]."""
        q, k, xn, wv, bv, wo, bo, r, S, D = self._args(q, k, xn, wv, bv, wo, bo, residual)
        idx = np.ascontiguousarray(rows, np.int64)
        out = np.empty((idx.size, D), np.float64)
        mag = np.empty_like(out) if with_mag else None
        rc = self.lib.attn_oracle_rows(q.ctypes.data, k.ctypes.data, xn.ctypes.data, wv.ctypes.data,
                                       bv.ctypes.data, wo.ctypes.data, bo.ctypes.data,
                                       None if r is None else r.ctypes.data, S, D, idx.ctypes.data, idx.size,
                                       out.ctypes.data, None if mag is None else mag.ctypes.data)
        if rc != 0:
            raise ValueError(f"attn_oracle_rows rejected its arguments (rc={rc})")
        return (out, mag) if with_mag else out


def build_attn(source: str = ATTN_SOURCE, out: str = ATTN_LIB_PATH, force: bool = False) -> str:
    return build(source=source, out=out, force=force)


def attn() -> AttnOracle:
    """The attention-block oracle built from ``attn_oracle.c``."""
    global _attn_default
    with _lock:
        if _attn_default is None:
            _attn_default = AttnOracle(build_attn())
        return _attn_default
