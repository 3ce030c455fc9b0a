"""Pins of the single-head attention-block oracle (value projection,
softmax attention, output projection, residual; unfolded), shared by the pin
tests and the mutation tests: each function takes an oracle object and
returns a list of failure messages (empty = pass).

Independent references:
  * PyTorch's CPU float64 `F.linear` and `F.scaled_dot_product_attention`
    (the library routines of the definition);
  * the page's fold (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
    quality=high", section "Modifications", item 2, attention bullet):
    W' = W_o W_v, b' = W_o b_v + b_o, out = A (xn W'^T + b') + residual,
    evaluated here in float64 with numpy;
  * closed forms (q = 0: uniform attention over the keys; one key), key
    permutation and key-shift invariance, and brute force in pure Python.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from channels_last_groupnorm_gb300 import workloads as wl


def _v(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64).reshape(np.asarray(bits).shape)


def _case(S, D, seed, residual=True):
    return wl.make_attn_case(S, D, seed, residual)


def _call(o, c, **kw):
    return o.forward(c["q"], c["k"], c["xn"], c["wv"], c["bv"], c["wo"], c["bo"], c["residual"], **kw)


def _close(got, want, what, rtol=1e-11, atol=1e-11):
    if got.shape != want.shape:
        return [f"{what}: shape {got.shape} != {want.shape}"]
    err = np.abs(got - want)
    bad = err > atol + rtol * np.abs(want)
    if bad.any():
        at = np.unravel_index(int(np.argmax(err)), err.shape)
        return [f"{what}: {int(bad.sum())} of {bad.size} differ, worst at {at}: {got[at]!r} vs {want[at]!r}"]
    return []


def _torch_reference(c):
    t = lambda k: torch.from_numpy(_v(c[k]))  # noqa: E731
    q, k, xn = t("q"), t("k"), t("xn")
    v = F.linear(xn, t("wv"), t("bv"))
    o = F.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None])[0, 0]
    out = F.linear(o, t("wo"), t("bo"))
    if c["residual"] is not None:
        out = out + t("residual")
    return out.numpy()


def pin_library(o):
    """Agrees with PyTorch's float64 linear + scaled_dot_product_attention."""
    out = []
    for (S, D, seed, res) in ((7, 8, 1, True), (33, 16, 2, False), (64, 32, 3, True), (1, 4, 4, True)):
        c = _case(S, D, seed, res)
        out += _close(_call(o, c), _torch_reference(c), f"torch reference S={S} D={D}")
    return out


def pin_fold_identity(o):
    """The page's fold: the same output from the folded value weight."""
    out = []
    for (S, D, seed) in ((20, 8, 5), (40, 16, 6)):
        c = _case(S, D, seed)
        q, k, xn = _v(c["q"]), _v(c["k"]), _v(c["xn"])
        wv, bv, wo, bo = _v(c["wv"]), _v(c["bv"]), _v(c["wo"]), _v(c["bo"])
        w_f = wo @ wv
        b_f = wo @ bv + bo
        s = q @ k.T / math.sqrt(D)
        a = np.exp(s - s.max(axis=1, keepdims=True))
        a /= a.sum(axis=1, keepdims=True)
        want = a @ (xn @ w_f.T + b_f) + _v(c["residual"])
        out += _close(_call(o, c), want, f"folded evaluation S={S} D={D}", rtol=1e-10, atol=1e-10)
    return out


def pin_uniform_attention(o):
    """q = 0: every key gets weight 1/S, so out = bo + wo (mean_j v_j) + residual."""
    S, D = 9, 8
    c = _case(S, D, 7)
    c["q"] = np.zeros((S, D), np.uint16)
    v = _v(c["xn"]) @ _v(c["wv"]).T + _v(c["bv"])
    want = np.tile(_v(c["wo"]) @ v.mean(axis=0) + _v(c["bo"]), (S, 1)) + _v(c["residual"])
    return _close(_call(o, c), want, "uniform attention", rtol=1e-12, atol=1e-12)


def pin_single_key(o):
    """S = 1: the only key has weight 1, so out = wo (wv xn + bv) + bo + residual."""
    c = _case(1, 16, 8)
    want = (_v(c["wo"]) @ (_v(c["wv"]) @ _v(c["xn"])[0] + _v(c["bv"])) + _v(c["bo"]))[None] + _v(c["residual"])
    return _close(_call(o, c), want, "single key", rtol=1e-12, atol=1e-12)


def pin_key_permutation_and_shift(o):
    """Permuting the keys together with their value inputs changes nothing;
    permuting the queries permutes the output rows; adding one vector to all
    keys shifts each row's scores by a constant and changes nothing."""
    S, D = 24, 8
    c = _case(S, D, 9)
    y = _call(o, c)
    p = np.random.default_rng(1).permutation(S)
    ck = dict(c, k=np.ascontiguousarray(c["k"][p]), xn=np.ascontiguousarray(c["xn"][p]))
    out = _close(_call(o, ck), y, "key permutation", rtol=1e-11, atol=1e-11)
    cq = dict(c, q=np.ascontiguousarray(c["q"][p]), residual=np.ascontiguousarray(c["residual"][p]))
    out += _close(_call(o, cq), y[p], "query permutation", rtol=1e-12, atol=1e-12)
    # keys on a grid of 1/8 in [-4, 4] and a shift of multiples of 1/8: every
    # shifted key is exactly representable in bf16, so only the scores move
    kq = np.clip(np.round(_v(c["k"]) * 8) / 8, -4, 4).astype(np.float32)
    shift = np.array([0.5, -1.0, 0.25, 0.0, 2.0, -0.5, 1.0, 0.125], np.float32)
    k0 = wl.f32_to_bf16_bits(kq).reshape(S, D)
    k1 = wl.f32_to_bf16_bits(kq + shift).reshape(S, D)
    if not np.array_equal(_v(k1), _v(k0) + shift):
        out.append("key shift: shifted keys not exact (test set-up)")
    else:
        y0 = _call(o, dict(c, k=k0))
        out += _close(_call(o, dict(c, k=k1)), y0, "key shift", rtol=1e-9, atol=1e-9)
    return out


def pin_brute_force(o):
    """Pure-Python loops on a tiny block (S = 3, D = 2)."""
    S, D = 3, 2
    c = _case(S, D, 10)
    q, k, xn, r = (_v(c[n]).tolist() for n in ("q", "k", "xn", "residual"))
    wv, wo = _v(c["wv"]).tolist(), _v(c["wo"]).tolist()
    bv, bo = _v(c["bv"]).tolist(), _v(c["bo"]).tolist()
    v = [[bv[cc] + sum(xn[j][i] * wv[cc][i] for i in range(D)) for cc in range(D)] for j in range(S)]
    want = []
    for rr in range(S):
        s = [sum(q[rr][d] * k[j][d] for d in range(D)) / math.sqrt(D) for j in range(S)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        a = [x / sum(e) for x in e]
        oo = [sum(a[j] * v[j][cc] for j in range(S)) for cc in range(D)]
        want.append([bo[ee] + sum(oo[cc] * wo[ee][cc] for cc in range(D)) + r[rr][ee] for ee in range(D)])
    return _close(_call(o, c), np.array(want), "brute force", rtol=1e-12, atol=1e-12)


def pin_rows_and_magnitude(o):
    """The row-sampled entry equals the full one; magnitudes bound |out|
    and equal out for all-positive operands (q = k = 0, positive rest); a
    row index outside [0, S) is rejected."""
    S, D = 16, 8
    c = _case(S, D, 11)
    y, m = _call(o, c, with_mag=True)
    rows = np.array([0, 5, 15, 5])
    yr, mr = o.rows(c["q"], c["k"], c["xn"], c["wv"], c["bv"], c["wo"], c["bo"], c["residual"], rows,
                    with_mag=True)
    out = _close(yr, y[rows], "rows() vs forward()", rtol=0, atol=0)
    out += _close(mr, m[rows], "rows() magnitudes", rtol=0, atol=0)
    if np.any(m < np.abs(y) * (1 - 1e-12)):
        out.append("magnitudes below |out|")
    pos = {n: (wl.f32_to_bf16_bits(np.abs(wl.bf16_bits_to_f32(c[n]))).reshape(np.shape(c[n]))
               if c[n] is not None else None) for n in c}
    pos["q"] = np.zeros_like(c["q"])
    yp, mp = _call(o, pos, with_mag=True)
    out += _close(mp, yp, "magnitudes of positive operands", rtol=1e-12, atol=0)
    try:
        o.rows(c["q"], c["k"], c["xn"], c["wv"], c["bv"], c["wo"], c["bo"], None, np.array([S]))
        out.append("out-of-range row accepted")
    except ValueError:
        pass
    return out


ALL_PINS = [pin_library, pin_fold_identity, pin_uniform_attention, pin_single_key,
            pin_key_permutation_and_shift, pin_brute_force, pin_rows_and_magnitude]


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
