"""Pins for the fp64 oracle: checks against things other than the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` (the real library or a
deliberately broken copy built by ``test_oracle_mutations.py``) and raises
AssertionError when the oracle disagrees with

  * brute force: pure-Python loops over the definition on tiny tensors,
  * a library special case: ``torch.nn.functional.group_norm`` in float64 on
    the NCHW permutation of the same tensor, followed by
    ``torch.nn.functional.silu``,
  * closed forms (a single-element group, a two-element group, a constant
    group),
  * invariants (zero mean and var/(var+eps) second moment of the plain
    normalisation, affine invariance, permutation equivariance, batch
    independence).

The definition is the one on the sglang PR #33451 page ("FLUX.2 VAE decoder
fast path behind quality=high", section "Modifications", item 1): statistics
per (batch, group) over (N, L, C) rows, affine per channel, optional SiLU.
"""
from __future__ import annotations

import math

import numpy as np

from channels_last_groupnorm_gb300.workloads import bf16_bits_to_f32, make_case

TIGHT = 1e-12


def _close(a, b, rtol=TIGHT, atol=TIGHT, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    if not np.all(err <= bound):
        k = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: max excess at flat {k}: got {a.flat[k]!r} "
                             f"want {b.flat[k]!r}")


# --------------------------------------------------------------------------
# brute force
# --------------------------------------------------------------------------
def brute_force(x_bits, gamma, beta, G, eps, apply_silu):
    """The definition, one element at a time, in Python floats."""
    xs = bf16_bits_to_f32(x_bits).astype(np.float64)
    N, L, C = xs.shape
    Cg = C // G
    y = [[[0.0] * C for _ in range(L)] for _ in range(N)]
    mean = [[0.0] * G for _ in range(N)]
    rstd = [[0.0] * G for _ in range(N)]
    for n in range(N):
        for g in range(G):
            members = [(l, c) for l in range(L) for c in range(g * Cg, (g + 1) * Cg)]
            vals = [float(xs[n, l, c]) for (l, c) in members]
            mu = math.fsum(vals) / len(vals)
            var = math.fsum((v - mu) ** 2 for v in vals) / len(vals)
            r = 1.0 / math.sqrt(var + eps)
            mean[n][g], rstd[n][g] = mu, r
            for (l, c) in members:
                z = (float(xs[n, l, c]) - mu) * r * float(gamma[c]) + float(beta[c])
                if apply_silu:
                    z = z * (1.0 / (1.0 + math.exp(-z)))
                y[n][l][c] = z
    return np.array(y), np.array(mean), np.array(rstd)


BRUTE_CASES = [
    # (N, L, C, G, silu, seed, kind)
    (1, 1, 32, 32, True, 11, "normal"),
    (1, 2, 32, 32, False, 12, "normal"),
    (1, 3, 64, 32, True, 13, "normal"),
    (2, 5, 64, 32, True, 14, "normal"),
    (2, 3, 32, 8, False, 15, "normal"),
    (1, 5, 16, 1, True, 16, "normal"),
    (3, 2, 8, 2, True, 17, "normal"),
    (1, 7, 32, 4, True, 18, "normal"),
]


def pin_brute_force(orc):
    for (N, L, C, G, silu, seed, kind) in BRUTE_CASES:
        case = make_case(N, L, C, seed, std=1.5, mean=0.25, kind=kind)
        y, mean, rstd = orc.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, silu)
        by, bm, br = brute_force(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, silu)
        tag = f"brute N={N} L={L} C={C} G={G} silu={silu}"
        _close(mean, bm, what=tag + " mean")
        _close(rstd, br, rtol=1e-11, what=tag + " rstd")
        _close(y, by, rtol=1e-10, atol=1e-12, what=tag + " y")


# --------------------------------------------------------------------------
# library special case
# --------------------------------------------------------------------------
TORCH_CASES = [
    # (N, C, H, W, G, silu, seed, eps)
    (2, 64, 5, 7, 32, True, 21, 1e-6),
    (1, 128, 8, 8, 32, False, 22, 1e-6),
    (2, 32, 3, 3, 8, True, 23, 1e-5),
    (1, 16, 4, 4, 1, True, 24, 1e-6),
    (1, 512, 16, 16, 32, True, 25, 1e-6),
    (3, 256, 6, 10, 16, False, 26, 1e-3),
]


def torch_reference(x_bits, gamma, beta, H, W, G, eps, apply_silu):
    import torch
    import torch.nn.functional as F
    xs = torch.from_numpy(bf16_bits_to_f32(x_bits).astype(np.float64))
    N, L, C = xs.shape
    nchw = xs.reshape(N, H, W, C).permute(0, 3, 1, 2).contiguous()
    out = F.group_norm(nchw, G, torch.from_numpy(gamma.astype(np.float64)),
                       torch.from_numpy(beta.astype(np.float64)), eps)
    if apply_silu:
        out = F.silu(out)
    return out.permute(0, 2, 3, 1).reshape(N, L, C).numpy()


def pin_torch_group_norm(orc):
    for (N, C, H, W, G, silu, seed, eps) in TORCH_CASES:
        case = make_case(N, H * W, C, seed, std=2.0, mean=-0.5)
        y, _, _ = orc.forward(case["x_bits"], case["gamma"], case["beta"], G, eps, silu)
        ref = torch_reference(case["x_bits"], case["gamma"], case["beta"], H, W, G, eps, silu)
        _close(y, ref, rtol=1e-9, atol=1e-11,
               what=f"torch group_norm N={N} C={C} HxW={H}x{W} G={G} silu={silu}")


def pin_torch_offset_stress(orc):
    """Large common offset and per-channel offsets (the cancellation stress
    shape, shrunk): the two-pass fp64 statistics must still agree with
    torch's float64 GroupNorm."""
    N, C, H, W, G = 1, 512, 12, 12, 32
    case = make_case(N, H * W, C, 31, mean=4.0, std=0.25, channel_offset=1.0)
    for silu in (True, False):
        y, _, _ = orc.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, silu)
        ref = torch_reference(case["x_bits"], case["gamma"], case["beta"], H, W, G, 1e-6, silu)
        _close(y, ref, rtol=1e-9, atol=1e-11, what=f"offset stress silu={silu}")


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def pin_single_element_group(orc):
    """L = 1 and one channel per group: mean = x, var = 0, so z = beta
    exactly and rstd = 1/sqrt(eps)."""
    case = make_case(2, 1, 32, 41)
    for silu in (False, True):
        y, mean, rstd = orc.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, silu)
        b = case["beta"].astype(np.float64)
        want = b / (1.0 + np.exp(-b)) if silu else b
        _close(y, np.broadcast_to(want, y.shape), rtol=1e-15, atol=0.0,
               what=f"single-element group silu={silu}")
        _close(mean, bf16_bits_to_f32(case["x_bits"][:, 0, :]).astype(np.float64),
               rtol=0, atol=0, what="single-element mean")
        _close(rstd, np.full_like(rstd, 1.0 / math.sqrt(1e-6)), rtol=1e-15, atol=0,
               what="single-element rstd")


def pin_two_element_group(orc):
    """A group {a, b}: mean (a+b)/2, var ((a-b)/2)^2, and
    z(a) = gamma * h / sqrt(h^2 + eps) + beta with h = (a - b)/2."""
    eps = 1e-3
    rng = np.random.default_rng(42)
    for trial in range(20):
        a, b = rng.uniform(-3, 3, 2)
        # an L=2, C=G=8 tensor: each group holds one channel over two rows
        from channels_last_groupnorm_gb300.workloads import f32_to_bf16_bits
        xb = f32_to_bf16_bits(np.array([[a] * 8, [b] * 8], np.float32)).reshape(1, 2, 8)
        av, bv = bf16_bits_to_f32(xb[0, :, 0]).astype(np.float64)
        gamma = rng.uniform(0.5, 1.5, 8).astype(np.float32)
        beta = rng.normal(0, 0.1, 8).astype(np.float32)
        y, mean, rstd = orc.forward(xb, gamma, beta, 8, eps, False)
        h = (av - bv) / 2.0
        za = gamma.astype(np.float64) * h / math.sqrt(h * h + eps) + beta.astype(np.float64)
        zb = -gamma.astype(np.float64) * h / math.sqrt(h * h + eps) + beta.astype(np.float64)
        _close(y[0, 0], za, rtol=1e-13, atol=1e-14, what=f"two-element z(a) trial {trial}")
        _close(y[0, 1], zb, rtol=1e-13, atol=1e-14, what=f"two-element z(b) trial {trial}")
        _close(mean[0], np.full(8, (av + bv) / 2.0), rtol=1e-15, atol=0, what="two-element mean")
        _close(rstd[0], np.full(8, 1.0 / math.sqrt(h * h + eps)), rtol=1e-14, atol=0,
               what="two-element rstd")


def pin_constant_input(orc):
    """Every x equal: y = beta exactly (SiLU off), mean = the constant,
    rstd = 1/sqrt(eps)."""
    for value in (4.0, -1.5, 0.0):
        case = make_case(2, 9, 64, 51, mean=value, kind="constant")
        y, mean, rstd = orc.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-6, False)
        _close(y, np.broadcast_to(case["beta"].astype(np.float64), y.shape), rtol=0, atol=0,
               what=f"constant {value} y")
        _close(mean, np.full_like(mean, value), rtol=0, atol=0, what=f"constant {value} mean")
        _close(rstd, np.full_like(rstd, 1.0 / math.sqrt(1e-6)), rtol=1e-15, atol=0,
               what=f"constant {value} rstd")


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def pin_plain_normalisation_moments(orc):
    """gamma = 1, beta = 0, SiLU off: every (n, g) has output mean 0 and
    output mean square var / (var + eps), var being numpy's population
    variance of the group."""
    N, L, C, G, eps = 2, 37, 64, 8, 1e-2
    case = make_case(N, L, C, 61, mean=3.0, std=0.7)
    ones = np.ones(C, np.float32)
    zeros = np.zeros(C, np.float32)
    y, _, _ = orc.forward(case["x_bits"], ones, zeros, G, eps, False)
    xs = bf16_bits_to_f32(case["x_bits"]).astype(np.float64)
    Cg = C // G
    for n in range(N):
        for g in range(G):
            yg = y[n, :, g * Cg:(g + 1) * Cg]
            var = np.var(xs[n, :, g * Cg:(g + 1) * Cg])
            _close(yg.mean(), 0.0, rtol=0, atol=1e-13, what=f"moment mean n={n} g={g}")
            _close((yg * yg).mean(), var / (var + eps), rtol=1e-12, atol=0,
                   what=f"moment var n={n} g={g}")


def pin_affine_invariance(orc):
    """x -> 2x + 1 with eps -> 4 eps leaves the output unchanged (the
    values are on a grid where 2x + 1 is an exact bf16 number)."""
    from channels_last_groupnorm_gb300.workloads import f32_to_bf16_bits
    case = make_case(1, 23, 64, 71, kind="grid")
    xs = bf16_bits_to_f32(case["x_bits"])
    moved = f32_to_bf16_bits(2.0 * xs + 1.0)
    assert np.array_equal(bf16_bits_to_f32(moved), 2.0 * xs + 1.0)
    y0, _, _ = orc.forward(case["x_bits"], case["gamma"], case["beta"], 32, 1e-4, True)
    y1, _, _ = orc.forward(moved, case["gamma"], case["beta"], 32, 4e-4, True)
    _close(y1, y0, rtol=1e-12, atol=1e-14, what="affine invariance")


def pin_permutation_equivariance(orc):
    """Permuting positions l permutes y the same way; permuting channels
    inside each group, together with gamma and beta, permutes y the same
    way."""
    N, L, C, G = 2, 19, 64, 8
    Cg = C // G
    case = make_case(N, L, C, 81, std=1.3)
    y, m, r = orc.forward(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, True)
    rng = np.random.default_rng(82)
    pl = rng.permutation(L)
    yl, ml, rl = orc.forward(case["x_bits"][:, pl, :], case["gamma"], case["beta"], G, 1e-6, True)
    _close(yl, y[:, pl, :], rtol=1e-12, atol=1e-14, what="position permutation y")
    _close(ml, m, rtol=1e-13, atol=1e-15, what="position permutation mean")
    pc = np.concatenate([g * Cg + rng.permutation(Cg) for g in range(G)])
    yc, _, _ = orc.forward(case["x_bits"][:, :, pc], case["gamma"][pc], case["beta"][pc],
                           G, 1e-6, True)
    _close(yc, y[:, :, pc], rtol=1e-12, atol=1e-14, what="channel permutation y")


def pin_batch_independence(orc):
    """Each batch entry is normalised on its own."""
    case = make_case(3, 11, 32, 91)
    y, m, r = orc.forward(case["x_bits"], case["gamma"], case["beta"], 4, 1e-6, True)
    for n in range(3):
        yn, mn, rn = orc.forward(case["x_bits"][n:n + 1], case["gamma"], case["beta"], 4,
                                 1e-6, True)
        _close(yn[0], y[n], rtol=0, atol=0, what=f"batch {n} y")
        _close(mn[0], m[n], rtol=0, atol=0, what=f"batch {n} mean")


def pin_stats_and_sampled_apply(orc):
    """``stats`` agrees with numpy's mean / population variance per group,
    and ``apply_at`` at sampled flat indices agrees with brute force."""
    N, L, C, G = 2, 13, 64, 16
    case = make_case(N, L, C, 101, mean=1.0, std=0.9)
    mean, var, rstd = orc.stats(case["x_bits"], G, 1e-6)
    xs = bf16_bits_to_f32(case["x_bits"]).astype(np.float64)
    Cg = C // G
    for n in range(N):
        for g in range(G):
            grp = xs[n, :, g * Cg:(g + 1) * Cg]
            _close(mean[n, g], grp.mean(), rtol=1e-14, atol=1e-15, what="stats mean")
            _close(var[n, g], np.var(grp), rtol=1e-12, atol=1e-15, what="stats var")
            _close(rstd[n, g], 1.0 / math.sqrt(np.var(grp) + 1e-6), rtol=1e-12, atol=0,
                   what="stats rstd")
    by, _, _ = brute_force(case["x_bits"], case["gamma"], case["beta"], G, 1e-6, True)
    idx = np.random.default_rng(102).integers(0, N * L * C, 300)
    ys = orc.apply_at(case["x_bits"], case["gamma"], case["beta"], G, mean, rstd, True, idx)
    _close(ys, by.reshape(-1)[idx], rtol=1e-10, atol=1e-12, what="apply_at")


ALL_PINS = [
    pin_brute_force,
    pin_torch_group_norm,
    pin_torch_offset_stress,
    pin_single_element_group,
    pin_two_element_group,
    pin_constant_input,
    pin_plain_normalisation_moments,
    pin_affine_invariance,
    pin_permutation_equivariance,
    pin_batch_independence,
    pin_stats_and_sampled_apply,
]


def failing_pins(orc):
    """Names of the pins the given oracle fails (an empty list for a correct
    oracle)."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError) as exc:  # noqa: PERF203
            failed.append(f"{pin.__name__}: {str(exc)[:160]}")
    return failed
