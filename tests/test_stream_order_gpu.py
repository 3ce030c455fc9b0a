"""Calls chained on one stream read what the call before them wrote.

The cluster, fused and residual-gate kernels are launched with programmatic
stream serialization: their CTAs may start while the kernel ahead of them in
the stream is still running, and must not touch global memory before that
kernel has finished.  Each test here chains calls whose input is the previous
call's output, in a buffer first filled with NaN, and checks every result
against the oracle applied to the previous call's output as it ended up.  A
call that read its input early would see NaN (or a half-written tensor) and
fail the comparison.  The first chain puts a 128 MiB fused call ahead of a
cluster call on its first rows: the fused kernel's second pass walks its
pieces in reverse, so those rows are among the last it writes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from channels_last_groupnorm_gb300 import build as gnbuild
from channels_last_groupnorm_gb300 import gnsilu as gs
from tests import gpu_util as gu
from tests import rga_pins as rp

pytestmark = pytest.mark.gpu

G, EPS = 32, 1e-6


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gnbuild.build()
    gs.lib()
    yield
    gu.assert_clean_device()


def seeded(shape, seed, scale=1.0, offset=0.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, device="cuda", generator=g) * scale + offset).to(torch.bfloat16)


def affine(C, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    gamma = torch.rand(C, device="cuda", generator=g) + 0.5
    beta = torch.randn(C, device="cuda", generator=g) * 0.2
    return gamma, beta


def gn_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_gn(y, x_final, gamma, beta, what):
    """y (bf16, on the device) against the oracle's GroupNorm + SiLU of x as it ended up."""
    y_ref, _, _ = oracle.forward(gn_bits(x_final), gamma.cpu().numpy(), beta.cpu().numpy(), G, EPS, True)
    gu.check_y(gu.bf16_to_f64(y), y_ref, what)


def nan_like(x):
    return torch.full_like(x, float("nan"))


@pytest.mark.parametrize("rep", range(3))
def test_cluster_call_reads_the_rows_a_fused_call_writes_last(rep):
    N, L, C, head = 1, 262144, 512, 16384
    assert gs.gn_silu_pick_variant(N, L, C, G) == gs.VARIANT_FUSED
    assert gs.gn_silu_pick_variant(N, head, C, G) == gs.VARIANT_CLUSTER
    x1 = seeded((N, L, C), 100 + rep, scale=2.0, offset=0.5)
    gamma, beta = affine(C, 200 + rep)
    y1 = nan_like(x1)
    y2 = nan_like(x1[:, :head])
    torch.cuda.synchronize()
    assert gs.gn_silu_rows(x1, gamma, beta, G=G, eps=EPS, out=y1) is not None
    assert gs.gn_silu_rows(y1[:, :head], gamma, beta, G=G, eps=EPS, out=y2) is not None
    torch.cuda.synchronize()
    assert not torch.isnan(y1.float()).any(), "the fused call left outputs unwritten"
    check_gn(y2, y1[:, :head], gamma, beta, f"cluster after fused, rep {rep}")


@pytest.mark.parametrize("rep", range(3))
def test_fused_call_reads_the_rows_a_cluster_call_wrote(rep):
    N, L, C, head = 1, 65536, 512, 16384
    assert gs.gn_silu_pick_variant(N, L, C, G) == gs.VARIANT_FUSED
    x0 = seeded((N, head, C), 300 + rep)
    gamma, beta = affine(C, 400 + rep)
    # the fused call's input: random rows, the first `head` of them NaN until
    # the cluster call writes its output there
    x1 = seeded((N, L, C), 500 + rep, scale=0.5)
    x1[:, :head] = float("nan")
    y1 = nan_like(x1)
    torch.cuda.synchronize()
    assert gs.gn_silu_rows(x0, gamma, beta, G=G, eps=EPS, out=x1[:, :head]) is not None
    assert gs.gn_silu_rows(x1, gamma, beta, G=G, eps=EPS, out=y1) is not None
    torch.cuda.synchronize()
    assert not torch.isnan(x1.float()).any(), "the cluster call left outputs unwritten"
    check_gn(y1, x1, gamma, beta, f"fused after cluster, rep {rep}")


@pytest.mark.parametrize("rep", range(3))
def test_residual_gate_and_cluster_calls_read_each_others_output(rep):
    N, L, C = 1, 4096, 512
    assert gs.gn_silu_pick_variant(N, L, C, G) == gs.VARIANT_CLUSTER
    x0 = seeded((N, L, C), 600 + rep)
    gamma, beta = affine(C, 700 + rep)
    residual = seeded((N, L, C), 800 + rep)
    gate = seeded((C,), 900 + rep, scale=0.5)
    h = nan_like(x0)   # GroupNorm output, the update of the residual-gate call
    r = nan_like(x0)   # residual-gate output, the input of the second GroupNorm call
    y = nan_like(x0)
    torch.cuda.synchronize()
    assert gs.gn_silu_rows(x0, gamma, beta, G=G, eps=EPS, out=h) is not None
    assert gs.residual_gate_add(residual, h, gate, out=r) is not None
    assert gs.gn_silu_rows(r, gamma, beta, G=G, eps=EPS, out=y) is not None
    torch.cuda.synchronize()
    check_gn(h, x0, gamma, beta, f"first GroupNorm, rep {rep}")
    want = oracle.rga().forward(rp.bits(residual.cpu().reshape(-1, C)), rp.bits(h.cpu().reshape(-1, C)),
                                rp.bits(gate.cpu()), "bf16")
    ok = rp.same(rp.bits(r.cpu().reshape(-1, C)), want, "bf16")
    assert ok.all(), f"residual-gate after GroupNorm, rep {rep}: {int((~ok).sum())} outputs differ"
    check_gn(y, r, gamma, beta, f"GroupNorm after residual-gate, rep {rep}")


def attn_check(got, ref, mag, what):
    # the bound of the attention parity tests
    err = np.abs(got - ref)
    bound = 2.0 ** -6 * mag + 2.0 ** -7 * np.abs(ref)
    assert not (err > bound).any(), f"{what}: {int((err > bound).sum())} of {err.size} outside the bound"


@pytest.mark.parametrize("schedule", [gs.ATTN_ONE_PASS, gs.ATTN_STORED_WEIGHTS], ids=["one_pass", "stored_weights"])
def test_attention_reads_q_and_k_written_just_before(schedule):
    """q from a GroupNorm call and k from a residual-gate call, each into a
    NaN-filled buffer right before the attention call: the one-pass kernel's
    score side reads q and k without waiting itself, so this also checks that
    it cannot start before everything ahead of the value-row GEMM is done."""
    from channels_last_groupnorm_gb300 import workloads as wl

    S, D = 1024, 512
    c = wl.make_attn_case(S, D, 77, True)
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(torch.bfloat16)
    wf, bf = gs.attn_fold(dev(c["wv"]), dev(c["bv"]), dev(c["wo"]), dev(c["bo"]))
    x0 = seeded((1, S, D), 1000)
    gamma, beta = affine(D, 1001)
    residual2 = seeded((S, D), 1002)
    update = seeded((S, D), 1003)
    gate = seeded((D,), 1004, scale=0.5)
    q = nan_like(x0)
    k = torch.full((S, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    xn, res = dev(c["xn"]), dev(c["residual"])
    torch.cuda.synchronize()
    assert gs.gn_silu_rows(x0, gamma, beta, G=G, eps=EPS, out=q) is not None
    assert gs.residual_gate_add(residual2, update, gate, out=k) is not None
    y = gs.attention_folded(q[0], k, xn, wf, bf, residual=res, schedule=schedule)
    assert y is not None
    torch.cuda.synchronize()
    assert gs.gn_device_status(False) == 0
    qb, kb = gn_bits(q[0]), gn_bits(k)
    assert not np.isnan(gu.bf16_to_f64(q)).any() and not np.isnan(gu.bf16_to_f64(k)).any()
    ref, mag = oracle.attn().forward(qb, kb, c["xn"], c["wv"], c["bv"], c["wo"], c["bo"], c["residual"],
                                     with_mag=True)
    attn_check(y.float().cpu().numpy().astype(np.float64), ref, mag, f"attention after GroupNorm / residual-gate")
