"""Spatial split of one GroupNorm across ranks, simulated on the CPU: each
of two or three gloo ranks takes a slice of the rows, computes its partial
(count, mean, M2) per (n, g) with the fp64 oracle, and the exchange step
(channels_last_groupnorm_gb300.spatial) must reproduce the statistics of
the whole tensor on every rank."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from channels_last_groupnorm_gb300 import spatial
from channels_last_groupnorm_gb300 import workloads as wl

N, L, C, G = 2, 997, 64, 8     # ragged: the row split is uneven


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _slices(world):
    cuts = np.linspace(0, L, world + 1).round().astype(int)
    cuts[1] = 1 if world > 1 else cuts[1]          # rank 0 gets a single row
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        case = wl.make_case(N, L, C, seed=77, mean=3.0, std=0.5, channel_offset=1.0)
        lo, hi = _slices(world)[rank]
        part = np.ascontiguousarray(case["x_bits"][:, lo:hi])
        mean, var, _ = oracle.stats(part, G, 1e-6)
        count = np.full((N, G), (hi - lo) * (C // G), np.float64)
        n, m, m2 = spatial.allgather_combine(count, mean, var * count)
        out[rank] = (n.tolist(), m.tolist(), m2.tolist())
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
@pytest.mark.parametrize("world", [2, 3])
def test_split_rows_reproduce_whole_tensor_statistics(world):
    import oracle
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                       join=True)
    results = [out[r] for r in range(world)]
    for r in range(1, world):
        assert results[r] == results[0], "ranks disagree"
    n, m, m2 = (np.array(v) for v in results[0])
    case = wl.make_case(N, L, C, seed=77, mean=3.0, std=0.5, channel_offset=1.0)
    mean_ref, var_ref, rstd_ref = oracle.stats(case["x_bits"], G, 1e-6)
    assert np.all(n == L * (C // G))
    mean, var, rstd = spatial.finalize(n, m, m2, 1e-6)
    np.testing.assert_allclose(mean, mean_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(var, var_ref, rtol=1e-10)
    np.testing.assert_allclose(rstd, rstd_ref, rtol=1e-10)


def test_chan_merge_matches_numpy_on_random_parts():
    rng = np.random.default_rng(3)
    data = rng.standard_normal(1000) * 2.0 + 5.0
    cuts = [0, 1, 7, 300, 301, 1000]
    counts, means, m2s = [], [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = data[a:b]
        counts.append(len(part))
        means.append(part.mean())
        m2s.append(((part - part.mean()) ** 2).sum())
    counts.append(0)          # an empty part changes nothing
    means.append(123.0)
    m2s.append(456.0)
    n, m, m2 = spatial.chan_merge(np.array(counts)[:, None], np.array(means)[:, None],
                                  np.array(m2s)[:, None])
    assert n[0] == 1000
    assert abs(m[0] - data.mean()) < 1e-12
    assert abs(m2[0] - ((data - data.mean()) ** 2).sum()) < 1e-9
