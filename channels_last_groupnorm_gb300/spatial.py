"""Statistics combine for a spatial split of one GroupNorm across ranks.

When the rows (L = H * W positions) of one image are cut across ranks, every
rank can run pass 1 on its own rows, but the per-(n, g) statistics span the
whole image, so the ranks must exchange their partial statistics once
before pass 2.  This module holds that host-side exchange step: each rank
contributes, per (n, g), the element count, the mean and the sum of squared
deviations M2 of its rows; the triples of all ranks are all-gathered and
merged with Chan's parallel formula in rank order, so every rank obtains
bit-identical statistics regardless of which rank it is.

The library itself runs one GPU per process and uses none of this on its
hot path (the workloads have N = 1 and run as independent replicas); the
combine is exercised by a multi-process CPU test against the single-rank
statistics.
"""
from __future__ import annotations

import numpy as np


def chan_merge(counts, means, m2s):
    """Merge per-part (count, mean, M2) triples, arrays shaped [R, ...], in
    the order of the first axis.  Returns (count, mean, M2) shaped [...]
    in float64.  Parts with a zero count contribute nothing."""
    counts = np.asarray(counts, np.float64)
    means = np.asarray(means, np.float64)
    m2s = np.asarray(m2s, np.float64)
    n = np.zeros(counts.shape[1:], np.float64)
    mean = np.zeros(counts.shape[1:], np.float64)
    m2 = np.zeros(counts.shape[1:], np.float64)
    for r in range(counts.shape[0]):
        nb, mb, m2b = counts[r], means[r], m2s[r]
        tot = n + nb
        safe = np.where(tot > 0, tot, 1.0)
        delta = mb - mean
        mean = np.where(tot > 0, mean + delta * nb / safe, mean)
        m2 = np.where(nb > 0, m2 + m2b + delta * delta * n * nb / safe, m2)
        n = tot
    return n, mean, m2


def allgather_combine(count, mean, m2, group=None):
    """All-gather this rank's (count, mean, M2) arrays (same shape on every
    rank) over torch.distributed and merge them in rank order.  Returns the
    merged (count, mean, M2) as float64 numpy arrays, identical on every
    rank."""
    import torch
    import torch.distributed as dist

    local = torch.from_numpy(np.stack([np.asarray(count, np.float64), np.asarray(mean, np.float64),
                                       np.asarray(m2, np.float64)]))
    world = dist.get_world_size(group)
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local, group=group)
    stacked = torch.stack(parts).numpy()          # [R, 3, ...]
    return chan_merge(stacked[:, 0], stacked[:, 1], stacked[:, 2])


def finalize(count, mean, m2, eps):
    """(mean, biased variance, rstd) from merged statistics."""
    var = np.maximum(np.asarray(m2, np.float64) / np.asarray(count, np.float64), 0.0)
    return np.asarray(mean, np.float64), var, 1.0 / np.sqrt(var + eps)
