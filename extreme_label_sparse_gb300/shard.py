"""Host-side sharding of the layer over GPUs by group range.

HASTE's feature gradient is a Split-K over groups (key design "gather-once +
dense MMA kernel"); across GPUs the same reduction is one more level: GPU p
owns the groups [k_p, k_{p+1}), their labels, W rows, fan-in sets and the
positives that fall in its labels, and h is replicated.  Z, dZ, dW and the BCE
terms are then local, and only dh (B x H) and the scalar loss are summed over
GPUs (one all-reduce each).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def group_range(K: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced split of K groups over `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    return K * rank // world, K * (rank + 1) // world


@dataclass
class Shard:
    k0: int
    k1: int
    labels: np.ndarray      # global label ids owned by the shard, ascending
    groups: np.ndarray      # local group id of each owned label
    idx: np.ndarray         # [k1-k0, F] fan-in sets
    W: np.ndarray           # [(k1-k0)*G, F] rows of the shard's slots
    pos_rowptr: np.ndarray  # positives restricted to the shard, local label ids
    pos_label: np.ndarray


def shard_problem(groups, idx, W, pos_rowptr, pos_label, G: int, world: int, rank: int) -> Shard:
    """The rank's part of a problem given in global ids (W in slot order)."""
    groups = np.asarray(groups)
    K = len(groups) // G
    k0, k1 = group_range(K, world, rank)
    own = (groups >= k0) & (groups < k1)
    labels = np.flatnonzero(own)
    local_of = np.full(len(groups), -1, dtype=np.int64)
    local_of[labels] = np.arange(len(labels))
    rows = []
    for b in range(len(pos_rowptr) - 1):
        r = np.asarray(pos_label[pos_rowptr[b]:pos_rowptr[b + 1]])
        rows.append(local_of[r[own[r]]])
    rp = np.zeros(len(pos_rowptr), dtype=np.int32)
    rp[1:] = np.cumsum([len(r) for r in rows])
    lb = np.concatenate(rows).astype(np.int32) if rows else np.zeros(0, np.int32)
    return Shard(k0, k1, labels, (groups[labels] - k0).astype(np.int32),
                 np.asarray(idx)[k0:k1], np.asarray(W)[k0 * G:k1 * G], rp, lb)
