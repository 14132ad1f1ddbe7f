"""CPU oracle for the rewiring of the groups' fan-in sets.

TEST INFRASTRUCTURE ONLY: the tests may import this module; the product
library never does.  Plain numpy in float64.

HASTE, "Method / overall framework" and "Loss and training strategy":
training alternates a continuous phase (weights fitted, index sets frozen) with
a discrete phase that periodically re-selects each group's fan-in set I_k by
the dynamic-sparse-training protocol of RigL, keeping |I_k| = F.  The pages do
not give the selection rule (their algorithm listing is not part of them), so
this is a labelled reading of RigL for group-shared fan-in:
  * prune score of an active fan-in index f of group k: the group's summed
    weight magnitude  m_k(f) = sum over the group's labels l of |W[l][f]|;
  * grow score of a feature j not in I_k: the group's summed magnitude of the
    dense gradient a weight at (l, j) would get,
        g_k(j) = sum over l in the group of |sum_b dZ[b][l] h[b][j]|;
  * per group, drop the n_drop active indices with the smallest prune score
    (ties: the smaller feature index first), then grow the n_drop features
    outside the old I_k with the largest grow score (ties: the smaller
    feature index first);
  * kept indices keep their weights, grown ones start at zero (RigL), and the
    new I_k is stored sorted ascending with the weights' columns following it.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def prune_scores(W, G: int) -> np.ndarray:
    """m[k][f] = sum over the G labels of group k of |W[l][f]| (W [L][F] in
    slot order)."""
    W = np.abs(_f64(W))
    L, F = W.shape
    return W.reshape(L // G, G, F).sum(axis=1)


def grow_scores(h, dZ, G: int) -> np.ndarray:
    """g[k][j] = sum over the labels l of group k of |sum_b dZ[b][l] h[b][j]|
    (h [B][H], dZ [B][L] in slot order)."""
    dense = _f64(dZ).T @ _f64(h)  # [L][H]: the gradient of every would-be weight
    L, H = dense.shape
    return np.abs(dense).reshape(L // G, G, H).sum(axis=1)


def rewire(idx_sorted, W, h, dZ, G: int, n_drop: int):
    """One discrete phase.  idx_sorted [K][F] (each row ascending), W [L][F]
    (columns follow idx_sorted), h [B][H], dZ [B][L].  Returns (new idx
    [K][F] ascending, new W [L][F] float64, dropped [K][n_drop], grown
    [K][n_drop]) with dropped and grown listed in selection order."""
    idx = np.asarray(idx_sorted, dtype=np.int64)
    K, F = idx.shape
    Wf = _f64(W)
    H = _f64(h).shape[1]
    m = prune_scores(W, G)
    gs = grow_scores(h, dZ, G)
    new_idx = np.zeros_like(idx)
    new_W = np.zeros_like(Wf)
    dropped = np.zeros((K, n_drop), dtype=np.int64)
    grown = np.zeros((K, n_drop), dtype=np.int64)
    for k in range(K):
        order = sorted(range(F), key=lambda f: (m[k][f], idx[k][f]))
        drop_pos = order[:n_drop]
        keep_pos = sorted(set(range(F)) - set(drop_pos))
        members = set(idx[k].tolist())
        cand = [j for j in range(H) if j not in members]
        cand.sort(key=lambda j: (-gs[k][j], j))
        grow = cand[:n_drop]
        dropped[k] = [idx[k][p] for p in drop_pos]
        grown[k] = grow
        # new set, ascending; kept columns carry their weights, grown ones 0
        entries = [(int(idx[k][p]), p) for p in keep_pos] + [(j, -1) for j in grow]
        entries.sort()
        rows = slice(k * G, (k + 1) * G)
        for q, (j, p) in enumerate(entries):
            new_idx[k][q] = j
            if p >= 0:
                new_W[rows, q] = Wf[rows, p]
    return new_idx, new_W, dropped, grown
