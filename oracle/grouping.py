"""CPU oracle for the semantic grouping of labels.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
leg may import this module; the product library never does.  Plain numpy in
float64; pure-Python loops only where the steps are sequential.

HASTE, "Key designs / group-shared fixed fan-in sparsity": labels are grouped
so that a group's members are close in embedding space (maximise the summed
similarity of each label to its group's mean), with label embeddings taken
from the encoder outputs of each label's positive samples, normalised.  Exact
partitioning is out of reach for millions of labels, so the method runs two
stages: mini-batch spherical k-means into about L / (beta G) coarse clusters,
then, inside each cluster, greedy groups of a seed and its G - 1 nearest
remaining neighbours.

Readings where the page leaves a step open (each also recorded with the
design notes):
  * e_l = Normalize(sum of h_i over the samples i with l positive); a sample
    counts once per label however often l repeats in its row.  A label with
    no positive sample has no embedding (e_l undefined): it takes part in
    neither k-means nor the greedy stage and is grouped last.
  * Embeddings are stored as bf16 (round to nearest even), the layer's
    precision; centroids are kept in float64 here and rounded to bf16 when
    scored, so that every similarity is a dot product of two bf16 vectors.
  * Similarity = dot product of those (unit-norm) vectors.
  * Mini-batch k-means (web-scale k-means with per-centre learning rates
    1/n_c), projected back to the sphere after each batch: the batch is
    assigned with the centroids of the batch start (argmax similarity, ties
    to the smaller centroid index), then each member in batch order moves its
    centroid by (e - mu) / n_c with n_c the centroid's running count, and
    every centroid the batch moved is normalised.  Initial centroids are the
    embeddings of given distinct labels; the batches are given too (random
    draws are inputs).
  * Greedy stage: clusters in ascending index; inside a cluster, while at
    least G members remain: the seed is the remaining member most similar to
    the cluster's centroid, its group is the seed plus the G - 1 remaining
    members most similar to the seed (ties to the smaller label id); groups
    are numbered in the order they are formed.
  * Groups have exactly G labels (the layer's definition): the members a
    cluster leaves over (fewer than G), in cluster order and ascending label
    id, followed by the labels without embedding in ascending id, are cut
    into consecutive groups of G numbered after the greedy ones.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x) -> np.ndarray:
    """float64 -> nearest fp32 -> nearest bf16 (ties to even), as float64."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    keep_odd = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_odd) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def label_embeddings(h, rowptr, labels, L: int):
    """-> (E [L, D] float64 holding bf16 values, has [L] bool).

    E[l] = bf16(Normalize(sum over the distinct samples i with l in row i of
    h_i)); rows of labels without a positive (or with a zero sum) are zero and
    has[l] is False."""
    h = _f64(h)
    N, D = h.shape
    S = np.zeros((L, D))
    for i in range(N):
        seen = set()
        for l in labels[rowptr[i]:rowptr[i + 1]]:
            l = int(l)
            if 0 <= l < L and l not in seen:
                seen.add(l)
                S[l] += h[i]
    norms = np.sqrt(np.sum(S * S, axis=1))
    has = norms > 0
    E = np.zeros((L, D))
    E[has] = round_bf16(S[has] / norms[has, None])
    return E, has


def assign(E_rows, centroids) -> np.ndarray:
    """argmax_c <e, bf16(mu_c)> for each row (ties to the smaller c)."""
    scores = np.asarray(E_rows, dtype=np.float64) @ round_bf16(centroids).T
    return np.argmax(scores, axis=1).astype(np.int64)


def kmeans_batch(E, centroids, counts, batch):
    """One mini-batch of spherical k-means.  E [L, D], centroids [C, D]
    (float64, unit rows), counts [C] int64, batch: label ids in batch order.
    Returns (new centroids, new counts, the batch's assignment)."""
    a = assign(E[batch], np.asarray(centroids, dtype=np.float64))
    mu, n = kmeans_update(E, centroids, counts, batch, a)
    return mu, n, a


def kmeans_update(E, centroids, counts, batch, a):
    """The update half of a batch, given its assignment a: each member in
    batch order moves its centroid by (e - mu) / n_c, then every moved
    centroid is normalised.  Returns (centroids, counts)."""
    mu = np.array(centroids, dtype=np.float64, copy=True)
    n = np.array(counts, dtype=np.int64, copy=True)
    moved = set()
    for l, c in zip(batch, a):
        n[c] += 1
        mu[c] += (E[l] - mu[c]) / n[c]
        moved.add(int(c))
    for c in moved:
        nrm = np.sqrt(np.dot(mu[c], mu[c]))
        if nrm > 0:
            mu[c] /= nrm
    return mu, n


def kmeans(E, init_labels, batches):
    """Centroids start at E[init_labels] (normalised), counts at 0; then one
    kmeans_batch per batch.  Returns (centroids, counts)."""
    mu = np.array(E[np.asarray(init_labels)], dtype=np.float64)
    mu /= np.sqrt(np.sum(mu * mu, axis=1, keepdims=True))
    n = np.zeros(len(mu), dtype=np.int64)
    for b in batches:
        mu, n, _ = kmeans_batch(E, mu, n, np.asarray(b))
    return mu, n


def greedy_groups(E, has, cluster, centroids, G: int):
    """The greedy stage and the leftover pool.  cluster[l] is the cluster of
    every label with an embedding.  Returns groups[L] (int64 group ids)."""
    L = len(has)
    groups = np.full(L, -1, dtype=np.int64)
    mu_b = round_bf16(centroids)
    C = len(centroids)
    members = [[] for _ in range(C)]
    for l in range(L):
        if has[l]:
            members[int(cluster[l])].append(l)
    gid = 0
    pool = []
    for c in range(C):
        R = list(members[c])  # ascending label id
        to_mu = {l: float(np.dot(E[l], mu_b[c])) for l in R}
        while len(R) >= G:
            seed = max(R, key=lambda l: (to_mu[l], -l))
            rest = [l for l in R if l != seed]
            rest.sort(key=lambda l: (-float(np.dot(E[l], E[seed])), l))
            grp = [seed] + rest[:G - 1]
            for l in grp:
                groups[l] = gid
            gid += 1
            chosen = set(grp)
            R = [l for l in R if l not in chosen]
        pool.extend(R)
    pool.extend(l for l in range(L) if not has[l])
    for p, l in enumerate(pool):
        groups[l] = gid + p // G
    return groups


def semantic_grouping(h, rowptr, labels, L: int, G: int, init_labels, batches):
    """The whole grouping: embeddings, mini-batch k-means, final assignment of
    every label with an embedding, greedy groups.  Returns a dict with E, has,
    centroids, counts, cluster (-1 without embedding) and groups."""
    E, has = label_embeddings(h, rowptr, labels, L)
    mu, n = kmeans(E, init_labels, batches)
    cluster = np.full(L, -1, dtype=np.int64)
    idx = np.flatnonzero(has)
    if len(idx):
        cluster[idx] = assign(E[idx], mu)
    groups = greedy_groups(E, has, cluster, mu, G)
    return dict(E=E, has=has, centroids=mu, counts=n, cluster=cluster, groups=groups)


def objective(E, has, groups, K: int) -> float:
    """sum over groups k of sum over members l (with an embedding) of
    <e_l, Normalize(mean of the members' embeddings)>: the quantity the
    grouping maximises."""
    total = 0.0
    for k in range(K):
        mem = [l for l in np.flatnonzero(groups == k) if has[l]]
        if not mem:
            continue
        m = np.sum(E[mem], axis=0)
        nrm = np.sqrt(np.dot(m, m))
        if nrm > 0:
            total += float(np.sum(E[mem] @ (m / nrm)))
    return total
