"""Pins for the semantic-grouping oracle (oracle/grouping.py), CPU only.

HASTE, "Key designs / group-shared fixed fan-in sparsity": label embeddings
from the positives' encoder outputs, mini-batch spherical k-means into coarse
clusters, greedy seed + top-(G - 1) groups inside each cluster.  The pins: two
hand-worked examples, the k-means update against its closed form and against
a spherical Lloyd step, the maximising property of a normalised sum, recovery
of a planted partition (the optimum by brute force on a tiny case), and the
output's invariants."""
import itertools
import json
from pathlib import Path

import numpy as np
import pytest

from oracle import grouping as gr

GOLD = Path(__file__).resolve().parent / "golden"


def test_embeddings_hand_example():
    d = json.loads((GOLD / "grouping_embeddings.json").read_text())
    E, has = gr.label_embeddings(np.array(d["h"]), np.array(d["rowptr"]), np.array(d["labels"]), d["L"])
    assert has.tolist() == d["has"]
    np.testing.assert_array_equal(E, np.array(d["E"]))


def test_greedy_hand_example():
    d = json.loads((GOLD / "grouping_greedy.json").read_text())
    groups = gr.greedy_groups(np.array(d["E"]), np.array(d["has"]), np.array(d["cluster"]),
                              np.array(d["centroids"]), d["G"])
    assert groups.tolist() == d["groups"]


def test_round_bf16_values():
    u = 2.0 ** -7
    for x, want in [(1.0, 1.0), (1 + u / 2, 1.0), (1 + 1.5 * u, 1 + 2 * u), (-(1 + 1.5 * u), -(1 + 2 * u)),
                    (0.6, 0.6015625), (0.8, 0.80078125)]:
        assert gr.round_bf16(np.array([x]))[0] == want, x


def _unit(rng, n, D):
    x = rng.standard_normal((n, D))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def test_assignment_takes_the_best_centroid_and_the_smaller_index_on_ties():
    rng = np.random.default_rng(1)
    E = gr.round_bf16(_unit(rng, 50, 8))
    mu = _unit(rng, 6, 8)
    mu[4] = mu[1]  # a duplicate centroid: every tie goes to 1
    a = gr.assign(E, mu)
    S = E @ gr.round_bf16(mu).T
    for i in range(len(E)):
        assert S[i, a[i]] == S[i].max()
        assert a[i] != 4


def test_first_full_batch_is_a_spherical_lloyd_step():
    """From zero counts, one batch holding every label moves each centroid to
    the normalised mean of the embeddings assigned to it."""
    rng = np.random.default_rng(2)
    E = gr.round_bf16(_unit(rng, 40, 5))
    mu0 = _unit(rng, 4, 5)
    mu, n, a = gr.kmeans_batch(E, mu0, np.zeros(4, np.int64), np.arange(40))
    for c in range(4):
        mem = E[a == c]
        assert n[c] == len(mem)
        if len(mem):
            s = mem.sum(axis=0)
            np.testing.assert_allclose(mu[c], s / np.linalg.norm(s), rtol=1e-12, atol=1e-12)
        else:
            np.testing.assert_array_equal(mu[c], mu0[c])


def test_batch_update_equals_its_closed_form():
    """With running counts n_c, the sequential per-member update of a batch
    equals Normalize((n_c mu_c + sum of the batch's members of c) / (n_c + m_c))."""
    rng = np.random.default_rng(3)
    E = gr.round_bf16(_unit(rng, 60, 6))
    mu0 = _unit(rng, 5, 6)
    n0 = rng.integers(0, 20, 5)
    batch = rng.permutation(60)[:25]
    mu, n, a = gr.kmeans_batch(E, mu0, n0, batch)
    for c in range(5):
        m = E[batch][a == c]
        assert n[c] == n0[c] + len(m)
        if len(m):
            v = (n0[c] * mu0[c] + m.sum(axis=0)) / (n0[c] + len(m))
            np.testing.assert_allclose(mu[c], v / np.linalg.norm(v), rtol=1e-12, atol=1e-12)


def test_normalised_sum_maximises_the_cluster_similarity():
    """The centroid update's fixed point: among unit vectors, the normalised
    sum of a cluster's embeddings maximises their summed similarity."""
    rng = np.random.default_rng(4)
    X = _unit(rng, 30, 7)
    s = X.sum(axis=0)
    best = float(np.sum(X @ (s / np.linalg.norm(s))))
    for v in _unit(rng, 200, 7):
        assert float(np.sum(X @ v)) <= best + 1e-12


def _planted(rng, n_clusters, groups_per_cluster, G, D, spread=0.02, sep=0.35):
    """Unit embeddings: cluster directions far apart, group directions around
    them, members tightly around their group's direction."""
    cdirs = _unit(rng, n_clusters, D)
    E, truth_group, truth_cluster = [], [], []
    g = 0
    for c in range(n_clusters):
        for _ in range(groups_per_cluster):
            gd = cdirs[c] + sep * _unit(rng, 1, D)[0]
            gd /= np.linalg.norm(gd)
            for _ in range(G):
                x = gd + spread * rng.standard_normal(D)
                E.append(x / np.linalg.norm(x))
                truth_group.append(g)
                truth_cluster.append(c)
            g += 1
    perm = rng.permutation(len(E))  # label ids unrelated to the structure
    E = gr.round_bf16(np.array(E)[perm])
    return E, np.array(truth_group)[perm], np.array(truth_cluster)[perm], cdirs


def _same_partition(a, b):
    pairs_a = {(x, y) for x, y in zip(a, b)}
    return len(pairs_a) == len(set(a)) == len(set(b))


def test_greedy_recovers_a_planted_partition():
    rng = np.random.default_rng(5)
    G = 4
    E, tg, tc, cdirs = _planted(rng, 4, 3, G, 24)
    has = np.ones(len(E), bool)
    mu = np.array([gr.round_bf16(E[tc == c]).sum(axis=0) for c in range(4)])
    mu /= np.linalg.norm(mu, axis=1, keepdims=True)
    groups = gr.greedy_groups(E, has, tc, mu, G)
    assert _same_partition(groups, tg)


def test_pipeline_recovers_a_planted_partition():
    """Embeddings from positives (each planted label positive in its own
    samples, whose h is the label's direction plus noise), k-means from one
    seed label per cluster over two full batches, then the greedy stage."""
    rng = np.random.default_rng(6)
    G, D = 4, 24
    E0, tg, tc, _ = _planted(rng, 3, 2, G, D)
    L = len(E0)
    # two samples per label, h = direction + small noise; row i holds label i // 2
    h = np.repeat(E0, 2, axis=0) + 0.01 * rng.standard_normal((2 * L, D))
    rowptr = np.arange(2 * L + 1)
    labels = np.repeat(np.arange(L), 2)
    init = [int(np.flatnonzero(tc == c)[0]) for c in range(3)]
    out = gr.semantic_grouping(h, rowptr, labels, L, G, init, [np.arange(L), np.arange(L)])
    assert _same_partition(out["cluster"], tc)
    assert _same_partition(out["groups"], tg)


def test_greedy_matches_the_brute_force_optimum_on_a_tiny_planted_case():
    """Six labels, G = 3, one cluster: the greedy partition is the one of the
    ten partitions into two groups that maximises the grouping objective."""
    rng = np.random.default_rng(7)
    E, tg, tc, _ = _planted(rng, 1, 2, 3, 6, spread=0.05, sep=1.0)
    has = np.ones(6, bool)
    mu = E.sum(axis=0, keepdims=True)
    mu /= np.linalg.norm(mu)
    groups = gr.greedy_groups(E, has, np.zeros(6, np.int64), mu, 3)
    best, best_obj = None, -np.inf
    for first in itertools.combinations(range(1, 6), 2):
        part = np.ones(6, np.int64)
        part[[0, *first]] = 0
        obj = gr.objective(E, has, part, 2)
        if obj > best_obj:
            best, best_obj = part, obj
    assert _same_partition(groups, best)
    assert _same_partition(groups, tg)


def test_objective_closed_forms():
    E = np.array([[1.0, 0.0], [1.0, 0.0], [1.0, 0.0], [0.0, 1.0]])
    has = np.ones(4, bool)
    # two identical unit vectors: 2; two orthogonal ones: 2 / sqrt(2)
    assert gr.objective(E, has, np.array([0, 0, 1, 1]), 2) == pytest.approx(2 + np.sqrt(2), rel=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_grouping_invariants(seed):
    """Every group has exactly G labels; every label is in one group; labels
    without a positive are grouped after every label with one."""
    rng = np.random.default_rng(seed)
    N, D, L, G = 40, 12, 96, 8
    h = rng.standard_normal((N, D))
    rowptr = np.concatenate([[0], np.cumsum(rng.integers(0, 4, N))])
    labels = rng.integers(0, 60, rowptr[-1])  # labels 60.. never positive
    E, has = gr.label_embeddings(h, rowptr, labels, L)
    act = np.flatnonzero(has)
    init = rng.choice(act, 3, replace=False)
    batches = [rng.permutation(act)[:16] for _ in range(4)]
    out = gr.semantic_grouping(h, rowptr, labels, L, G, init, batches)
    g = out["groups"]
    assert sorted(np.bincount(g, minlength=L // G).tolist()) == [G] * (L // G)
    # labels without embedding take the last positions of the pool, in
    # ascending id: their group ids never decrease, and only the first group
    # holding one of them may also hold labels with an embedding
    no = np.flatnonzero(~has)
    assert np.all(np.diff(g[no]) >= 0)
    for k in np.unique(g[no])[1:]:
        assert not has[g == k].any()
