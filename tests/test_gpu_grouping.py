"""Semantic grouping on the GPU against the CPU oracle (oracle/grouping.py),
through the C ABI.

HASTE, "Key designs / group-shared fixed fan-in sparsity": label embeddings
from the positives' encoder outputs, mini-batch spherical k-means into coarse
clusters, greedy seed + top-(G - 1) groups inside each cluster.

Where a floating-point comparison decides an integer (an argmax, a greedy
pick), the GPU sums in fp32 and the oracle in double over the same bf16
values, so exact ties can break apart by rounding: those results are checked
for validity (the GPU's choice scores within 1e-5 of the best, which bounds
the fp32 rounding of a dot product of D <= 128 bf16 unit-vector entries),
and compared exactly on data whose margins exceed that bound.
"""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import draw_bf16_matrix, to_bf16_bits

from gpu_common import dev_i32

pytestmark = pytest.mark.gpu
EPS = 1e-5


def _bits_to_f64(t):
    u = t.detach().cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _dev_bits(x):
    return torch.from_numpy(np.ascontiguousarray(to_bf16_bits(x)).view(np.int16)).cuda()


def _unit(rng, n, D):
    x = rng.standard_normal((n, D))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _positives(rng, N, L, per_row, live):
    """Rows of per_row labels drawn from [0, live) with repeats (a label may
    occur twice in a row); labels live..L-1 never occur."""
    rowptr = np.zeros(N + 1, np.int32)
    rows = []
    for i in range(N):
        k = int(rng.integers(0, per_row + 1))
        r = rng.integers(0, live, k).astype(np.int32)
        if k >= 2 and rng.random() < 0.3:
            r[-1] = r[0]
        rows.append(r)
        rowptr[i + 1] = rowptr[i] + k
    return rowptr, np.concatenate(rows) if rows else np.zeros(0, np.int32)


def test_embeddings_against_oracle(oracle_mod):
    from oracle import grouping as gr
    sg.build()
    rng = np.random.default_rng(0)
    N, D, L, G = 300, 64, 512, 16
    hbits = draw_bf16_matrix(11, N, D, 1.0)
    rowptr, labels = _positives(rng, N, L, 6, 400)
    E_ref, has_ref = gr.label_embeddings(hbits, rowptr, labels, L)
    g = sg.sg_grouping_create(L, D, G, 8)
    try:
        n = sg.sg_grouping_embed(g, torch.from_numpy(hbits.view(np.int16)).cuda(), dev_i32(rowptr),
                                 dev_i32(labels if len(labels) else np.zeros(1)), len(labels))
        E = torch.empty((L, D), dtype=torch.int16, device="cuda")
        has = torch.empty(L, dtype=torch.uint8, device="cuda")
        sg.sg_grouping_export(g, E=E, has=has)
        assert sg.sg_grouping_status(g) == 0
    finally:
        g.close()
    assert n == int(has_ref.sum())
    np.testing.assert_array_equal(has.cpu().numpy().astype(bool), has_ref)
    got = _bits_to_f64(E)
    # both round the same normalised sum to bf16: at most one bf16 step apart
    # (where the two sums straddle a rounding boundary), and almost always equal
    assert np.all(np.abs(got - E_ref) <= 2.0 ** -8 * np.abs(E_ref) + 1e-30)
    assert np.mean(got == E_ref) > 0.999


def _set_state(g, E, has, mu, counts=None):
    sg.sg_grouping_set_embeddings(g, _dev_bits(E), torch.from_numpy(has.astype(np.uint8)).cuda())
    sg.sg_grouping_set_centroids(g, torch.from_numpy(mu.astype(np.float32)).cuda(),
                                 None if counts is None else torch.from_numpy(counts.astype(np.int64)).cuda())


def test_kmeans_batch_against_oracle(oracle_mod):
    """One batch: the assignment is the oracle's argmax (valid within EPS,
    equal where the margin exceeds it), and the updated centroids and counts
    match the oracle's update under the GPU's assignment."""
    from oracle import grouping as gr
    sg.build()
    rng = np.random.default_rng(1)
    L, D, C, G, M = 2048, 128, 200, 16, 1500
    E = gr.round_bf16(_unit(rng, L, D))
    has = np.ones(L, bool)
    mu0 = _unit(rng, C, D).astype(np.float32).astype(np.float64)
    n0 = rng.integers(0, 30, C)
    batch = rng.permutation(L)[:M].astype(np.int32)
    g = sg.sg_grouping_create(L, D, G, C)
    try:
        _set_state(g, E, has, mu0, n0)
        a = torch.empty(M, dtype=torch.int32, device="cuda")
        sg.sg_grouping_kmeans_batch(g, dev_i32(batch), a)
        cent = torch.empty((C, D), dtype=torch.float32, device="cuda")
        cnt = torch.empty(C, dtype=torch.int64, device="cuda")
        sg.sg_grouping_export(g, centroids=cent, counts=cnt)
        assert sg.sg_grouping_status(g) == 0
    finally:
        g.close()
    a = a.cpu().numpy().astype(np.int64)
    S = E[batch] @ gr.round_bf16(mu0).T
    best = S.max(axis=1)
    assert np.all(S[np.arange(M), a] >= best - EPS)
    a_ref = gr.assign(E[batch], mu0)
    top2 = np.sort(S, axis=1)[:, -2:]
    clear = top2[:, 1] - top2[:, 0] > EPS
    np.testing.assert_array_equal(a[clear], a_ref[clear])
    mu_ref, n_ref = gr.kmeans_update(E, mu0, n0, batch, a)
    np.testing.assert_array_equal(cnt.cpu().numpy(), n_ref)
    np.testing.assert_allclose(cent.cpu().numpy(), mu_ref, atol=2e-6, rtol=0)


def _planted(rng, n_clusters, groups_per_cluster, G, D, spread=0.02, sep=0.35):
    cdirs = _unit(rng, n_clusters, D)
    E, tg, tc = [], [], []
    gid = 0
    for c in range(n_clusters):
        for _ in range(groups_per_cluster):
            gd = cdirs[c] + sep * _unit(rng, 1, D)[0]
            gd /= np.linalg.norm(gd)
            for _ in range(G):
                x = gd + spread * rng.standard_normal(D)
                E.append(x / np.linalg.norm(x))
                tg.append(gid)
                tc.append(c)
            gid += 1
    perm = rng.permutation(len(E))
    return np.array(E)[perm], np.array(tg)[perm], np.array(tc)[perm]


def _same_partition(a, b):
    return len({(x, y) for x, y in zip(a, b)}) == len(set(a)) == len(set(b))


@pytest.mark.parametrize("leftover", [False, True])
def test_greedy_against_oracle(oracle_mod, leftover):
    """The final assignment and the greedy stage on planted clusters (margins
    well above EPS): groups and clusters equal the oracle's exactly.  With
    `leftover`, every cluster holds a group's worth plus extra labels, some
    labels have no embedding, and the pool rules decide the last groups."""
    from oracle import grouping as gr
    sg.build()
    rng = np.random.default_rng(2)
    G, D, nc, gpc = 8, 64, 6, 5
    E0, tg, tc = _planted(rng, nc, gpc, G, D)
    L = len(E0)
    has = np.ones(L, bool)
    if leftover:
        # drop G + 3 labels' embeddings: clusters lose members unevenly, the
        # pool gets leftovers and labels without embedding
        has[rng.permutation(L)[:G + 3]] = False
    E = np.where(has[:, None], gr.round_bf16(E0), 0.0)
    mu = np.array([E[(tc == c) & has].sum(axis=0) for c in range(nc)])
    mu = (mu / np.linalg.norm(mu, axis=1, keepdims=True)).astype(np.float32).astype(np.float64)
    g = sg.sg_grouping_create(L, D, G, nc)
    try:
        _set_state(g, E, has, mu)
        groups = torch.empty(L, dtype=torch.int32, device="cuda")
        clus = torch.empty(L, dtype=torch.int32, device="cuda")
        sg.sg_grouping_groups(g, groups, clus)
        assert sg.sg_grouping_status(g) == 0
    finally:
        g.close()
    cluster_ref = np.full(L, -1)
    cluster_ref[has] = gr.assign(E[has], mu)
    np.testing.assert_array_equal(clus.cpu().numpy(), cluster_ref)
    groups_ref = gr.greedy_groups(E, has, cluster_ref, mu, G)
    np.testing.assert_array_equal(groups.cpu().numpy(), groups_ref)
    if not leftover:
        assert _same_partition(groups.cpu().numpy(), tg)


def test_greedy_random_data_is_valid(oracle_mod):
    """Unstructured data (near-ties possible): every group has exactly G
    labels, and the grouping objective is within 1e-4 of the oracle's."""
    from oracle import grouping as gr
    sg.build()
    rng = np.random.default_rng(3)
    L, D, G, C = 1024, 32, 16, 10
    E = gr.round_bf16(_unit(rng, L, D))
    has = np.ones(L, bool)
    has[rng.permutation(L)[:40]] = False
    E[~has] = 0
    mu = _unit(rng, C, D).astype(np.float32).astype(np.float64)
    g = sg.sg_grouping_create(L, D, G, C)
    try:
        _set_state(g, E, has, mu)
        groups = torch.empty(L, dtype=torch.int32, device="cuda")
        sg.sg_grouping_groups(g, groups)
    finally:
        g.close()
    got = groups.cpu().numpy()
    assert sorted(np.bincount(got, minlength=L // G).tolist()) == [G] * (L // G)
    cluster_ref = np.full(L, -1)
    cluster_ref[has] = gr.assign(E[has], mu)
    ref = gr.greedy_groups(E, has, cluster_ref, mu, G)
    o_gpu, o_ref = gr.objective(E, has, got, L // G), gr.objective(E, has, ref, L // G)
    assert abs(o_gpu - o_ref) <= 1e-4 * abs(o_ref)


def test_pipeline_against_oracle(oracle_mod):
    """Embeddings from positives, k-means from one seed label per cluster
    over full batches, final assignment and greedy groups: the planted
    partition, equal to the oracle's groups."""
    from oracle import grouping as gr
    sg.build()
    rng = np.random.default_rng(4)
    G, D = 8, 64
    E0, tg, tc = _planted(rng, 4, 3, G, D)
    L = len(E0)
    h = np.repeat(E0, 2, axis=0) + 0.01 * rng.standard_normal((2 * L, D))
    hbits = to_bf16_bits(h)
    rowptr = np.arange(2 * L + 1, dtype=np.int32)
    labels = np.repeat(np.arange(L, dtype=np.int32), 2)
    init = np.array([int(np.flatnonzero(tc == c)[0]) for c in range(4)], np.int32)
    batches = [np.arange(L, dtype=np.int32), rng.permutation(L).astype(np.int32)]
    ref = gr.semantic_grouping(hbits, rowptr, labels, L, G, init, batches)
    g = sg.sg_grouping_create(L, D, G, 4)
    try:
        sg.sg_grouping_embed(g, torch.from_numpy(hbits.view(np.int16)).cuda(), dev_i32(rowptr), dev_i32(labels),
                             len(labels))
        sg.sg_grouping_kmeans_init(g, dev_i32(init))
        for b in batches:
            sg.sg_grouping_kmeans_batch(g, dev_i32(b))
        groups = torch.empty(L, dtype=torch.int32, device="cuda")
        sg.sg_grouping_groups(g, groups)
        cent = torch.empty((4, D), dtype=torch.float32, device="cuda")
        sg.sg_grouping_export(g, centroids=cent)
        assert sg.sg_grouping_status(g) == 0
    finally:
        g.close()
    np.testing.assert_allclose(cent.cpu().numpy(), ref["centroids"], atol=1e-4, rtol=0)
    np.testing.assert_array_equal(groups.cpu().numpy(), ref["groups"])
    assert _same_partition(groups.cpu().numpy(), tg)


def test_groups_feed_the_layout():
    """The groups a grouping writes build a layout (every group exactly G)."""
    sg.build()
    rng = np.random.default_rng(5)
    N, D, L, G, C = 500, 32, 4096, 32, 16
    hbits = draw_bf16_matrix(12, N, D, 1.0)
    rowptr, labels = _positives(rng, N, L, 8, 3000)
    g = sg.sg_grouping_create(L, D, G, C)
    try:
        n = sg.sg_grouping_embed(g, torch.from_numpy(hbits.view(np.int16)).cuda(), dev_i32(rowptr),
                                 dev_i32(labels), len(labels))
        E = torch.empty((L, D), dtype=torch.int16, device="cuda")
        has = torch.empty(L, dtype=torch.uint8, device="cuda")
        sg.sg_grouping_export(g, E=E, has=has)
        act = np.flatnonzero(has.cpu().numpy())
        assert len(act) == n
        sg.sg_grouping_kmeans_init(g, dev_i32(rng.choice(act, C, replace=False)))
        for _ in range(3):
            sg.sg_grouping_kmeans_batch(g, dev_i32(rng.choice(act, 512, replace=False)))
        groups = torch.empty(L, dtype=torch.int32, device="cuda")
        sg.sg_grouping_groups(g, groups)
        assert sg.sg_grouping_status(g) == 0
    finally:
        g.close()
    got = groups.cpu().numpy()
    assert sorted(np.bincount(got, minlength=L // G).tolist()) == [G] * (L // G)
    F, H = 16, 64
    idx = np.stack([rng.permutation(H)[:F] for _ in range(L // G)]).astype(np.int32)
    lay = sg.sg_layout_build(groups, L, G, dev_i32(idx.reshape(-1)), F, H, 8, 1)
    lay.close()


def test_init_label_without_embedding_sets_the_status():
    sg.build()
    L, D, G, C = 64, 16, 8, 2
    E = np.zeros((L, D))
    E[:, 0] = 1.0
    has = np.ones(L, np.uint8)
    has[5] = 0
    E[5] = 0
    g = sg.sg_grouping_create(L, D, G, C)
    try:
        sg.sg_grouping_set_embeddings(g, _dev_bits(E), torch.from_numpy(has).cuda())
        sg.sg_grouping_kmeans_init(g, dev_i32(np.array([1, 5], np.int32)))
        torch.cuda.synchronize()
        assert sg.sg_grouping_status(g) == sg.SG_ERR_DATA
        assert sg.sg_grouping_status(g) == 0  # read and cleared
    finally:
        g.close()
