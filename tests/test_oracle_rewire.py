"""Pins for the rewiring oracle (oracle/rewire.py), CPU only.

HASTE, "Method / overall framework" and "Loss and training strategy": each
group's fan-in set is re-selected periodically with |I_k| = F.  The pins: a
hand-worked example (including a grow tie), the grow score against the
layer's own weight gradient (an active index's grow score is the group-summed
|dW| of the oracle's O5), brute-force selection on random tiny cases, and the
output's invariants."""
import json
from pathlib import Path

import numpy as np
import pytest

import oracle
from oracle import rewire as rw
from workloads import Workload, generate

GOLD = Path(__file__).resolve().parent / "golden"


def test_hand_example():
    d = json.loads((GOLD / "rewire_hand.json").read_text())
    new_idx, new_W, dropped, grown = rw.rewire(np.array(d["idx"]), np.array(d["W"]), np.array(d["h"]),
                                               np.array(d["dZ"]), d["G"], d["n_drop"])
    assert new_idx.tolist() == d["new_idx"]
    np.testing.assert_array_equal(new_W, np.array(d["new_W"]))
    assert dropped.tolist() == d["dropped"] and grown.tolist() == d["grown"]


def test_grow_score_of_an_active_index_is_the_group_summed_weight_gradient(oracle_mod):
    """For f in I_k the would-be weight (l, I_k[f]) is the real weight W[l][f],
    so the grow score there is sum over the group of |dW[l][f]| with dW the
    layer's weight gradient (oracle O5)."""
    w = Workload("rw", B=24, H=40, L=12 * 8, G=8, F=6, pos=2, pos_dist="uniform", zipf_s=1.1,
                 idx_mode="uniform")
    p = generate(w)
    ref = oracle_mod.step(p, want_Z=True)
    dZ = ref["dZ"]
    gs = rw.grow_scores(p.h, dZ, w.G)
    dW = oracle_mod.weight_grad(p.h, dZ, ref["idx_sorted"], w.G, w.F)
    want = np.abs(dW).reshape(w.K, w.G, w.F).sum(axis=1)
    ids = ref["idx_sorted"].astype(np.int64)
    np.testing.assert_allclose(gs[np.arange(w.K)[:, None], ids], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_selection_against_brute_force(seed):
    """Dropped = the n smallest prune scores (by value, then feature); grown =
    the n largest grow scores outside the old set (by value, then feature);
    kept weights unchanged, grown weights zero, every row sorted and
    distinct."""
    rng = np.random.default_rng(seed)
    K, G, F, H, B, n = 5, 3, 6, 15, 7, int(rng.integers(0, 7))
    idx = np.sort(np.stack([rng.permutation(H)[:F] for _ in range(K)]), axis=1)
    # a few exact ties in both scores
    W = rng.integers(-3, 4, (K * G, F)).astype(np.float64) / 4
    h = rng.integers(-2, 3, (B, H)).astype(np.float64)
    dZ = rng.integers(-2, 3, (B, K * G)).astype(np.float64) / 2
    new_idx, new_W, dropped, grown = rw.rewire(idx, W, h, dZ, G, n)
    m = np.abs(W).reshape(K, G, F).sum(axis=1)
    dense = dZ.T @ h
    gsc = np.abs(dense).reshape(K, G, H).sum(axis=1)
    for k in range(K):
        pairs = sorted((m[k][f], idx[k][f]) for f in range(F))
        assert sorted(dropped[k].tolist()) == sorted(j for _, j in pairs[:n])
        outside = sorted(((-gsc[k][j], j) for j in range(H) if j not in set(idx[k])))
        assert sorted(grown[k].tolist()) == sorted(j for _, j in outside[:n])
        row = new_idx[k]
        assert np.all(np.diff(row) > 0) and len(row) == F
        assert set(row) == (set(idx[k]) - set(dropped[k])) | set(grown[k])
        for q, j in enumerate(row):
            cols = new_W[k * G:(k + 1) * G, q]
            if j in set(grown[k]):
                assert np.all(cols == 0)
            else:
                p = int(np.flatnonzero(idx[k] == j)[0])
                np.testing.assert_array_equal(cols, W[k * G:(k + 1) * G, p])


def test_no_drop_is_the_identity():
    rng = np.random.default_rng(9)
    idx = np.sort(np.stack([rng.permutation(20)[:5] for _ in range(3)]), axis=1)
    W = rng.standard_normal((6, 5))
    new_idx, new_W, _, _ = rw.rewire(idx, W, rng.standard_normal((4, 20)), rng.standard_normal((4, 6)), 2, 0)
    np.testing.assert_array_equal(new_idx, idx)
    np.testing.assert_array_equal(new_W, W)
