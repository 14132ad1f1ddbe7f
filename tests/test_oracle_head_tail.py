"""Pins for the head-tail oracle (oracle/head_tail.py), CPU only.

HASTE, "Method / overall framework" and "Key designs / head-tail split": the
encoder output feeds a dense head and the group-shared sparse tail through two
projections, and the loss is the sum of both branches' BCE terms.  The oracle
is pinned to central finite differences of that loss for every parameter, and
with identity projections its head reduces to the tail oracle's own forward
(one group of all head labels sharing the full index set) and its tail to the
plain step."""
import numpy as np
import pytest

from oracle import forward as or_forward
from oracle import head_tail as ht
from workloads import Workload, generate


def _problem(rng, B=3, E=5, Dh=4, H=6, Lh=3, L=8, G=2, F=3, npos=2):
    K = L // G
    groups = rng.permutation(L).astype(np.int32) // G
    idx = np.stack([rng.choice(H, F, replace=False) for _ in range(K)]).astype(np.int32)
    lists = [rng.choice(L, npos, replace=False) for _ in range(B)]
    rowptr = np.zeros(B + 1, np.int32)
    rowptr[1:] = np.cumsum([len(x) for x in lists])
    labels = np.concatenate(lists).astype(np.int32)
    return dict(h=rng.standard_normal((B, E)), P_head=rng.standard_normal((Dh, E)) * 0.5,
                P_tail=rng.standard_normal((H, E)) * 0.5, W_head=rng.standard_normal((Lh, Dh)) * 0.5,
                Y_head=(rng.random((B, Lh)) < 0.4).astype(np.float64),
                W_tail=rng.standard_normal((L, F)) * 0.5, groups=groups, idx=idx, G=G, F=F,
                pos_rowptr=rowptr, pos_label=labels)


def _loss(p):
    return ht.step(**p)["loss"]


@pytest.mark.parametrize("seed", [0, 1])
def test_head_tail_gradients_finite_difference(seed):
    rng = np.random.default_rng(seed)
    p = _problem(rng)
    out = ht.step(**p)
    grads = {"h": out["dh"], "P_head": out["dP_head"], "P_tail": out["dP_tail"],
             "W_head": out["dW_head"], "W_tail": out["dW_tail"]}
    eps = 1e-6
    for name, g in grads.items():
        a = p[name]
        for _ in range(6):
            i = tuple(int(rng.integers(0, n)) for n in a.shape)
            old = a[i]
            a[i] = old + eps
            up = _loss(p)
            a[i] = old - eps
            dn = _loss(p)
            a[i] = old
            fd = (up - dn) / (2 * eps)
            assert abs(fd - g[i]) <= 1e-6 * (1.0 + abs(fd)), (name, i, fd, g[i])


def test_head_tail_identity_projections_reduce_to_the_layer():
    """E = Dh = H and P_head = P_tail = I: the head's logits are the tail
    oracle's forward for one group holding every head label with I = [0, H),
    and the tail's gradients are the plain step's on h."""
    rng = np.random.default_rng(5)
    w = Workload("ht_id", B=4, H=16, L=32, G=4, F=6, pos=2, pos_dist="uniform", zipf_s=1.1,
                 idx_mode="uniform")
    prob = generate(w)
    h = (prob.h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    W_tail = (prob.W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    I = np.eye(w.H)
    Lh = 5
    W_head = rng.standard_normal((Lh, w.H))
    Y_head = (rng.random((w.B, Lh)) < 0.3).astype(np.float64)
    out = ht.step(h, I, I, W_head, Y_head, W_tail, prob.groups, prob.idx, w.G, w.F,
                  prob.pos_rowptr, prob.pos_label)
    full = np.arange(w.H, dtype=np.uint16)[None, :]
    A_ref = or_forward(h, W_head, full, Lh)
    np.testing.assert_allclose(out["A"], A_ref, rtol=1e-12, atol=1e-12)
    from oracle import step as tail_step
    ref = tail_step(prob)  # the tail sees h itself through the identity projection
    np.testing.assert_allclose(out["dW_tail"], ref["dW"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dh_tail"], ref["dh"], rtol=1e-12, atol=1e-12)
    assert out["tail_loss"] == pytest.approx(ref["loss"], rel=1e-12)
