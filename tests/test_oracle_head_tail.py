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


def test_round_bf16_values():
    """Rounding to bf16 (8 significant bits): exact values stay, halfway cases
    go to the even neighbour, anything past halfway goes up; signs are kept."""
    u = 2.0 ** -7  # one bf16 ulp at 1
    cases = [(1.0, 1.0), (1.0 + u / 2, 1.0), (1.0 + 1.5 * u, 1.0 + 2 * u), (1.0 + u / 2 + 2 ** -20, 1.0 + u),
             (-(1.0 + 1.5 * u), -(1.0 + 2 * u)), (3.0, 3.0), (0.0, 0.0), (2.0 ** -130, 2.0 ** -130),
             (255.5, 256.0), (254.5, 254.0), (1e-3, 0.00099945068359375)]
    for x, want in cases:
        assert ht.round_bf16(np.array([x]))[0] == want, x


def test_round_bf16_matches_torch_on_fp32():
    """On fp32 inputs (no first rounding) the result is torch's own
    float32 -> bfloat16 conversion, which rounds to nearest even."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ht.round_bf16(x.astype(np.float64)), want)


def test_hidden_bf16_rounds_only_the_activations():
    """hidden_bf16 changes nothing when both projections already give bf16
    values (identity projections of a bf16 h); otherwise the tail's gradients
    are the plain layer's on the rounded activations, and dP, dh are taken
    from the same branch gradients as without rounding."""
    rng = np.random.default_rng(7)
    p = _problem(rng, B=4, E=6, Dh=6, H=6)
    hb = ht.round_bf16(p["h"])
    I = np.eye(6)
    base = dict(p, h=hb, P_head=I, P_tail=I)
    a = ht.step(**base)
    b = ht.step(**base, hidden_bf16=True)
    for k in ("loss", "dW_head", "dW_tail", "dP_head", "dP_tail", "dh"):
        np.testing.assert_array_equal(a[k], b[k])
    r = ht.step(**p, hidden_bf16=True)
    assert np.array_equal(r["h_tail"], ht.round_bf16(r["h_tail"]))
    assert np.array_equal(r["h_head"], ht.round_bf16(p["h"] @ p["P_head"].T))
    # the rounded activations change the loss of this draw
    assert r["loss"] != ht.step(**p)["loss"]
    # tail gradients: the unrounded oracle run on h_tail as the encoder output
    # with an identity tail projection
    q = dict(p, h=r["h_tail"], P_tail=np.eye(p["P_tail"].shape[0]), P_head=np.zeros_like(p["P_head"]))
    t = ht.step(**q)
    np.testing.assert_allclose(r["dW_tail"], t["dW_tail"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dP_tail"], r["dh_tail"].T @ p["h"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dh"], r["dh_head"] @ p["P_head"] + r["dh_tail"] @ p["P_tail"], rtol=1e-12,
                               atol=1e-12)
