"""Pins for the CPU oracle: checks it against things other than itself.

Each test ties one oracle function to a fact the HASTE page or plain mathematics
fixes: a hand-worked example, a library routine the definition reduces to
(numpy sort / matmul, Python's math), a special case (G=1 per-label fan-in,
dense F=H, one shared contiguous block), closed forms of BCE, or central finite
differences of the summed loss.  A dropped term, a wrong sign, a transposed
operand or a wrong index in the oracle fails at least one of these.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest

from workloads import CONFIGS, generate, to_bf16_bits, bf16_bits_to_f32

GOLDEN = Path(__file__).parent / "golden"


def _rand_problem(rng, B, H, L, G, F, npos=3):
    K = L // G
    groups = (rng.permutation(L) // G).astype(np.int32)
    idx = np.stack([rng.permutation(H)[:F] for _ in range(K)]).astype(np.int32)
    h = rng.standard_normal((B, H))
    W = rng.standard_normal((L, F)) / math.sqrt(F)
    rows = [rng.choice(L, size=min(npos, L), replace=False) for _ in range(B)]
    rowptr = np.zeros(B + 1, dtype=np.int32)
    rowptr[1:] = np.cumsum([len(r) for r in rows])
    labels = np.concatenate(rows).astype(np.int32) if B else np.zeros(0, np.int32)
    return groups, idx, h, W, rowptr, labels


def _densify(W, idx_sorted, G, H):
    """Wd[s, I_k(s)[f]] = W[s, f]  (the L x H matrix the sparse layer stands for)."""
    L, F = W.shape
    Wd = np.zeros((L, H))
    for s in range(L):
        Wd[s, idx_sorted[s // G]] = W[s]
    return Wd


def _loss(oracle_mod, h, W, ids, G, srp, ssl):
    Z = oracle_mod.forward(h, W, ids, G)
    return oracle_mod.bce(Z, srp, ssl)


# ------------------------------------------------------------ hand example
def test_hand_worked_example(oracle_mod):
    g = json.loads((GOLDEN / "hand_example.json").read_text())
    e = g["expect"]
    h = np.array(g["h"])
    W = np.array(g["W"])
    st, sol, los, ids = oracle_mod.layout_build(np.array(g["groups"]), np.array(g["idx"]),
                                                g["L"], g["G"], g["F"], g["H"])
    assert st == 0
    assert sol.tolist() == e["slot_of_label"]
    assert los.tolist() == e["label_of_slot"]
    assert ids.tolist() == e["idx_sorted"]
    st, srp, ssl = oracle_mod.pos_slots(np.array(g["pos_rowptr"]), np.array(g["pos_label"]),
                                        g["L"], sol)
    assert st == 0
    assert srp.tolist() == e["srowptr"] and ssl.tolist() == e["sslots"]
    # the same values given as bf16 bits (all exact in bf16)
    for hh, WW in ((h, W), (to_bf16_bits(h), to_bf16_bits(W))):
        Z = oracle_mod.forward(hh, WW, ids, g["G"])
        assert Z.tolist() == e["Z"]
    dZ, loss = oracle_mod.bce(Z, srp, ssl)
    assert dZ[0, 1] == e["dZ_0_1"]
    # BCE by hand with Python's math library
    Y = np.zeros((2, 4))
    Y[0, 1] = Y[1, 0] = Y[1, 3] = 1
    want = 0.0
    for b in range(2):
        for s in range(4):
            z = e["Z"][b][s]
            p = 1.0 / (1.0 + math.exp(-z))
            # -log sigma(z) = log(1 + e^-z);  -log(1 - sigma(z)) = log(1 + e^z)
            want += math.log1p(math.exp(-z)) if Y[b, s] else math.log1p(math.exp(z))
            assert dZ[b, s] == pytest.approx(p - Y[b, s], rel=1e-14, abs=1e-15)
    assert loss == pytest.approx(want, rel=1e-13)
    # feature gradient by hand: dh[b, i] = sum over (slot, f) with I[f] = i
    dh = oracle_mod.feature_grad(W, dZ, ids, g["G"], g["H"])
    I = e["idx_sorted"]
    for b in range(2):
        want_row = [0.0] * 4
        for s in range(4):
            for f in range(2):
                want_row[I[s // 2][f]] += dZ[b, s] * W[s, f]
        assert dh[b].tolist() == pytest.approx(want_row, rel=1e-14, abs=1e-15)
    # weight gradient: dW[s, f] = sum_b dZ[b, s] h[b, I[f]]
    dW = oracle_mod.weight_grad(h, dZ, ids, g["G"], g["F"])
    for s in range(4):
        for f in range(2):
            want_v = sum(dZ[b, s] * h[b, I[s // 2][f]] for b in range(2))
            assert dW[s, f] == pytest.approx(want_v, rel=1e-14, abs=1e-15)


# ------------------------------------------------------------ O1 / O2
@pytest.mark.parametrize("G,F,H", [(1, 3, 7), (4, 5, 16), (16, 32, 256)])
def test_layout_is_stable_sort_by_group(oracle_mod, G, F, H):
    rng = np.random.default_rng(1)
    L = 64 * G
    groups, idx, *_ = _rand_problem(rng, 1, H, L, G, F)
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, F, H)
    assert st == 0
    ref_los = np.argsort(groups, kind="stable")   # library stable sort
    assert np.array_equal(los, ref_los)
    assert np.array_equal(sol[ref_los], np.arange(L))
    assert np.array_equal(ids, np.sort(idx, axis=1))
    # invariants: every slot used once, G labels per group, strictly increasing rows
    assert np.array_equal(np.sort(sol), np.arange(L))
    assert np.all(groups[los] == np.arange(L) // G)
    if F > 1:
        assert np.all(np.diff(ids.astype(np.int64), axis=1) > 0)


def test_layout_rejects_bad_inputs(oracle_mod):
    L, G, F, H = 32, 4, 3, 10
    rng = np.random.default_rng(2)
    groups, idx, *_ = _rand_problem(rng, 1, H, L, G, F)
    assert oracle_mod.layout_build(groups, idx, L, G, F, H)[0] == 0
    bad = groups.copy(); bad[0] = L // G           # group id out of range
    assert oracle_mod.layout_build(bad, idx, L, G, F, H)[0] == oracle_mod.OR_ERR_DATA
    bad = groups.copy(); bad[0] = bad[1] if bad[0] != bad[1] else bad[2]   # unequal group sizes
    if not np.array_equal(bad, groups):
        assert oracle_mod.layout_build(bad, idx, L, G, F, H)[0] == oracle_mod.OR_ERR_DATA
    bad = idx.copy(); bad[3, 1] = bad[3, 0]        # duplicate index
    assert oracle_mod.layout_build(groups, bad, L, G, F, H)[0] == oracle_mod.OR_ERR_DATA
    bad = idx.copy(); bad[5, 2] = H                # index out of range
    assert oracle_mod.layout_build(groups, bad, L, G, F, H)[0] == oracle_mod.OR_ERR_DATA
    assert oracle_mod.layout_build(groups[:30], idx, 30, G, F, H)[0] == oracle_mod.OR_ERR_INVALID


def test_pos_slots_sorted_dedup(oracle_mod):
    rng = np.random.default_rng(3)
    L, B = 50, 6
    sol = rng.permutation(L).astype(np.int32)
    rows = [rng.integers(0, L, size=rng.integers(0, 9)) for _ in range(B)]
    rows[2] = np.array([7, 7, 7])
    rows[4] = np.array([], dtype=np.int64)
    rowptr = np.zeros(B + 1, np.int32)
    rowptr[1:] = np.cumsum([len(r) for r in rows])
    labels = np.concatenate(rows).astype(np.int32)
    st, srp, ssl = oracle_mod.pos_slots(rowptr, labels, L, sol)
    assert st == 0
    for b in range(B):
        assert ssl[srp[b]:srp[b + 1]].tolist() == sorted(set(sol[rows[b]].tolist()))
    bad = labels.copy(); bad[0] = L
    assert oracle_mod.pos_slots(rowptr, bad, L, sol)[0] == oracle_mod.OR_ERR_DATA


# ------------------------------------------------------------ O3 forward
@pytest.mark.parametrize("G,F", [(1, 4), (2, 3), (4, 8), (16, 32)])
def test_forward_equals_densified_matmul(oracle_mod, G, F):
    rng = np.random.default_rng(4)
    B, H, L = 5, 40, 64
    groups, idx, h, W, *_ = _rand_problem(rng, B, H, L, G, F)
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, F, H)
    Z = oracle_mod.forward(h, W, ids, G)
    Wd = _densify(W, np.sort(idx, axis=1), G, H)
    Zref = h @ Wd.T                              # library matmul
    assert np.allclose(Z, Zref, rtol=1e-12, atol=1e-12)


def test_forward_bitwise_equals_naive_dense_loop(oracle_mod):
    """Ascending-column dense loop adds the same nonzero terms in the same
    order plus exact zeros, so the result is bitwise equal."""
    rng = np.random.default_rng(5)
    B, H, L, G, F = 3, 12, 16, 4, 5
    groups, idx, h, W, *_ = _rand_problem(rng, B, H, L, G, F)
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, F, H)
    Z = oracle_mod.forward(h, W, ids, G)
    Wd = _densify(W, np.sort(idx, axis=1), G, H)
    for b in range(B):
        for s in range(L):
            acc = 0.0
            for i in range(H):
                if Wd[s, i] != 0.0:
                    acc += Wd[s, i] * h[b, i]
            assert Z[b, s] == acc


def test_forward_g1_is_per_label_fan_in(oracle_mod):
    rng = np.random.default_rng(6)
    B, H, L, F = 4, 30, 20, 6
    groups, idx, h, W, *_ = _rand_problem(rng, B, H, L, 1, F)
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, 1, F, H)
    Z = oracle_mod.forward(h, W, ids, 1)
    # per-label fixed fan-in: label l owns index set idx[groups[l]] and the
    # weights stored at its slot; summation order of the set is irrelevant
    for l in range(L):
        s = sol[l]
        I = idx[groups[l]]
        w = W[s][np.argsort(np.argsort(I))]      # weights follow sorted order
        for b in range(B):
            assert Z[b, s] == pytest.approx(sum(wv * h[b, i] for wv, i in zip(w, I)), rel=1e-13)


def test_forward_dense_special_case(oracle_mod):
    """F = H and every I_k = [0, H): the layer is the dense layer Z = h W^T."""
    rng = np.random.default_rng(7)
    B, H, L, G = 3, 16, 32, 8
    K = L // G
    groups = (rng.permutation(L) // G).astype(np.int32)
    idx = np.stack([rng.permutation(H) for _ in range(K)]).astype(np.int32)
    h = rng.standard_normal((B, H))
    W = rng.standard_normal((L, H))
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, H, H)
    Z = oracle_mod.forward(h, W, ids, G)
    assert np.allclose(Z, h @ W.T, rtol=1e-12, atol=1e-12)


def test_forward_block_sparse_special_case(oracle_mod):
    """Every group bound to the same contiguous block [c, c+F): block sparse."""
    rng = np.random.default_rng(8)
    B, H, L, G, F, c = 3, 40, 24, 4, 8, 13
    K = L // G
    groups = (rng.permutation(L) // G).astype(np.int32)
    idx = np.stack([rng.permutation(np.arange(c, c + F)) for _ in range(K)]).astype(np.int32)
    h = rng.standard_normal((B, H))
    W = rng.standard_normal((L, F))
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, F, H)
    Z = oracle_mod.forward(h, W, ids, G)
    assert np.allclose(Z, h[:, c:c + F] @ W.T, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ O4 BCE
def test_bce_closed_forms(oracle_mod):
    assert oracle_mod.sigmoid(0.0) == 0.5
    assert oracle_mod.bce_term(0.0, 0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert oracle_mod.bce_term(0.0, 1) == pytest.approx(math.log(2.0), rel=1e-15)
    for z in (0.3, 2.0, 7.5):
        # l(z,1) = -log sigma(z), l(z,0) = -log(1 - sigma(z)) (textbook forms)
        p = 1.0 / (1.0 + math.exp(-z))
        assert oracle_mod.bce_term(z, 1) == pytest.approx(-math.log(p), rel=1e-12)
        assert oracle_mod.bce_term(z, 0) == pytest.approx(-math.log1p(-p), rel=1e-12)
        assert oracle_mod.bce_term(-z, 0) == pytest.approx(oracle_mod.bce_term(z, 1), rel=1e-15)
        assert oracle_mod.sigmoid(-z) == pytest.approx(1.0 - oracle_mod.sigmoid(z), rel=1e-14)
    # saturation stays finite and exact to the leading term
    assert oracle_mod.bce_term(100.0, 0) == pytest.approx(100.0, rel=1e-15)
    assert oracle_mod.bce_term(-100.0, 1) == pytest.approx(100.0, rel=1e-15)
    assert 0.0 < oracle_mod.bce_term(100.0, 1) < 1e-40
    assert oracle_mod.sigmoid(-800.0) == 0.0 and oracle_mod.sigmoid(800.0) == 1.0


def test_bce_gradient_finite_difference(oracle_mod):
    rng = np.random.default_rng(9)
    B, L = 3, 7
    Z = rng.standard_normal((B, L)) * 2
    srp = np.array([0, 2, 2, 3], np.int32)
    ssl = np.array([1, 5, 0], np.int32)
    dZ, loss = oracle_mod.bce(Z, srp, ssl)
    eps = 1e-6
    for b in range(B):
        for s in range(L):
            Zp = Z.copy(); Zp[b, s] += eps
            Zm = Z.copy(); Zm[b, s] -= eps
            fd = (oracle_mod.bce(Zp, srp, ssl)[1] - oracle_mod.bce(Zm, srp, ssl)[1]) / (2 * eps)
            assert fd == pytest.approx(dZ[b, s], rel=1e-6, abs=1e-9)


# ------------------------------------------------------------ O5 / O6 gradients
@pytest.mark.parametrize("G,F", [(1, 2), (2, 3), (4, 4), (2, 2)])
def test_gradients_finite_difference(oracle_mod, G, F):
    rng = np.random.default_rng(10 + G * 7 + F)
    B, H, L = 2, 8, 8
    groups, idx, h, W, rowptr, labels = _rand_problem(rng, B, H, L, G, F, npos=2)
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, F, H)
    st, srp, ssl = oracle_mod.pos_slots(rowptr, labels, L, sol)
    Z = oracle_mod.forward(h, W, ids, G)
    dZ, loss = oracle_mod.bce(Z, srp, ssl)
    dW = oracle_mod.weight_grad(h, dZ, ids, G, F)
    dh = oracle_mod.feature_grad(W, dZ, ids, G, H)
    eps = 1e-6
    for s in range(L):
        for f in range(F):
            Wp = W.copy(); Wp[s, f] += eps
            Wm = W.copy(); Wm[s, f] -= eps
            fd = (_loss(oracle_mod, h, Wp, ids, G, srp, ssl)[1] -
                  _loss(oracle_mod, h, Wm, ids, G, srp, ssl)[1]) / (2 * eps)
            assert fd == pytest.approx(dW[s, f], rel=1e-6, abs=1e-8)
    for b in range(B):
        for i in range(H):
            hp = h.copy(); hp[b, i] += eps
            hm = h.copy(); hm[b, i] -= eps
            fd = (_loss(oracle_mod, hp, W, ids, G, srp, ssl)[1] -
                  _loss(oracle_mod, hm, W, ids, G, srp, ssl)[1]) / (2 * eps)
            assert fd == pytest.approx(dh[b, i], rel=1e-6, abs=1e-8)


def test_gradients_dense_restatement(oracle_mod):
    """dW[s, f] = (dZ^T h)[s, I_k(s)[f]] and dh = dZ Wd (library matmuls)."""
    rng = np.random.default_rng(11)
    B, H, L, G, F = 6, 24, 48, 4, 7
    groups, idx, h, W, rowptr, labels = _rand_problem(rng, B, H, L, G, F)
    st, sol, los, ids = oracle_mod.layout_build(groups, idx, L, G, F, H)
    dZ = rng.standard_normal((B, L))
    dW = oracle_mod.weight_grad(h, dZ, ids, G, F)
    dh = oracle_mod.feature_grad(W, dZ, ids, G, H)
    full = dZ.T @ h
    I = np.sort(idx, axis=1)
    for s in range(L):
        assert np.allclose(dW[s], full[s, I[s // G]], rtol=1e-12, atol=1e-12)
    Wd = _densify(W, I, G, H)
    assert np.allclose(dh, dZ @ Wd, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ sampled forms
def test_sampled_functions_match_full(oracle_mod):
    w = CONFIGS["tiny"]
    p = generate(w)
    full = oracle_mod.step(p, want_Z=True)
    ids, srp, ssl = full["idx_sorted"], full["srowptr"], full["sslots"]
    rng = np.random.default_rng(12)
    bs = rng.integers(0, w.B, 50).astype(np.int32)
    ss = rng.integers(0, w.L, 50)
    zat = oracle_mod.forward_at(p.h, p.W, ids, w.G, bs, ss)
    assert np.array_equal(zat, full["Z"][bs, ss])
    slots = np.array([0, 17, w.L - 1] + [int(x) for x in ssl[:3]])
    dWr = oracle_mod.weight_grad_rows(p.h, p.W, ids, w.G, srp, ssl, slots)
    assert np.allclose(dWr, full["dW"][slots], rtol=1e-12, atol=1e-12)
    rows = np.array([0, 5, w.B - 1], np.int32)
    dhr, rl = oracle_mod.feature_grad_rows(p.h, p.W, ids, w.G, srp, ssl, rows)
    assert np.allclose(dhr, full["dh"][rows], rtol=1e-11, atol=1e-11)
    _, rl_all = oracle_mod.feature_grad_rows(p.h, p.W, ids, w.G, srp, ssl,
                                             np.arange(w.B, dtype=np.int32), want_dh=False)
    assert rl_all.sum() == pytest.approx(full["loss"], rel=1e-12)


def test_bf16_widening_is_exact(oracle_mod):
    vals = np.array([0.0, 1.0, -2.5, 3.140625, 1e-30, -7e20], dtype=np.float32)
    bits = to_bf16_bits(vals)
    for b, v in zip(bits, bf16_bits_to_f32(bits)):
        assert oracle_mod.bf16_value(int(b)) == float(v)


# ------------------------------------------------------------------ O7: momentum SGD
def test_sgd_momentum_matches_torch_optimizer(oracle_mod):
    """The output layer's momentum SGD (Loss and training strategy) against an
    independent implementation: torch.optim.SGD (heavy ball, no dampening, no
    weight decay) in double, three steps with the momentum carried.  Each step
    starts torch from the oracle's bf16 weights, so the double update must
    round to the same bf16 and the momentum must agree exactly."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    shape = (64, 48)
    W = to_bf16_bits(rng.standard_normal(shape) * 0.1)
    m = np.zeros(shape)
    lr, mu = 0.05, 0.9
    p = torch.nn.Parameter(torch.zeros(shape, dtype=torch.float64))
    opt = torch.optim.SGD([p], lr=lr, momentum=mu, dampening=0.0, nesterov=False, weight_decay=0.0)
    for step in range(3):
        g = rng.standard_normal(shape)
        with torch.no_grad():
            p.copy_(torch.from_numpy(bf16_bits_to_f32(W).astype(np.float64)))
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        W, m = oracle_mod.sgd_momentum(W, g, m, lr, mu)
        buf = opt.state[p]["momentum_buffer"].numpy()
        np.testing.assert_array_equal(m, buf)
        assert np.array_equal(W, to_bf16_bits(p.detach().numpy())), step


def test_sgd_momentum_special_cases(oracle_mod):
    """lr = 0 leaves W bit-identical; mu = 0 makes the momentum the gradient
    itself (plain SGD: W - lr dW, rounded once to bf16)."""
    rng = np.random.default_rng(11)
    W = to_bf16_bits(rng.standard_normal((16, 32)))
    g = rng.standard_normal((16, 32))
    m0 = rng.standard_normal((16, 32))
    W1, m1 = oracle_mod.sgd_momentum(W, g, m0, 0.0, 0.5)
    assert np.array_equal(W1, W)
    np.testing.assert_array_equal(m1, 0.5 * m0 + g)
    W2, m2 = oracle_mod.sgd_momentum(W, g, m0, 0.25, 0.0)
    np.testing.assert_array_equal(m2, g)
    assert np.array_equal(W2, to_bf16_bits(bf16_bits_to_f32(W).astype(np.float64) - 0.25 * g))
