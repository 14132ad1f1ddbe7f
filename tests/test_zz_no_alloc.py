"""The allocation-free BCE entry point (sg_bce_grad_noalloc) against the
regular sg_bce_grad, through the C ABI.

Some callers cannot allocate device memory: a framework's caching allocator
may already own all of it, or a deployment may forbid allocation after
start-up.  For them the library offers one entry point whose working memory is
a fixed device array built into the library.  This file runs last so that a
failure here stops a `-x` run only after every other test has run; it passes
alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import Workload, bf16_bits_to_f32, draw_bf16_matrix, generate

from gpu_common import LOSS_RTOL, assert_close, build_layout, dev_bf16, dev_i32, host_bf16_to_f64

pytestmark = pytest.mark.gpu


def _slots_csr(p, sol):
    """The problem's positives as slot ids (label -> slot on the host)."""
    return p.pos_rowptr.astype(np.int32), sol[p.pos_label].astype(np.int32)


def _case(seed):
    w = Workload("noalloc", B=96, H=256, L=32 * 700, G=32, F=64, pos=12, pos_dist="zipf",
                 zipf_s=1.1, idx_mode="uniform", seed=seed)
    p = generate(w)
    lay = build_layout(p)
    sol = sg.sg_layout_export(lay)[0].cpu().numpy()
    Z = dev_bf16(draw_bf16_matrix(100 + seed, w.B, w.L, 3.0))
    return w, p, lay, sol, Z


def _reference(w, p, lay, Z):
    dZ = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_bce_grad(lay, Z, w.B, dev_i32(p.pos_rowptr), dev_i32(p.pos_label), p.nnz, dZ, loss)
    return host_bf16_to_f64(dZ), float(loss.item())


def test_noalloc_matches_bce_grad_on_two_calls():
    sg.build()
    runs = []
    for seed in (0, 1):
        w, p, lay, sol, Z = _case(seed)
        want_dZ, want_loss = _reference(w, p, lay, Z)
        rp, slots = _slots_csr(p, sol)
        runs.append((w, Z, rp, slots, p.nnz, want_dZ, want_loss))
    # the same call twice in a row, then the other problem: the shared
    # working array must not carry anything from one call to the next
    for w, Z, rp, slots, nnz, want_dZ, want_loss in (runs[0], runs[0], runs[1]):
        dZ = torch.full((w.B, w.L), 0x7fc0, dtype=torch.int16, device="cuda")
        loss = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
        sg.sg_bce_grad_noalloc(Z, w.B, w.L, w.G, dev_i32(rp), dev_i32(slots), nnz, dZ, loss)
        torch.cuda.synchronize()
        assert_close(host_bf16_to_f64(dZ), want_dZ, what="dZ")
        assert float(loss.item()) == pytest.approx(want_loss, rel=LOSS_RTOL)


def test_noalloc_rejects_sizes_above_its_limits():
    sg.build()
    Z = torch.zeros(8, dtype=torch.int16, device="cuda")
    rp = torch.zeros(2, dtype=torch.int32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    big_L = 16 * 400000  # L / G above the fixed limit
    lib = sg.load()
    import ctypes as C
    rc = lib.sg_bce_grad_noalloc(C.c_void_p(Z.data_ptr()), 1, big_L, 16, C.c_void_p(rp.data_ptr()),
                                 None, 0, C.c_void_p(Z.data_ptr()), C.c_void_p(loss.data_ptr()), None)
    assert rc == sg.SG_ERR_UNSUPPORTED
    assert "limits" in sg.last_error()


def _canonical(rowptr, slots, nnz, L):
    """What the entry point promises to use as Y: per sample, the valid
    in-range slots of a well-formed row, deduplicated and sorted (the oracle's
    positive lists); malformed rows (r0 < 0, r1 < r0, r1 > nnz, or a start
    below an earlier row's start, which could overlap it) are empty."""
    B = len(rowptr) - 1
    out_rp = [0]
    out = []
    for b in range(B):
        r0, r1 = int(rowptr[b]), int(rowptr[b + 1])
        row = []
        if 0 <= r0 <= r1 <= nnz and all(r0 >= int(rowptr[c]) for c in range(b)):
            row = sorted({int(v) for v in slots[r0:r1] if 0 <= int(v) < L})
        out.extend(row)
        out_rp.append(len(out))
    return np.array(out_rp, dtype=np.int32), np.array(out, dtype=np.int32)


def _noalloc(Zbits, B, L, G, rowptr, slots, nnz):
    dZ = torch.full((B, L), 0x7fc0, dtype=torch.int16, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
    sl = slots if len(slots) else np.zeros(1, np.int32)
    sg.sg_bce_grad_noalloc(dev_bf16(Zbits), B, L, G, dev_i32(rowptr), dev_i32(sl), nnz, dZ, loss)
    torch.cuda.synchronize()
    return host_bf16_to_f64(dZ), float(loss.item())


def test_noalloc_matches_oracle_on_two_calls(oracle_mod):
    """Element by element against the CPU oracle's BCE (dZ = sigmoid(Z) - Y and
    the summed loss), the same call twice in a row: the shared working array
    is cleared by every call."""
    sg.build()
    B, L, G = 64, 32 * 300, 32
    Zbits = draw_bf16_matrix(7, B, L, 3.0)
    rng = np.random.default_rng(11)
    rowptr = np.zeros(B + 1, np.int32)
    rowptr[1:] = np.cumsum(rng.integers(0, 9, B))
    slots = rng.integers(0, L, int(rowptr[-1])).astype(np.int32)
    crp, csl = _canonical(rowptr, slots, int(rowptr[-1]), L)
    want_dZ, want_loss = oracle_mod.bce(Zbits, crp, csl)
    for _ in range(2):
        got_dZ, got_loss = _noalloc(Zbits, B, L, G, rowptr, slots, int(rowptr[-1]))
        assert_close(got_dZ, want_dZ, what="dZ")
        assert got_loss == pytest.approx(want_loss, rel=LOSS_RTOL)


def test_noalloc_edge_cases_against_oracle(oracle_mod):
    """The behaviour the header documents for this entry point, against the
    oracle on the positive lists it promises to use: duplicate slots count
    once, slots outside [0, L) (including negative ones) are dropped, a
    malformed row is dropped whole, rowptr[0] may be non-zero, and nnz = 0
    leaves every sample without positives."""
    sg.build()
    B, L, G = 6, 16 * 40, 16
    Zbits = draw_bf16_matrix(5, B, L, 2.0)
    # rowptr[0] = 1; sample 0: a duplicate (7); 1: out of range (>= L and
    # negative) and a duplicate; 2: empty; 3: malformed (its end before its
    # start); 4: starts inside sample 1 (overlap: dropped); 5: ordinary with a
    # duplicate
    slots = np.array([9,            # before rowptr[0]: never read
                      7, 7, 3, 12,
                      L, -4, 12, 0,
                      99, 101, 5, 600, 600], dtype=np.int32)
    rowptr = np.array([1, 5, 9, 9, 7, 11, 14], dtype=np.int32)
    nnz = len(slots)
    crp, csl = _canonical(rowptr, slots, nnz, L)
    want_dZ, want_loss = oracle_mod.bce(Zbits, crp, csl)
    got_dZ, got_loss = _noalloc(Zbits, B, L, G, rowptr, slots, nnz)
    assert_close(got_dZ, want_dZ, what="dZ")
    assert got_loss == pytest.approx(want_loss, rel=LOSS_RTOL)
    # nnz = 0: no positives anywhere
    want0_dZ, want0_loss = oracle_mod.bce(Zbits, np.zeros(B + 1, np.int32), np.zeros(0, np.int32))
    got0_dZ, got0_loss = _noalloc(Zbits, B, L, G, np.zeros(B + 1, np.int32), np.zeros(0, np.int32), 0)
    assert_close(got0_dZ, want0_dZ, what="dZ (nnz = 0)")
    assert got0_loss == pytest.approx(want0_loss, rel=LOSS_RTOL)
    # every sample's dZ is sigmoid(Z) - Y: the positives the oracle used are
    # exactly the de-duplicated valid ones (a spot check of the reading)
    z = bf16_bits_to_f32(Zbits).astype(np.float64)
    assert abs(got_dZ[0, 12] - (1 / (1 + np.exp(-z[0, 12])) - 1)) <= 2e-2
