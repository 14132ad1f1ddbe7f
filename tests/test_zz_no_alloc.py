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
from workloads import Workload, draw_bf16_matrix, generate

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
