"""Full-size parity: every workload at its real size, run through sg_step as
bench.py runs it (engine chosen automatically), checked against the oracle on
outputs it can compute one by one -- the layout (bit-exact), dW rows of
sampled slots (including slots with positives), dh rows of sampled samples --
and on the loss summed over every (sample, label)."""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import CONFIGS, generate

from gpu_common import LOSS_RTOL, assert_close, build_layout, dev_problem, host_bf16_to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FULL = ["amazon670k_tail", "amazon3m_tail", "lf8p6m_tail", "sweep_g1_uniform",
        "sweep_g16_clustered", "sweep_g32_uniform", "sweep_g64_clustered"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_step_sampled(name, oracle_mod):
    sg.build()
    w = CONFIGS[name]
    p = generate(w)
    st, sol, los, ids = oracle_mod.layout_build(p.groups, p.idx, w.L, w.G, w.F, w.H)
    assert st == 0
    st, srp, ssl = oracle_mod.pos_slots(p.pos_rowptr, p.pos_label, w.L, sol)
    assert st == 0

    lay = build_layout(p)
    g_sol, g_los, g_ids = sg.sg_layout_export(lay)
    assert np.array_equal(g_sol.cpu().numpy(), sol)
    assert np.array_equal(g_los.cpu().numpy(), los)
    assert np.array_equal(g_ids.cpu().numpy().view(np.uint16), ids)

    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
    torch.cuda.synchronize()
    assert sg.sg_layout_status(lay) == 0

    rng = np.random.default_rng(2024)
    slots = np.unique(np.concatenate([rng.integers(0, w.L, 48), ssl[:16], [0, w.L - 1]]))
    want_dW = oracle_mod.weight_grad_rows(p.h, p.W, ids, w.G, srp, ssl, slots)
    got_dW = host_bf16_to_f64(dW[torch.from_numpy(slots).cuda()])
    assert_close(got_dW, want_dW, what=f"{name} dW rows")

    rows = np.array(sorted({0, w.B - 1, int(rng.integers(0, w.B))}), dtype=np.int32)
    want_dh, _ = oracle_mod.feature_grad_rows(p.h, p.W, ids, w.G, srp, ssl, rows)
    got_dh = dh.cpu().numpy()[rows].astype(np.float64)
    assert_close(got_dh, want_dh, what=f"{name} dh rows")

    _, row_loss = oracle_mod.feature_grad_rows(p.h, p.W, ids, w.G, srp, ssl,
                                               np.arange(w.B, dtype=np.int32), want_dh=False)
    assert float(loss.item()) == pytest.approx(float(row_loss.sum()), rel=LOSS_RTOL)
    lay.close()
