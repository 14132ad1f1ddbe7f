"""Run-to-run determinism and the layout round trip (checkpoint / resume).

dW is computed per group without atomics (tensor cores: one MMA chain per
group; CUDA cores: one thread per output), and the loss is summed in a fixed
order, so two runs of the same step give the same bits.  dh is accumulated
with atomics across CTAs and may differ in its last bits.  A layout exported
with sg_layout_export and built again from what it exported (groups from the
slot maps, the sorted index rows) is the same layout and gives the same step.
"""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import Workload, generate

from gpu_common import assert_close, build_layout, dev_i32, dev_problem, host_bf16_to_f64

pytestmark = pytest.mark.gpu

SHAPES = [
    ("two_kernel", Workload("d1", B=128, H=768, L=32 * 300, G=32, F=128, pos=36, pos_dist="zipf", zipf_s=1.1,
                            idx_mode="uniform")),
    ("one_kernel", Workload("d2", B=70, H=200, L=32 * 45, G=32, F=48, pos=3, pos_dist="uniform", zipf_s=1.1,
                            idx_mode="uniform")),
    ("streamed_dW", Workload("d3", B=256, H=768, L=64 * 40, G=64, F=128, pos=5, pos_dist="zipf", zipf_s=1.1,
                             idx_mode="uniform")),
    ("cuda_cores_g5", Workload("d4", B=33, H=64, L=5 * 41, G=5, F=24, pos=2, pos_dist="uniform", zipf_s=1.1,
                               idx_mode="uniform")),
    ("per_label", Workload("d5", B=100, H=256, L=700, G=1, F=64, pos=4, pos_dist="zipf", zipf_s=1.1,
                           idx_mode="uniform")),
    ("paired_groups", Workload("d6", B=48, H=256, L=32 * 40, G=32, F=64, pos=4, pos_dist="zipf", zipf_s=1.1,
                               idx_mode="uniform")),
]


def _step(lay, p, d):
    w = p.w
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
    torch.cuda.synchronize()
    return dW.cpu().numpy().copy(), dh.cpu().numpy().copy(), float(loss.item())


@pytest.mark.parametrize("name,w", SHAPES, ids=[s[0] for s in SHAPES])
def test_dW_and_loss_are_bit_identical_across_runs(name, w):
    sg.build()
    p = generate(w)
    lay = build_layout(p)
    try:
        d = dev_problem(p)
        dW1, dh1, l1 = _step(lay, p, d)
        dW2, dh2, l2 = _step(lay, p, d)
        assert sg.sg_layout_status(lay) == 0
    finally:
        lay.close()
    np.testing.assert_array_equal(dW1, dW2)
    assert l1 == l2
    np.testing.assert_allclose(dh1, dh2, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("name,w", SHAPES[:3] + SHAPES[4:], ids=[s[0] for s in SHAPES[:3] + SHAPES[4:]])
def test_layout_export_and_rebuild(name, w):
    """Export the layout, build a new one from the export alone (group of a
    label = its slot // G; index rows as exported), and compare the maps and
    a step on both."""
    sg.build()
    p = generate(w)
    lay = build_layout(p)
    lay2 = None
    try:
        sol, los, ids = sg.sg_layout_export(lay)
        groups = (sol // w.G).to(torch.int32)
        idx = ids.view(torch.int16).to(torch.int32) & 0xFFFF
        lay2 = sg.sg_layout_build(groups, w.L, w.G, idx.reshape(-1).contiguous(), w.F, w.H, w.B, max(p.nnz, 1))
        sol2, los2, ids2 = sg.sg_layout_export(lay2)
        assert torch.equal(sol, sol2) and torch.equal(los, los2) and torch.equal(ids, ids2)
        d = dev_problem(p)
        dW1, dh1, l1 = _step(lay, p, d)
        dW2, dh2, l2 = _step(lay2, p, d)
        np.testing.assert_array_equal(dW1, dW2)
        assert l1 == l2
        assert_close(dh2, dh1, tol=1e-5, what="dh after the round trip")
    finally:
        lay.close()
        if lay2 is not None:
            lay2.close()
