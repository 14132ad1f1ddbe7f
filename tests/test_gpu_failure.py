"""Failure detection on the GPU, without faulting it: a kernel's bounded wait
on a barrier that nothing completes gives up, records SG_ERR_TIMEOUT, frees
its TMEM and returns; the context stays usable for the next call."""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import CONFIGS, generate

from gpu_common import LOSS_RTOL, assert_close, build_layout, dev_problem, host_bf16_to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_context_survives(oracle_mod):
    sg.build()
    assert sg.sg_selftest_wait_timeout() == sg.SG_ERR_TIMEOUT
    # the context is still usable: a full step on a fresh layout matches the oracle
    w = CONFIGS["tiny"]
    p = generate(w)
    ref = oracle_mod.step(p)
    lay = build_layout(p)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
    assert sg.sg_layout_status(lay) == 0
    assert_close(host_bf16_to_f64(dW), ref["dW"], what="dW")
    assert_close(dh.cpu().numpy(), ref["dh"], what="dh")
    assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)
