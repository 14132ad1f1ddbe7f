"""The head-tail split of the output layer on the GPU, against the CPU oracle
(oracle/head_tail.py), through the C ABI.

HASTE, "Method / overall framework" and "Key designs / head-tail split": the
encoder output h feeds a dense head and the group-shared sparse tail through
two projections; the loss is the sum of both branches' BCE terms.  The library
runs the projections and their backward as tcgen05 GEMMs and the head as the
layer itself with every group's index set [0, Dh).

Precision: the layer takes bf16 inputs, so the projected activations h_head
and h_tail are rounded to bf16; the oracle takes the same reading
(hidden_bf16=True) and otherwise stays in double.  The layer's tolerance
max |gpu - ref| <= 2e-2 (1 + |ref|) applies to dW_head, dW_tail and the loss.
dP and dh are products of the branch gradients dh_head, dh_tail, and those
come from dZ rounded to fp16 (unit roundoff 2^-11), so each of their entries
may be off by up to 2^-11 times the same sum taken over absolute values
(|dZ| |W|).  Summed again over the batch (dP) or the projection rows (dh), that
bound can exceed the result itself where terms cancel; the check for dP and dh
adds it, computed from the oracle's dZ, dA and weights, to the tolerance.
The branch gradients enter the backward GEMMs as two bf16 planes (about 16
bits), well inside it.
"""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import Workload, draw_bf16_matrix, generate, to_bf16_bits

from gpu_common import LOSS_RTOL, assert_close, build_layout, dev_bf16, dev_i32, host_bf16_to_f64

pytestmark = pytest.mark.gpu


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _assert_close_bound(gpu, ref, bound, what):
    """max |gpu - ref| <= 2e-2 (1 + |ref|) + bound, element by element."""
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref) - 2e-2 * (1.0 + np.abs(ref)) - bound
    worst = int(np.argmax(err))
    assert err.flat[worst] <= 0, (f"{what}: max violation at {np.unravel_index(worst, err.shape)}: "
                                  f"gpu={gpu.flat[worst]!r} ref={ref.flat[worst]!r} bound={bound.flat[worst]!r}")


def _scaled_bf16(seed, rows, cols, scale):
    return draw_bf16_matrix(seed, rows, cols, scale)


@pytest.mark.parametrize("B,E,D", [(64, 256, 256), (37, 136, 40), (128, 768, 768), (300, 200, 136)])
def test_proj_fwd_bwd_against_oracle(oracle_mod, B, E, D):
    """sg_proj_fwd and sg_proj_bwd alone: out = bf16(h P^T), dP = g^T h,
    dh = g P (and dh += g P), against double products of the same inputs."""
    from oracle import head_tail as ht
    sg.build()
    h = _scaled_bf16(1, B, E, 1.0)
    P = _scaled_bf16(2, D, E, 1.0 / np.sqrt(E))
    g = np.random.default_rng(3).standard_normal((B, D)).astype(np.float32)
    out = torch.empty((B, D), dtype=torch.int16, device="cuda")
    sg.sg_proj_fwd(dev_bf16(h), dev_bf16(P), out)
    work = torch.empty(2 * B * D, dtype=torch.int16, device="cuda")
    dP = torch.empty((D, E), dtype=torch.float32, device="cuda")
    dh = torch.full((B, E), 0.5, dtype=torch.float32, device="cuda")
    gd = torch.from_numpy(g).cuda()
    sg.sg_proj_bwd(dev_bf16(h), dev_bf16(P), gd, work, dP, dh, accumulate_dh=True)
    torch.cuda.synchronize()
    zeros_head = np.zeros((B, 8))
    ref = ht.projections_backward(h, np.zeros((8, E), np.uint16), P, zeros_head, g.astype(np.float64))
    assert_close(host_bf16_to_f64(out), _f64(h) @ _f64(P).T, tol=8e-3, what="h P^T")
    assert_close(dP.cpu().numpy(), ref["dP_tail"], tol=2e-3, what="dP")
    assert_close(dh.cpu().numpy(), ref["dh"] + 0.5, tol=2e-3, what="dh (accumulated)")
    sg.sg_proj_bwd(dev_bf16(h), dev_bf16(P), gd, work, dP, dh, accumulate_dh=False)
    torch.cuda.synchronize()
    assert_close(dh.cpu().numpy(), ref["dh"], tol=2e-3, what="dh (overwritten)")


def _head_problem(B, Dh, Lh, Gh, seed):
    """The head as a layer: groups of Gh consecutive labels, every index row
    [0, Dh), dense positives Y_head drawn with rate 0.05 (at least one sample
    row left empty)."""
    rng = np.random.default_rng(seed)
    W_head = _scaled_bf16(seed + 10, Lh, Dh, 1.0 / np.sqrt(Dh))
    Y = rng.random((B, Lh)) < 0.05
    Y[0] = False
    rowptr = np.zeros(B + 1, np.int32)
    labels = []
    for b in range(B):
        row = np.flatnonzero(Y[b]).astype(np.int32)
        rng.shuffle(row)  # the layer takes unsorted rows
        labels.extend(row.tolist())
        rowptr[b + 1] = len(labels)
    groups = (np.arange(Lh) // Gh).astype(np.int32)
    idx = np.tile(np.arange(Dh, dtype=np.int32), (Lh // Gh, 1))
    return W_head, Y.astype(np.float64), groups, idx, rowptr, np.asarray(labels, np.int32)


HT_CASES = [
    # B, E, Dh, Lh, Gh, tail workload (H, L, G, F, pos)
    (64, 256, 64, 128, 16, (256, 32 * 120, 32, 64, 8)),
    (37, 264, 32, 96, 32, (128, 16 * 90 + 16, 16, 32, 5)),
    (128, 768, 128, 512, 16, (768, 32 * 300, 32, 128, 36)),
]


@pytest.mark.parametrize("case", HT_CASES, ids=lambda c: f"B{c[0]}_E{c[1]}_Dh{c[2]}_H{c[5][0]}")
def test_headtail_step_against_oracle(oracle_mod, case):
    from oracle import head_tail as ht
    sg.build()
    B, E, Dh, Lh, Gh, (H, L, G, F, pos) = case
    tw = Workload("ht_tail", B=B, H=H, L=L, G=G, F=F, pos=pos, pos_dist="zipf", zipf_s=1.1,
                  idx_mode="uniform", seed=5)
    tp = generate(tw)
    h = _scaled_bf16(21, B, E, 1.0)
    P_head = _scaled_bf16(22, Dh, E, 1.0 / np.sqrt(E))
    P_tail = _scaled_bf16(23, H, E, 1.0 / np.sqrt(E))
    W_head, Y_head, hgroups, hidx, hrp, hlab = _head_problem(B, Dh, Lh, Gh, 31)
    ref = ht.step(h, P_head, P_tail, W_head, Y_head, tp.W, tp.groups, tp.idx, G, F, tp.pos_rowptr,
                  tp.pos_label, hidden_bf16=True)

    # absolute-value bounds of the branch gradients' fp16 rounding of dZ
    u16 = 2.0 ** -11
    hf, Ph, Pt = _f64(h), _f64(P_head), _f64(P_tail)
    abs_dh_head = np.abs(ref["dA"]) @ np.abs(_f64(W_head))
    abs_dh_tail = oracle_mod.feature_grad(np.abs(_f64(tp.W)), np.abs(ref["dZ"]), ref["idx_sorted"], G, H)
    bound_dP_head = u16 * (abs_dh_head.T @ np.abs(hf))
    bound_dP_tail = u16 * (abs_dh_tail.T @ np.abs(hf))
    bound_dh = u16 * (abs_dh_head @ np.abs(Ph) + abs_dh_tail @ np.abs(Pt))

    head = sg.sg_layout_build(dev_i32(hgroups), Lh, Gh, dev_i32(hidx.reshape(-1)), Dh, Dh, B,
                              max(int(hrp[-1]), 1))
    tail = build_layout(tp)
    try:
        hsol = sg.sg_layout_export(head)[0].cpu().numpy()
        W_head_slots = np.empty_like(W_head)
        W_head_slots[hsol] = W_head
        dW_head = torch.empty((Lh, Dh), dtype=torch.int16, device="cuda")
        dW_tail = torch.empty((L, F), dtype=torch.int16, device="cuda")
        dP_head = torch.empty((Dh, E), dtype=torch.float32, device="cuda")
        dP_tail = torch.empty((H, E), dtype=torch.float32, device="cuda")
        dh = torch.full((B, E), float("nan"), dtype=torch.float32, device="cuda")
        loss = torch.zeros(1, dtype=torch.float64, device="cuda")
        hl = hlab if len(hlab) else np.zeros(1, np.int32)
        tl = tp.pos_label if tp.nnz else np.zeros(1, np.int32)
        for _ in range(2):  # twice: scratch reuse must not carry state
            sg.sg_headtail_step(head, tail, dev_bf16(h), dev_bf16(P_head), dev_bf16(P_tail),
                                dev_bf16(W_head_slots), dev_i32(hrp), dev_i32(hl), int(hrp[-1]),
                                dev_bf16(tp.W), dev_i32(tp.pos_rowptr), dev_i32(tl), tp.nnz, dW_head,
                                dW_tail, dP_head, dP_tail, dh, loss)
            torch.cuda.synchronize()
            assert sg.sg_layout_status(head) == 0 and sg.sg_layout_status(tail) == 0
            assert_close(host_bf16_to_f64(dW_head)[hsol], ref["dW_head"], what="dW_head")
            assert_close(host_bf16_to_f64(dW_tail), ref["dW_tail"], what="dW_tail")
            _assert_close_bound(dP_head.cpu().numpy(), ref["dP_head"], bound_dP_head, "dP_head")
            _assert_close_bound(dP_tail.cpu().numpy(), ref["dP_tail"], bound_dP_tail, "dP_tail")
            _assert_close_bound(dh.cpu().numpy(), ref["dh"], bound_dh, "dh")
            assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)
    finally:
        head.close()
        tail.close()


def test_headtail_rejects_bad_sizes():
    sg.build()
    import ctypes as C
    lib = sg.load()
    rc = lib.sg_proj_fwd(C.c_void_p(16), 4, 12, C.c_void_p(16), 8, C.c_void_p(16), None)
    assert rc == sg.SG_ERR_INVALID and "multiples of 8" in sg.last_error()
