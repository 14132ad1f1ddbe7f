"""CPU oracle for the head-tail split of the output layer.

TEST INFRASTRUCTURE ONLY: the tests may import this module; the product library
never does.  Plain numpy in float64 (a matrix product is the only library
primitive used); bf16 inputs are widened exactly.

HASTE, "Method / overall framework" and "Key designs / head-tail split":
the encoder output h (B x E) feeds two branches through light projections,
    h_head = h P_head^T   (P_head: Dh x E),   h_tail = h P_tail^T   (P_tail: H x E);
the head's frequent labels get dense logits a_H = h_head W_head^T (W_head:
Lh x Dh), the tail's labels the group-shared fixed fan-in layer on h_tail, and
the objective is the sum of both branches' BCE terms (the page writes a 1/n
mean; the sum is the reading taken for the whole library, so every gradient
is the exact gradient of the returned loss).  Backward, by the chain rule:
    dA_H      = sigmoid(a_H) - Y_H
    dW_head   = dA_H^T h_head            dh_head = dA_H W_head
    dP_head   = dh_head^T h              dP_tail = dh_tail^T h
    dh        = dh_head P_head + dh_tail P_tail
with dh_tail the tail layer's feature gradient (the oracle's O6).

The pages leave the activations' precision open.  With hidden_bf16=True the
projected activations h_head and h_tail are rounded to bf16 (fp64 -> fp32 ->
bf16, round to nearest even each time) before the branches use them, which is
the reading for a library whose layer takes bf16 inputs; the backward treats
that rounding as the identity (the gradients reaching h are those of the
unrounded product).  The default keeps everything in double.
"""
from __future__ import annotations

import numpy as np

from . import bce, feature_grad, forward, layout_build, pos_slots, weight_grad


def as_f64(a) -> np.ndarray:
    """float64 array, or uint16 bf16 bit patterns widened exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """float64 -> nearest fp32 -> nearest bf16 (ties to even), as float64.
    A bf16 is the upper 16 bits of an fp32: keep them, adding half an ulp of
    the dropped 16 bits first, less one when the kept part is even."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    keep_odd = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_odd) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def bce_dense(A, Y):
    """dA = sigmoid(A) - Y and the summed BCE max(a, 0) - y a + log(1 + e^-|a|)
    over every entry (the overflow-free form of -y log s - (1 - y) log(1 - s))."""
    A = np.asarray(A, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    e = np.exp(-np.abs(A))
    s = np.where(A >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    loss = float(np.sum(np.maximum(A, 0.0) - Y * A + np.log1p(e)))
    return s - Y, loss


def head_step(h, P_head, W_head, Y_head, hidden_bf16: bool = False):
    """Head branch: forward, BCE and its gradients.  Returns a dict with
    h_head, A, dA, loss, dW_head, dh_head (dh_head is w.r.t. h_head)."""
    h, P_head, W_head = as_f64(h), as_f64(P_head), as_f64(W_head)
    h_head = h @ P_head.T
    if hidden_bf16:
        h_head = round_bf16(h_head)
    A = h_head @ W_head.T
    dA, loss = bce_dense(A, Y_head)
    return dict(h_head=h_head, A=A, dA=dA, loss=loss, dW_head=dA.T @ h_head, dh_head=dA @ W_head)


def projections_backward(h, P_head, P_tail, dh_head, dh_tail):
    """dP_head, dP_tail and the encoder-side dh from both branches."""
    h, P_head, P_tail = as_f64(h), as_f64(P_head), as_f64(P_tail)
    return dict(dP_head=dh_head.T @ h, dP_tail=dh_tail.T @ h, dh=dh_head @ P_head + dh_tail @ P_tail)


def step(h, P_head, P_tail, W_head, Y_head, W_tail, groups, idx, G: int, F: int,
         pos_rowptr, pos_label, hidden_bf16: bool = False):
    """The whole head-tail step.  The tail is the group-shared layer (labels
    `groups`, index rows `idx`, weights W_tail in slot order, positives as
    per-sample label lists) on h_tail = h P_tail^T, computed by the oracle's
    O1-O6 in double.  Returns the loss and every gradient."""
    h64, P_tail64 = as_f64(h), as_f64(P_tail)
    head = head_step(h64, P_head, W_head, Y_head, hidden_bf16)
    h_tail = h64 @ P_tail64.T
    if hidden_bf16:
        h_tail = round_bf16(h_tail)
    H = h_tail.shape[1]
    L = len(groups)
    st, sol, _, ids = layout_build(groups, idx, L, G, F, H)
    if st != 0:
        raise ValueError(f"oracle layout rejected the tail ({st})")
    st, srp, ssl = pos_slots(pos_rowptr, pos_label, L, sol)
    if st != 0:
        raise ValueError(f"oracle positives rejected the tail ({st})")
    Wt = as_f64(W_tail)
    Z = forward(h_tail, Wt, ids, G)
    dZ, tail_loss = bce(Z, srp, ssl)
    dh_tail = feature_grad(Wt, dZ, ids, G, H)
    proj = projections_backward(h64, P_head, P_tail64, head["dh_head"], dh_tail)
    return dict(loss=head["loss"] + tail_loss, head_loss=head["loss"], tail_loss=tail_loss,
                A=head["A"], Z=Z, dA=head["dA"], dZ=dZ, dW_head=head["dW_head"], dW_tail=weight_grad(h_tail, dZ, ids, G, F),
                dh_head=head["dh_head"], dh_tail=dh_tail, h_head=head["h_head"], h_tail=h_tail,
                idx_sorted=ids, **proj)
