"""Guard bands around every output buffer: each entry point writes exactly the
elements its header gives it and nothing before or after them.

Every output is carved out of a larger device allocation whose bands on both
sides (4 KB of a sentinel byte pattern) are compared with their initial value
after the call, on ragged shapes (sample counts that are not multiples of the
tiles, a group count that is not a multiple of the cluster) and on each
engine.  A kernel that stored past the end of a tile, or wrote the padding
rows of a sample tile into the caller's buffer, changes a band."""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import Workload, draw_bf16_matrix, generate

from gpu_common import build_layout, dev_bf16, dev_i32, dev_problem

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
SENTINEL = 0x5A


class Guarded:
    """A contiguous tensor of `shape` inside a buffer with sentinel bands."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        esz = torch.empty(0, dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + n * esz,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n * esz].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        head = self.raw[:GUARD].cpu().numpy()
        tail = self.raw[-GUARD:].cpu().numpy()
        return bool(np.all(head == SENTINEL) and np.all(tail == SENTINEL))


SHAPES = [
    # name, B, H, L, G, F
    ("tc_ragged", 37, 320, 16 * 61, 16, 128),
    ("fused_b100", 100, 768, 32 * 301, 32, 128),
    ("b256_g64", 256, 768, 64 * 21, 64, 128),
    ("b200_g64_f64", 200, 640, 64 * 27, 64, 64),
    ("b256_g256", 256, 512, 256 * 5, 256, 128),
    ("one_kernel_f48", 70, 200, 32 * 45, 32, 48),
    ("g1", 45, 256, 333, 1, 64),
    ("pair_b40", 40, 256, 16 * 60, 16, 128),
    ("g5", 9, 64, 5 * 41, 5, 24),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("engine", [sg.SG_ENGINE_AUTO, sg.SG_ENGINE_SIMT], ids=["auto", "simt"])
def test_step_and_stages_stay_inside_their_outputs(shape, engine):
    sg.build()
    name, B, H, L, G, F = shape
    w = Workload(name, B=B, H=H, L=L, G=G, F=F, pos=3, pos_dist="zipf", zipf_s=1.1, idx_mode="uniform")
    p = generate(w)
    lay = build_layout(p, engine=engine)
    try:
        d = dev_problem(p)
        dW = Guarded((L, F), torch.int16)
        dh = Guarded((B, H), torch.float32)
        loss = Guarded((1,), torch.float64)
        sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW.t, dh.t, loss.t)
        assert dW.intact() and dh.intact() and loss.intact()
        Z = Guarded((B, L), torch.int16)
        sg.sg_fwd(lay, d["h"], d["W"], Z.t)
        assert Z.intact()
        dZ = Guarded((B, L), torch.int16)
        loss2 = Guarded((1,), torch.float64)
        sg.sg_fwd_bce(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dZ.t, loss2.t)
        assert dZ.intact() and loss2.intact()
        dW2 = Guarded((L, F), torch.int16)
        dh2 = Guarded((B, H), torch.float32)
        sg.sg_bwd(lay, dZ.t, d["h"], d["W"], dW2.t, dh2.t)
        assert dW2.intact() and dh2.intact()
        assert sg.sg_layout_status(lay) == 0
    finally:
        lay.close()


def test_headtail_rewire_and_grouping_stay_inside_their_outputs():
    sg.build()
    B, E, Dh, Lh, Gh = 37, 136, 32, 96, 32
    tw = Workload("g_tail", B=B, H=128, L=16 * 91, G=16, F=32, pos=3, pos_dist="uniform", zipf_s=1.1,
                  idx_mode="uniform")
    tp = generate(tw)
    h = dev_bf16(draw_bf16_matrix(1, B, E, 1.0))
    P_head = dev_bf16(draw_bf16_matrix(2, Dh, E, 0.1))
    P_tail = dev_bf16(draw_bf16_matrix(3, tw.H, E, 0.1))
    hgroups = (np.arange(Lh) // Gh).astype(np.int32)
    hidx = np.tile(np.arange(Dh, dtype=np.int32), (Lh // Gh, 1))
    head = sg.sg_layout_build(dev_i32(hgroups), Lh, Gh, dev_i32(hidx.reshape(-1)), Dh, Dh, B, 1)
    tail = build_layout(tp)
    try:
        outs = dict(dW_head=Guarded((Lh, Dh), torch.int16), dW_tail=Guarded((tw.L, tw.F), torch.int16),
                    dP_head=Guarded((Dh, E), torch.float32), dP_tail=Guarded((tw.H, E), torch.float32),
                    dh=Guarded((B, E), torch.float32), loss=Guarded((1,), torch.float64))
        hrp = np.zeros(B + 1, np.int32)
        sg.sg_headtail_step(head, tail, h, P_head, P_tail, dev_bf16(draw_bf16_matrix(4, Lh, Dh, 0.1)), dev_i32(hrp),
                            dev_i32(np.zeros(1, np.int32)), 0, dev_bf16(tp.W), dev_i32(tp.pos_rowptr),
                            dev_i32(tp.pos_label), tp.nnz, **{k: v.t for k, v in outs.items()})
        for k, v in outs.items():
            assert v.intact(), k
        idx_out = Guarded((tw.K, tw.F), torch.int32)
        W_out = Guarded((tw.L, tw.F), torch.int16)
        d = dev_problem(tp)
        sg.sg_rewire(tail, d["h"], dev_bf16(draw_bf16_matrix(5, B, tw.L, 0.5)), d["W"], 4, idx_out.t, W_out.t)
        assert idx_out.intact() and W_out.intact()
    finally:
        head.close()
        tail.close()
    L, D, G, C = 1024, 32, 16, 8
    g = sg.sg_grouping_create(L, D, G, C)
    try:
        rng = np.random.default_rng(0)
        N = 200
        rowptr = np.arange(0, 3 * N + 1, 3, dtype=np.int32)
        labels = rng.integers(0, 700, 3 * N).astype(np.int32)
        sg.sg_grouping_embed(g, dev_bf16(draw_bf16_matrix(6, N, D, 1.0)), dev_i32(rowptr), dev_i32(labels),
                             len(labels))
        act = np.unique(labels)
        sg.sg_grouping_kmeans_init(g, dev_i32(act[:C]))
        assign = Guarded((128,), torch.int32)
        sg.sg_grouping_kmeans_batch(g, dev_i32(act[:128]), assign.t)
        groups = Guarded((L,), torch.int32)
        clus = Guarded((L,), torch.int32)
        sg.sg_grouping_groups(g, groups.t, clus.t)
        assert assign.intact() and groups.intact() and clus.intact()
        E = Guarded((L, D), torch.int16)
        has = Guarded((L,), torch.uint8)
        cent = Guarded((C, D), torch.float32)
        cnt = Guarded((C,), torch.int64)
        sg.sg_grouping_export(g, E=E.t, has=has.t, centroids=cent.t, counts=cnt.t)
        assert E.intact() and has.intact() and cent.intact() and cnt.intact()
        assert sg.sg_grouping_status(g) == 0
    finally:
        g.close()
