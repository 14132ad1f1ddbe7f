"""The label-shard split of the multi-GPU path, run through the library on one
GPU: each shard of one problem (`shard.shard_problem`: a contiguous group
range, its labels, W rows, fan-in sets and positives) is its own layout and
its own `sg_step` call, launched one after another.  Summed over the shards,
dh and the loss must equal the unsharded step, and each shard's dW must equal
the rows of its slots in the full dW (the oracle's step on the whole problem).
This is the reduction the multi-GPU path performs with one all-reduce of dh
and one of the loss (HASTE, key design "gather-once + dense MMA kernel": the
feature gradient is a sum over groups)."""
import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from extreme_label_sparse_gb300.shard import shard_problem
from workloads import Workload, generate

from gpu_common import LOSS_RTOL, assert_close, dev_bf16, dev_i32, host_bf16_to_f64

pytestmark = pytest.mark.gpu

# group counts that the shard counts do not all divide (unequal shards);
# tensor-core shapes
# (B = 128, G = 32; B = 256, G = 16; B = 64, G = 32) and one the CUDA
# cores take (F = 24)
SHAPES = {
    "like3m": Workload("shard_like3m", B=128, H=768, L=32 * 301, G=32, F=128, pos=36,
                       pos_dist="zipf", zipf_s=1.1, idx_mode="uniform"),
    "g16_b256": Workload("shard_g16_b256", B=256, H=768, L=16 * 257, G=16, F=128, pos=5,
                         pos_dist="zipf", zipf_s=1.1, idx_mode="clustered"),
    # B <= 64: paired groups where a shard's count is even, single otherwise
    "pairs_b64": Workload("shard_pairs_b64", B=64, H=768, L=32 * 302, G=32, F=64, pos=10,
                          pos_dist="zipf", zipf_s=1.2, idx_mode="uniform"),
    "simt_f24": Workload("shard_simt_f24", B=40, H=200, L=8 * 45, G=8, F=24, pos=4,
                         pos_dist="uniform", zipf_s=0.0, idx_mode="uniform"),
}


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_label_shards_sum_to_full_step(shape, world, oracle_mod):
    w = SHAPES[shape]
    p = generate(w)
    ref = oracle_mod.step(p)
    h = dev_bf16(p.h)
    dh_sum = np.zeros((w.B, w.H), dtype=np.float64)
    loss_sum = 0.0
    covered = 0
    for rank in range(world):
        s = shard_problem(p.groups, p.idx, p.W, p.pos_rowptr, p.pos_label, w.G, world, rank)
        Ls = (s.k1 - s.k0) * w.G
        nnz = int(s.pos_rowptr[-1])
        lay = sg.sg_layout_build(dev_i32(s.groups), Ls, w.G, dev_i32(s.idx.reshape(-1)),
                                 w.F, w.H, w.B, max(nnz, 1))
        try:
            dW = torch.empty((Ls, w.F), dtype=torch.int16, device="cuda")
            dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
            loss = torch.zeros(1, dtype=torch.float64, device="cuda")
            labels = s.pos_label if nnz else np.zeros(1, np.int32)
            sg.sg_step(lay, h, dev_bf16(s.W), dev_i32(s.pos_rowptr), dev_i32(labels), nnz,
                       dW, dh, loss)
            assert sg.sg_layout_status(lay) == 0
            # the shard's slots are the full layout's slots k0*G .. k1*G - 1
            assert_close(host_bf16_to_f64(dW), ref["dW"][s.k0 * w.G:s.k1 * w.G],
                         what=f"dW of shard {rank}")
            dh_sum += dh.cpu().numpy()
            loss_sum += float(loss.item())
            covered += Ls
        finally:
            lay.close()
    assert covered == w.L
    assert_close(dh_sum, ref["dh"], what="summed dh")
    assert loss_sum == pytest.approx(ref["loss"], rel=LOSS_RTOL)
