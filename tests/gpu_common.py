"""Shared helpers of the GPU tests: move a workloads.Problem to the device,
run the library, bring results back as numpy, compare with the oracle."""
import numpy as np
import torch

import extreme_label_sparse_gb300 as sg

ZTOL = 2e-2     # max |gpu - ref| <= ZTOL * (1 + |ref|)  for Z, dZ, dW, dh
LOSS_RTOL = 1e-3


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda()


def host_bf16_to_f64(t):
    u = t.detach().cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def assert_close(gpu, ref, tol=ZTOL, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref) - tol * (1.0 + np.abs(ref))
    worst = int(np.argmax(err)) if err.size else 0
    assert err.size == 0 or err.flat[worst] <= 0, (
        f"{what}: max violation at {np.unravel_index(worst, err.shape)}: "
        f"gpu={gpu.flat[worst]!r} ref={ref.flat[worst]!r}")


def build_layout(p, max_B=None, max_nnz=None, engine=sg.SG_ENGINE_AUTO):
    w = p.w
    lay = sg.sg_layout_build(dev_i32(p.groups), w.L, w.G, dev_i32(p.idx.reshape(-1)),
                             w.F, w.H, max_B or p.h.shape[0],
                             max(max_nnz if max_nnz is not None else p.nnz, 1))
    sg.sg_layout_set_engine(lay, engine)
    return lay


def dev_problem(p):
    return dict(h=dev_bf16(p.h), W=dev_bf16(p.W), rowptr=dev_i32(p.pos_rowptr),
                labels=dev_i32(p.pos_label if p.nnz else np.zeros(1, np.int32)))
