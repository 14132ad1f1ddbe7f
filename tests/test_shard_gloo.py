"""Multi-GPU path on CPU: two gloo ranks each run the oracle on their label
shard and all-reduce dh and the loss; the sums must equal the unsharded step,
and each shard's dW rows must equal the full dW rows of its slots."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from extreme_label_sparse_gb300.shard import group_range, shard_problem
from workloads import Workload, generate


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = Workload("shard", B=6, H=40, L=16 * 9, G=16, F=8, pos=7, pos_dist="uniform",
                 zipf_s=0.0, idx_mode="uniform")
    p = generate(w)
    sh = shard_problem(p.groups, p.idx, p.W, p.pos_rowptr, p.pos_label, w.G, world, rank)
    Ls = (sh.k1 - sh.k0) * w.G
    st, sol, los, ids = oracle.layout_build(sh.groups, sh.idx, Ls, w.G, w.F, w.H)
    assert st == 0
    st, srp, ssl = oracle.pos_slots(sh.pos_rowptr, sh.pos_label, Ls, sol)
    assert st == 0
    Z = oracle.forward(p.h, sh.W, ids, w.G)
    dZ, loss = oracle.bce(Z, srp, ssl)
    dW = oracle.weight_grad(p.h, dZ, ids, w.G, w.F)
    dh = torch.from_numpy(oracle.feature_grad(sh.W, dZ, ids, w.G, w.H))
    lt = torch.tensor([loss], dtype=torch.float64)
    dist.all_reduce(dh)
    dist.all_reduce(lt)
    q.put((rank, sh.k0, sh.k1, dW, dh.numpy(), float(lt.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_group_range_partitions():
    for K in (1, 7, 90625):
        for world in (1, 2, 3, 8):
            spans = [group_range(K, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == K
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


def test_two_rank_gloo_allreduce_matches_full(oracle_mod):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    w = Workload("shard", B=6, H=40, L=16 * 9, G=16, F=8, pos=7, pos_dist="uniform",
                 zipf_s=0.0, idx_mode="uniform")
    full = oracle_mod.step(generate(w))
    for rank, k0, k1, dW, dh, loss in res:
        assert np.allclose(dh, full["dh"], rtol=1e-12, atol=1e-12)
        assert loss == pytest.approx(full["loss"], rel=1e-12)
        assert np.allclose(dW, full["dW"][k0 * w.G:k1 * w.G], rtol=1e-12, atol=1e-12)
