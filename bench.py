#!/usr/bin/env python
"""Benchmark of one training step of the group-shared fixed fan-in sparse
output layer (forward Z_k = H_k W_k^T, fused BCE gradient, dW_k and the
Split-K feature gradient dh) on synthetic data shaped like the Amazon-3M tail.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` = label-logits per second (B*L per s,
summed over ranks) with inputs resident in HBM, timed without per-kernel
instrumentation; `e2e` = the same through the public API from pinned host
buffers (h and positives copied in, loss copied out every step); `roofline` =
the dominant kernel's algorithmic bytes / its mean launch time (CUDA events
around each launch, in a separate loop) against the measured HBM peak;
`roofline_step` = the whole step's algorithmic bytes and FLOPs over the step
time against both peaks; `workloads` = step time, per-kernel split and step
roofline of the other label-space workloads and of the group-size sweep
(G = 1, 16, 32, 64 with uniform and clustered index sets);
`headtail` = the head-tail split's whole step (projections, dense head,
sparse tail) on the same tail with a 3% dense head; `grouping` = the semantic
grouping of the same L labels (embeddings, mini-batch k-means, greedy groups);
`rewire` = one re-selection of every group's fan-in set on the same layout;
`cpu_baseline` = the CPU oracle on a bounded sample of the same workload.
`--impl reference` times that oracle alone (there is no other implementation
of the method to run).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from workloads import CONFIGS, generate  # noqa: E402

METRIC = "fwd+bwd label-logits/s (B·L per s) and % of BF16/HBM roofline on 1 GB300"
UNIT = "label-logits/s"
DEFAULT_WORKLOAD = "amazon3m_tail"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ------------------------------------------------------------------ work model
# DRAM bytes per group measured by ncu (dram__bytes_read.sum +
# dram__bytes_write.sum of one launch / its groups) on the 3M shape at
# L = 524,288 (16,384 groups), for the kernels as they stand.  Scaled to a
# launch by the groups it processes; None for other shapes.
MEASURED_TRAFFIC_PER_GROUP = {
    ("amazon3m_tail", "fwd"): (138.859e6 + 210.617e6) / 16384,
    ("amazon3m_tail", "dh"): (273.069e6 + 3.250e6) / 16384,
}


SGD_LR, SGD_MU = 1e-3, 0.9  # momentum SGD of the --sgd step (values do not change the work)


def algorithmic(w, B, kind, fused_dW=False, sgd=False):
    """(bytes, flops) one launch of `kind` must move / do at minimum inside the
    training step.  bf16 W, dW, h; uint16 idx; fp32 dh; positives as int32.
    dZ is internal to the step (no call outputs it), so it is not counted;
    `fused_dW`: the forward launch also computes and writes dW."""
    L, K, F, H = w.L, w.K, w.F, w.H
    W_b = L * F * 2
    idx_b = K * F * 2
    h_b = B * H * 2
    dh_b = B * H * 4
    nnz_b = B * w.pos * 4 * 2
    flops_gemm = 2 * B * L * F
    if kind == "step":
        return W_b + W_b + idx_b + h_b + dh_b + nnz_b, 3 * flops_gemm
    if kind == "fwd":      # forward + fused BCE (+ dW when fused)
        if fused_dW and sgd:  # + the momentum-SGD update: W_out written, fp32 momentum read and written
            return W_b + W_b + 2 * L * F * 4 + idx_b + h_b + nnz_b, 2 * flops_gemm
        if fused_dW:
            return W_b + W_b + idx_b + h_b + nnz_b, 2 * flops_gemm
        return W_b + idx_b + h_b + nnz_b, flops_gemm
    if kind == "dW":
        return W_b + idx_b + h_b, flops_gemm
    if kind == "dh":
        return W_b + idx_b + dh_b, flops_gemm
    return 0, 0


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            for line in Path(self.path).read_text().splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
            os.unlink(self.path)
        except Exception:
            return None
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ oracle
def oracle_sample_step(p, ids, sol, n_groups):
    """The CPU oracle's step (positives, forward, BCE, dW, dh) on the slots of
    the first n_groups groups and every sample; returns seconds taken."""
    import oracle
    w = p.w
    Ls = n_groups * w.G
    t0 = time.perf_counter()
    st, srp, ssl = oracle.pos_slots(p.pos_rowptr, p.pos_label, w.L, sol)
    keep = ssl < Ls
    srp2 = np.zeros_like(srp)
    for b in range(len(srp) - 1):
        srp2[b + 1] = srp2[b] + int(keep[srp[b]:srp[b + 1]].sum())
    ssl2 = ssl[keep]
    Z = oracle.forward(p.h, p.W[:Ls], ids[:n_groups], w.G)
    dZ, loss = oracle.bce(Z, srp2, ssl2)
    oracle.weight_grad(p.h, dZ, ids[:n_groups], w.G, w.F)
    oracle.feature_grad(p.W[:Ls], dZ, ids[:n_groups], w.G, w.H)
    return time.perf_counter() - t0


def oracle_baseline(p, target_s: float):
    """Time the oracle on a bounded sample sized to about target_s seconds."""
    import oracle
    w = p.w
    st, sol, los, ids = oracle.layout_build(p.groups, p.idx, w.L, w.G, w.F, w.H)
    if st != 0:
        raise RuntimeError("oracle rejected the layout")
    n = max(1, min(w.K, 4096 // max(1, w.G)))
    t = oracle_sample_step(p, ids, sol, n)
    n2 = int(min(w.K, max(1, n * target_s / max(t, 1e-3))))
    if n2 > n:
        n = n2
        t = oracle_sample_step(p, ids, sol, n)
    return dict(value=p.h.shape[0] * n * w.G / t, seconds=t, n_groups=n,
                cores=oracle.num_threads(), ids=ids, sol=sol)


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = CONFIGS[args.workload]
    p = generate(w)
    calib = oracle_baseline(p, args.ref_step_seconds)
    n = calib["n_groups"]
    for _ in range(args.warmup):
        oracle_sample_step(p, calib["ids"], calib["sol"], n)
    times = [oracle_sample_step(p, calib["ids"], calib["sol"], n) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = w.B * n * w.G / t
    sample = (f"first {n} of {w.K} groups ({n * w.G} of {w.L} labels), all {w.B} samples; "
              "step = positives + forward + BCE + dW + dh in double")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "G": w.G, "F": w.F, "H": w.H},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": calib["cores"],
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
class Runner:
    """One workload on the device: inputs resident, a layout, and the step
    through the public API (sg_step, or sg_step_sgd)."""

    def __init__(self, sg, torch, dev, p, engine, sgd=False, world=1, dist=None):
        import numpy as _np
        self.sg, self.torch, self.dev, self.p, self.sgd = sg, torch, dev, p, sgd
        self.world, self.dist = world, dist
        w = p.w

        def i32(a):
            return torch.from_numpy(_np.ascontiguousarray(a, dtype=_np.int32)).to(dev)

        def bf(a):
            return torch.from_numpy(_np.ascontiguousarray(a).view(_np.int16)).to(dev)

        self.h, self.W = bf(p.h), bf(p.W)
        self.rowptr, self.labels = i32(p.pos_rowptr), i32(p.pos_label if p.nnz else _np.zeros(1))
        self.lay = sg.sg_layout_build(i32(p.groups), w.L, w.G, i32(p.idx.reshape(-1)), w.F, w.H,
                                      w.B, max(p.nnz, 1))
        sg.sg_layout_set_engine(self.lay, engine)
        self.dW = torch.empty((w.L, w.F), dtype=torch.int16, device=dev)
        self.dh = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
        self.loss = torch.zeros(1, dtype=torch.float64, device=dev)
        # --sgd: the step with the output layer's momentum-SGD update, weights
        # double-buffered as a training loop keeps them (dW is the second buffer)
        self.mom = torch.zeros((w.L, w.F), dtype=torch.float32, device=dev) if sgd else None
        self.bufs = [self.W, self.dW]

    def step(self, h=None, rp=None, lb=None):
        sg, p = self.sg, self.p
        h = self.h if h is None else h
        rp = self.rowptr if rp is None else rp
        lb = self.labels if lb is None else lb
        if self.sgd:
            sg.sg_step_sgd(self.lay, h, self.bufs[0], rp, lb, p.nnz, SGD_LR, SGD_MU, self.mom,
                           self.bufs[1], self.dh, self.loss)
            self.bufs.reverse()
        else:
            sg.sg_step(self.lay, h, self.W, rp, lb, p.nnz, self.dW, self.dh, self.loss)
        if self.world > 1:
            self.dist.all_reduce(self.dh)
            self.dist.all_reduce(self.loss)

    def timed(self, steps, stream, barrier=lambda: None):
        """ms per step over `steps` steps, CUDA events on `stream`, no
        per-kernel instrumentation inside the timed loop."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            self.step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return e0.elapsed_time(e1) / steps

    def per_kind(self, steps):
        """{kind: (total ms, launches)} over `steps` steps, every kernel
        bracketed by CUDA events on the stream it is launched on."""
        self.sg.sg_timing_start(self.lay, 64 * steps)
        for _ in range(steps):
            self.step()
        self.torch.cuda.synchronize()
        return self.sg.sg_timing_stop(self.lay)

    def status(self):
        return self.sg.sg_layout_status(self.lay)

    def close(self):
        self.lay.close()


def step_roofline(w, ms, hbm, tflops):
    """Whole-step work against the binding roofline: the step's algorithmic
    bytes (W read, dW written, idx, h, dh, positives) and FLOPs (6 B L F)
    over the measured step time."""
    bytes_, flops = algorithmic(w, w.B, "step")
    s = ms * 1e-3
    gbs, tfs = bytes_ / s / 1e9, flops / s / 1e12
    t_hbm, t_tc = bytes_ / (hbm * 1e9), flops / (tflops * 1e12)
    return {"bound": "hbm" if t_hbm >= t_tc else "tensor", "bytes": bytes_, "flops": flops,
            "achieved_gbs": gbs, "achieved_tflops": tfs, "frac_hbm": gbs / hbm,
            "frac_tensor": tfs / tflops, "frac": max(t_hbm, t_tc) / s,
            "t_bound_us": max(t_hbm, t_tc) * 1e6}


def measure_other(sg, torch, dev, p, engine, steps, warmup, stream, hbm, tflops):
    """Step time, per-kind split and the step roofline of one more workload."""
    r = Runner(sg, torch, dev, p, engine)
    try:
        for _ in range(warmup):
            r.step()
        torch.cuda.synchronize()
        ms = r.timed(steps, stream)
        kinds = r.per_kind(steps)
        st = r.status()
    finally:
        r.close()
    w = p.w
    out = {"ms_per_step": ms, "label_logits_per_s": w.B * w.L / (ms * 1e-3),
           "per_kind_ms_per_step": {k: v[0] / steps for k, v in kinds.items() if v[1]},
           "launches_per_step": {k: v[1] / steps for k, v in kinds.items() if v[1]},
           "roofline_step": step_roofline(w, ms, hbm, tflops), "status": st,
           "config": {"B": w.B, "L": w.L, "G": w.G, "F": w.F, "H": w.H, "idx": w.idx_mode}}
    return out


HEAD_SHARE_LABELS = 90_112   # ~3% of a 3M label space in the dense head (groups of 32)
HEAD_DIM, HEAD_G = 128, 32    # head projection width Dh; head layout groups of 32 labels over [0, Dh)


def measure_headtail(sg, torch, dev, p, steps, warmup, stream, hbm, tflops):
    """The head-tail split's whole step (sg_headtail_step) with the tail of
    workload p (h_tail = h P_tail^T, E = H) and a dense head of
    HEAD_SHARE_LABELS labels over a Dh = HEAD_DIM projection; 5 uniform head
    positives per sample."""
    from workloads import Workload, draw_bf16_matrix
    w = p.w
    B, E, H, Dh = w.B, w.H, w.H, HEAD_DIM
    hw = Workload("head", B=B, H=Dh, L=HEAD_SHARE_LABELS, G=HEAD_G, F=Dh, pos=5, pos_dist="uniform",
                  zipf_s=0.0, idx_mode="uniform", seed=7)
    hp = generate(hw)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    h = bf(draw_bf16_matrix(41, B, E, 1.0))
    P_head = bf(draw_bf16_matrix(42, Dh, E, 1.0 / np.sqrt(E)))
    P_tail = bf(draw_bf16_matrix(43, H, E, 1.0 / np.sqrt(E)))
    head = sg.sg_layout_build(i32(hp.groups), hw.L, hw.G, i32(hp.idx.reshape(-1)), hw.F, hw.H, B, hp.nnz)
    tail = sg.sg_layout_build(i32(p.groups), w.L, w.G, i32(p.idx.reshape(-1)), w.F, w.H, B, max(p.nnz, 1))
    try:
        args = dict(W_head=bf(hp.W), head_rowptr=i32(hp.pos_rowptr), head_label=i32(hp.pos_label),
                    head_nnz=hp.nnz, W_tail=bf(p.W), tail_rowptr=i32(p.pos_rowptr),
                    tail_label=i32(p.pos_label), tail_nnz=p.nnz,
                    dW_head=torch.empty((hw.L, hw.F), dtype=torch.int16, device=dev),
                    dW_tail=torch.empty((w.L, w.F), dtype=torch.int16, device=dev),
                    dP_head=torch.empty((Dh, E), dtype=torch.float32, device=dev),
                    dP_tail=torch.empty((H, E), dtype=torch.float32, device=dev),
                    dh=torch.empty((B, E), dtype=torch.float32, device=dev),
                    loss=torch.zeros(1, dtype=torch.float64, device=dev))

        def step():
            sg.sg_headtail_step(head, tail, h, P_head, P_tail, **args)

        for _ in range(max(warmup, 3)):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        st = sg.sg_layout_status(head) | sg.sg_layout_status(tail)
    finally:
        head.close()
        tail.close()
    tb, tf = algorithmic(w, B, "step")
    hb, hf = algorithmic(hw, B, "step")
    proj_b = (Dh + H) * E * (2 + 4) + B * E * (2 + 4)  # P read, dP written (fp32), h read, dh written
    proj_f = 3 * 2 * B * E * (Dh + H)                  # forward, dP, dh
    bytes_, flops = tb + hb + proj_b, tf + hf + proj_f
    s = ms * 1e-3
    return {"ms_per_step": ms, "status": st,
            "config": {"B": B, "E": E, "head": {"L": hw.L, "G": hw.G, "Dh": Dh, "pos": hw.pos},
                       "tail": {"L": w.L, "G": w.G, "F": w.F, "H": H}},
            "roofline_step": {"bytes": bytes_, "flops": flops, "achieved_gbs": bytes_ / s / 1e9,
                              "frac_hbm": bytes_ / s / 1e9 / hbm,
                              "achieved_tflops": flops / s / 1e12,
                              "frac_tensor": flops / s / 1e12 / tflops}}


GROUPING_SAMPLES, GROUPING_BETA, GROUPING_BATCHES, GROUPING_BATCH = 8192, 4, 10, 65536


def measure_grouping(sg, torch, dev, w, tflops):
    """Semantic grouping of the workload's L labels from GROUPING_SAMPLES
    samples (h ~ N(0, 1) bf16 of H features, w.pos positives each, drawn like
    the workload's): embeddings, k-means into C = (labels with an embedding)
    / (beta G) clusters over GROUPING_BATCHES batches, final assignment and
    greedy groups.  Host-timed around each call (they synchronise)."""
    from workloads import draw_bf16_matrix, draw_positives
    N, D, L, G = GROUPING_SAMPLES, w.H, w.L, w.G
    rowptr, labels = draw_positives(21, N, L, w.pos, w.pos_dist, w.zipf_s)
    hbits = draw_bf16_matrix(22, N, D, 1.0)
    active = np.unique(labels)
    C = max(1, int(round(len(active) / (GROUPING_BETA * G))))
    rng = np.random.default_rng(23)
    init = rng.choice(active, C, replace=False).astype(np.int32)
    M = min(GROUPING_BATCH, len(active))
    batches = [rng.choice(active, M, replace=False).astype(np.int32) for _ in range(GROUPING_BATCHES)]

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    h_d = torch.from_numpy(hbits.view(np.int16)).to(dev)
    rp_d, lb_d, init_d = i32(rowptr), i32(labels), i32(init)
    b_d = [i32(b) for b in batches]
    groups = torch.empty(L, dtype=torch.int32, device=dev)
    g = sg.sg_grouping_create(L, D, G, C, dev)
    try:
        def run():
            t = [time.perf_counter()]
            n = sg.sg_grouping_embed(g, h_d, rp_d, lb_d, len(labels))
            torch.cuda.synchronize()
            t.append(time.perf_counter())
            sg.sg_grouping_kmeans_init(g, init_d)
            for b in b_d:
                sg.sg_grouping_kmeans_batch(g, b)
            torch.cuda.synchronize()
            t.append(time.perf_counter())
            sg.sg_grouping_groups(g, groups)
            torch.cuda.synchronize()
            t.append(time.perf_counter())
            return n, [1e3 * (b - a) for a, b in zip(t, t[1:])]

        run()  # warm-up (allocation of the compact arrays, module load)
        n, ms = run()
        st = sg.sg_grouping_status(g)
    finally:
        g.close()
    sizes = np.bincount(groups.cpu().numpy(), minlength=L // G)
    gemm_flops = 2.0 * D * C * (GROUPING_BATCHES * M + n)  # batch assignments + the final one
    return {"config": {"L": L, "G": G, "D": D, "samples": N, "positives_per_sample": w.pos, "beta": GROUPING_BETA,
                       "clusters": C, "labels_with_embedding": n, "batches": GROUPING_BATCHES, "batch": M},
            "ms": {"embed": ms[0], "kmeans": ms[1], "groups": ms[2], "total": sum(ms)},
            "argmax_gemm_flops": gemm_flops, "status": st,
            "groups_all_of_size_G": bool(np.all(sizes == G))}


def measure_rewire(sg, torch, dev, p, steps, stream, hbm, tflops):
    """One rewiring phase (sg_rewire, n_drop = F / 8) on the workload's
    layout, with dZ = sigmoid(Z) - Y of its batch (sg_fwd_bce).  CUDA events
    around `steps` calls."""
    w = p.w
    r = Runner(sg, torch, dev, p, sg.SG_ENGINE_AUTO)
    try:
        dZ = torch.empty((w.B, w.L), dtype=torch.int16, device=dev)
        loss = torch.zeros(1, dtype=torch.float64, device=dev)
        sg.sg_fwd_bce(r.lay, r.h, r.W, r.rowptr, r.labels, p.nnz, dZ, loss)
        idx_out = torch.empty((w.K, w.F), dtype=torch.int32, device=dev)
        W_out = torch.empty((w.L, w.F), dtype=torch.int16, device=dev)
        nd = w.F // 8
        for _ in range(2):
            sg.sg_rewire(r.lay, r.h, dZ, r.W, nd, idx_out, W_out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            sg.sg_rewire(r.lay, r.h, dZ, r.W, nd, idx_out, W_out)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        st = r.status()
    finally:
        r.close()
    # dZ, W read, W_out written, idx read and written, the K x H scores written and read
    bytes_ = w.B * w.L * 2 + 2 * w.L * w.F * 2 + w.K * w.F * (2 + 4) + 2 * w.K * w.H * 4 + w.B * w.H * 2
    flops = 2.0 * w.L * w.H * w.B  # the grow-score GEMM dZ^T h
    s = ms * 1e-3
    return {"ms": ms, "n_drop": nd, "status": st, "bytes": bytes_, "flops": flops,
            "achieved_gbs": bytes_ / s / 1e9, "frac_hbm": bytes_ / s / 1e9 / hbm,
            "achieved_tflops": flops / s / 1e12, "frac_tensor": flops / s / 1e12 / tflops}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import extreme_label_sparse_gb300 as sg

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    sg.build()
    sg.load()
    w = CONFIGS[args.workload]
    if args.labels:
        w = w.with_(L=args.labels, name=f"{w.name}_L{args.labels}")
    engine = {"auto": sg.SG_ENGINE_AUTO, "simt": sg.SG_ENGINE_SIMT, "tc": sg.SG_ENGINE_TC,
              "fused": sg.SG_ENGINE_FUSED}[args.engine]
    hbm, tflops, peak_src = _peaks()

    # the other workloads (label-space shapes and the group-size sweep) are
    # drawn on host threads while the headline workload is measured
    others = []
    if rank == 0 and world == 1 and not args.labels:
        if not args.no_others:
            others += [n for n in ("amazon670k_tail", "lf8p6m_tail") if n != w.name]
        if not args.no_sweep:
            others += [f"sweep_g{g}_{m}" for g in (1, 16, 32, 64) for m in ("uniform", "clustered")]
    pool = None
    futures = []
    if others:
        from concurrent.futures import ThreadPoolExecutor
        pool = ThreadPoolExecutor(max_workers=3)
        futures = [(n, pool.submit(generate, CONFIGS[n])) for n in others]

    # weak scaling: every rank owns one shard of w.L labels (its own groups,
    # W rows and positives; h is shared); dh and the loss are summed over the
    # shards with one all-reduce each
    p = generate(w, shard=rank)
    r = Runner(sg, torch, dev, p, engine, sgd=args.sgd, world=world, dist=dist)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        r.step()
    torch.cuda.synchronize()
    if r.status() != 0:
        raise RuntimeError("device status set during warm-up")

    # ---- device-timed region: inputs resident in HBM, no instrumentation
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = r.timed(args.steps, stream, barrier)
    clk = clocks.stop()
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = world * w.B * w.L / (ms * 1e-3)
    # ---- per-kernel split (a separate loop: every kernel between CUDA events)
    kinds = r.per_kind(args.steps)

    # ---- end to end through the public API: host buffers, copies timed
    h_host = torch.from_numpy(np.ascontiguousarray(p.h).view(np.int16)).pin_memory()
    rp_host = torch.from_numpy(p.pos_rowptr.astype(np.int32)).pin_memory()
    lb_host = torch.from_numpy(p.pos_label.astype(np.int32)).pin_memory()
    loss_host = torch.zeros(1, dtype=torch.float64).pin_memory()
    h_d, rp_d, lb_d = torch.empty_like(r.h), torch.empty_like(r.rowptr), torch.empty_like(r.labels)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        h_d.copy_(h_host, non_blocking=True)
        rp_d.copy_(rp_host, non_blocking=True)
        lb_d.copy_(lb_host, non_blocking=True)
        r.step(h_d, rp_d, lb_d)
        loss_host.copy_(r.loss, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1) / args.steps
    if world > 1:
        t = torch.tensor([ms_e2e], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_e2e = float(t.item())
    h2d = h_host.numel() * 2 + rp_host.numel() * 4 + lb_host.numel() * 4
    if r.status() != 0:
        raise RuntimeError("device status set during the timed region")

    # ---- roofline of the dominant kernel (per launch) and of the whole step
    dom = max((k for k in kinds if kinds[k][1] > 0), key=lambda k: kinds[k][0])
    dom_ms, dom_n = kinds[dom]
    fused = kinds.get("dW", (0.0, 0))[1] == 0
    bytes_, flops = algorithmic(w, w.B, dom, fused_dW=fused, sgd=args.sgd)
    per_launch_s = dom_ms * 1e-3 / dom_n
    achieved = bytes_ / per_launch_s / 1e9
    per_group = None if args.sgd else MEASURED_TRAFFIC_PER_GROUP.get((w.name.split("_L")[0], dom))
    traffic = per_group * w.K if per_group is not None and dom_n else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "kernel": dom,
                "scope": "per launch of the dominant kernel",
                "peak_source": peak_src,
                "launch_ms": per_launch_s * 1e3,
                "tensor_tflops": flops / per_launch_s / 1e12 if flops else 0.0,
                "tensor_frac_of_bf16_peak": (flops / per_launch_s / 1e12) / tflops if flops else 0.0,
                "per_kind_ms_per_step": {k: v[0] / args.steps for k, v in kinds.items() if v[1]}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        b = oracle_baseline(p, args.cpu_seconds)
        cpu = {"value": b["value"], "unit": UNIT, "cores": b["cores"], "kind": "oracle",
               "sample": (f"first {b['n_groups']} of {w.K} groups ({b['n_groups'] * w.G} labels), "
                          f"all {w.B} samples; positives + forward + BCE + dW + dh in double, "
                          f"{b['seconds']:.1f} s")}
    launches = sum(v[1] for v in kinds.values())
    r.close()
    del r
    headtail = grouping = rewire = None
    if rank == 0 and world == 1 and not args.sgd and (args.extras or (not args.labels and not args.no_others)):
        headtail = measure_headtail(sg, torch, dev, p, args.other_steps, 2, stream, hbm, tflops)
        grouping = measure_grouping(sg, torch, dev, w, tflops)
        rewire = measure_rewire(sg, torch, dev, p, args.other_steps, stream, hbm, tflops)

    workloads = {}
    for name, fut in futures:
        po = fut.result()
        workloads[name] = measure_other(sg, torch, dev, po, engine, args.other_steps, 2, stream, hbm, tflops)
        del po
    if pool is not None:
        pool.shutdown()

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "G": w.G, "F": w.F, "H": w.H,
                   "nnz": p.nnz, "engine": args.engine,
                   **({"optimizer": f"momentum SGD lr {SGD_LR} mu {SGD_MU} (sg_step_sgd)"} if args.sgd else {}),
                   "l2": f"inputs larger than L2 (W {w.L * w.F * 2 / 1e6:.0f} MB read, dW written each step)",
                   "parallelism": "single GPU" if world == 1 else f"{world} label shards, dh all-reduce"},
        "roofline": roofline,
        "roofline_step": step_roofline(w, ms, hbm, tflops),
        "cpu_baseline": cpu,
        "e2e": {"value": world * w.B * w.L / (ms_e2e * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 8},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if workloads:
        line["workloads"] = workloads
    if headtail is not None:
        line["headtail"] = headtail
    if grouping is not None:
        line["grouping"] = grouping
    if rewire is not None:
        line["rewire"] = rewire
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(CONFIGS))
    ap.add_argument("--engine", choices=["auto", "simt", "tc", "fused"], default="auto",
                    help="fused: the whole step in one cluster kernel wherever it fits")
    ap.add_argument("--labels", type=int, default=0,
                    help="override L (a multiple of G) for small profiling runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sgd", action="store_true",
                    help="time sg_step_sgd (the step plus the momentum-SGD update of W)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the group-size sweep (G = 1, 16, 32, 64; uniform and clustered idx)")
    ap.add_argument("--extras", action="store_true",
                    help="measure the head-tail step, grouping and rewiring also with --labels "
                         "(on the reduced workload; for profiling runs)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the other label-space workloads (670K- and 8.6M-shaped tails)")
    ap.add_argument("--other-steps", type=int, default=5,
                    help="timed steps of each other workload and sweep point")
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
