"""GPU parity: every entry point of the C ABI against the CPU oracle on the
same seeded inputs, element by element (small and ragged sizes), for both
engines where they apply.  Bit-exact for the layout and the positive lists;
max |gpu - ref| <= 2e-2 (1 + |ref|) for Z, dZ, dW, dh; loss within 1e-3."""
import gc

import numpy as np
import pytest
import torch

import extreme_label_sparse_gb300 as sg
from workloads import CONFIGS, Workload, bf16_bits_to_f32, draw_bf16_matrix, generate

from gpu_common import (LOSS_RTOL, ZTOL, assert_close, build_layout, dev_bf16, dev_i32,
                        dev_problem, host_bf16_to_f64)

pytestmark = pytest.mark.gpu

SIMT, TC = sg.SG_ENGINE_SIMT, sg.SG_ENGINE_TC


def _w(name, B, H, L, G, F, pos=3, idx_mode="uniform", dist="uniform", seed=0):
    return Workload(name, B=B, H=H, L=L, G=G, F=F, pos=pos, pos_dist=dist, zipf_s=1.1,
                    idx_mode=idx_mode, seed=seed)


# (workload, engines): shapes spanning several tiles, ragged tails and the
# degenerate cases (B = 1, G = 1, F = H, odd G / F)
CASES = [
    (CONFIGS["tiny"], (SIMT, TC)),
    (_w("g1", B=37, H=96, L=300, G=1, F=24), (SIMT,)),
    (_w("g3_oddF", B=5, H=50, L=99, G=3, F=7), (SIMT,)),
    (_w("b1", B=1, H=64, L=512, G=16, F=16), (SIMT, TC)),
    (_w("g32_b100", B=100, H=200, L=32 * 70, G=32, F=48, dist="zipf"), (SIMT, TC)),
    (_w("g64_b200", B=200, H=768, L=64 * 40, G=64, F=128, pos=8, dist="zipf"), (SIMT, TC)),
    (_w("dense_F_eq_H", B=16, H=32, L=16 * 12, G=16, F=32), (SIMT, TC)),
    (_w("clustered", B=64, H=768, L=16 * 100, G=16, F=128, idx_mode="clustered"), (SIMT, TC)),
    (_w("b256_f256", B=256, H=512, L=32 * 20, G=32, F=256, pos=4), (SIMT, TC)),
    # shapes of the three label-space workloads, fewer groups
    (_w("like3m", B=128, H=768, L=32 * 300, G=32, F=128, pos=36, dist="zipf"), (SIMT, TC)),
    (_w("like670k", B=256, H=768, L=16 * 400, G=16, F=128, pos=5, dist="zipf"), (SIMT, TC)),
    (_w("like8p6m", B=64, H=768, L=32 * 500, G=32, F=64, pos=10, dist="zipf"), (SIMT, TC)),
    # ragged batch, one dh band; G above one 64-wide swizzle row; three bands
    (_w("tc_b37_h320", B=37, H=320, L=16 * 64, G=16, F=128, pos=4), (SIMT, TC)),
    (_w("tc_g128", B=100, H=768, L=128 * 20, G=128, F=128, pos=6, dist="zipf"), (SIMT, TC)),
    (_w("tc_h1000", B=130, H=1000, L=32 * 40, G=32, F=128, pos=6), (SIMT, TC)),
    # B = 256 at G = 64: the fused kernel takes the two sample tiles one
    # after the other (dW accumulated over both), F = 128 and F = 64; F = 256
    # the same way at G = 16 and G = 32 (ragged B), at G = 64 as subgroups of
    # 32; G = 256 as four subgroups of 64
    (_w("g64_b256", B=256, H=768, L=64 * 30, G=64, F=128, pos=5, dist="zipf"), (SIMT, TC)),
    (_w("g64_b200_f64", B=200, H=640, L=64 * 27, G=64, F=64, pos=5, dist="zipf"), (SIMT, TC)),
    (_w("g32_b150_f256", B=150, H=512, L=32 * 25, G=32, F=256, pos=4), (SIMT, TC)),
    (_w("g16_b256_f256", B=256, H=384, L=16 * 41, G=16, F=256, pos=4), (SIMT, TC)),
    (_w("g64_b256_f256", B=256, H=512, L=64 * 9, G=64, F=256, pos=4), (SIMT, TC)),
    (_w("g256_b256", B=256, H=512, L=256 * 5, G=256, F=128, pos=6, dist="zipf"), (SIMT, TC)),
    # the fused kernel on subgroups sharing I_k: G = 128 at B = 256, G = 256
    (_w("g128_b256_sub", B=256, H=512, L=128 * 12, G=128, F=128, pos=6, dist="zipf"), (SIMT, TC)),
    (_w("g256_f64_sub", B=100, H=384, L=256 * 8, G=256, F=64, pos=6, dist="zipf"), (SIMT, TC)),
    # groups of 192 (dh as three subgroups of 64); wide H (eleven dh bands,
    # and three column windows of the CUDA-core dh)
    (_w("tc_g192_f32", B=100, H=256, L=192 * 8, G=192, F=32, pos=5), (SIMT, TC)),
    (_w("tc_h4096", B=64, H=4096, L=32 * 60, G=32, F=64, pos=4), (SIMT, TC)),
    # B <= 64: the fused forward pairs consecutive groups (an even count);
    # with an odd count it runs them one by one
    (_w("pair_g16_b40", B=40, H=320, L=16 * 62, G=16, F=128, pos=4), (SIMT, TC)),
    (_w("like8p6m_oddK", B=64, H=768, L=32 * 301, G=32, F=64, pos=10, dist="zipf"), (SIMT, TC)),
    (_w("simt_h2500_g5", B=40, H=2500, L=5 * 120, G=5, F=40, pos=3), (SIMT,)),
    # per-label fan-in through the dedicated G = 1 kernels: several sample
    # tiles and label chunks, a ragged last tile, F = 64 and 128
    (_w("g1_f128", B=100, H=256, L=700, G=1, F=128, pos=4, dist="zipf"), (SIMT,)),
    (_w("g1_f64_b256", B=256, H=512, L=1000, G=1, F=64, pos=5, dist="zipf"), (SIMT,)),
]


def _run(fn, *args, **kw):
    """Call an entry point; a shape the pinned engine cannot run skips the test."""
    try:
        return fn(*args, **kw)
    except sg.SGError as e:
        if e.status == sg.SG_ERR_UNSUPPORTED:
            pytest.skip(f"engine does not run this shape: {e}")
        raise


def _ids(case):
    return case[0].name


@pytest.fixture(scope="module", autouse=True)
def _built():
    sg.build()
    sg.load()


@pytest.fixture(scope="module", params=CASES, ids=[c[0].name for c in CASES])
def case(request, oracle_mod):
    w, engines = request.param
    p = generate(w)
    ref = oracle_mod.step(p, want_Z=True)
    return w, engines, p, ref


def _engines(case_):
    w, engines, p, ref = case_
    return engines


def _layout(p, engine):
    lay = build_layout(p)
    if engine == TC:
        try:
            sg.sg_layout_set_engine(lay, TC)
        except sg.SGError as e:
            pytest.skip(f"tensor-core engine unavailable: {e}")
    else:
        sg.sg_layout_set_engine(lay, engine)
    return lay


def _status_ok(lay):
    assert sg.sg_layout_status(lay) == 0


@pytest.mark.parametrize("engine", [SIMT, TC], ids=["simt", "tc"])
def test_layout_and_positives_bit_exact(case, engine):
    w, engines, p, ref = case
    if engine not in engines:
        pytest.skip("engine not used for this shape")
    lay = _layout(p, engine)
    sol, los, ids = sg.sg_layout_export(lay)
    assert np.array_equal(sol.cpu().numpy(), ref["slot_of_label"])
    assert np.array_equal(los.cpu().numpy(), ref["label_of_slot"])
    assert np.array_equal(ids.cpu().numpy().view(np.uint16), ref["idx_sorted"])
    d = dev_problem(p)
    orp, osl, ogp, oge = sg.sg_pos_export(lay, w.B, d["rowptr"], d["labels"], p.nnz)
    orp = orp.cpu().numpy()
    assert np.array_equal(orp, ref["srowptr"])
    assert np.array_equal(osl.cpu().numpy()[:orp[-1]], ref["sslots"])
    # per-group lists: the oracle's canonical slot lists regrouped by group
    want = [[] for _ in range(w.K)]
    for b in range(w.B):
        for s in ref["sslots"][ref["srowptr"][b]:ref["srowptr"][b + 1]]:
            want[s // w.G].append((b << 16) | (s % w.G))
    gp = ogp.cpu().numpy()
    ge = oge.cpu().numpy()
    assert gp[0] == 0 and gp[-1] == len(ref["sslots"])
    for k in range(w.K):
        assert sorted(ge[gp[k]:gp[k + 1]].tolist()) == sorted(want[k]), k
    _status_ok(lay)


@pytest.mark.parametrize("engine", [SIMT, TC], ids=["simt", "tc"])
def test_fwd(case, engine):
    w, engines, p, ref = case
    if engine not in engines:
        pytest.skip("engine not used for this shape")
    lay = _layout(p, engine)
    d = dev_problem(p)
    Z = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    _run(sg.sg_fwd, lay, d["h"], d["W"], Z)
    assert_close(host_bf16_to_f64(Z), ref["Z"], what="Z")
    _status_ok(lay)


@pytest.mark.parametrize("engine", [SIMT, TC], ids=["simt", "tc"])
def test_fwd_bce(case, engine, oracle_mod):
    w, engines, p, ref = case
    if engine not in engines:
        pytest.skip("engine not used for this shape")
    lay = _layout(p, engine)
    d = dev_problem(p)
    dZ = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    Z = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    for with_z in (False, True):
        _run(sg.sg_fwd_bce, lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dZ, loss,
             Z if with_z else None)
        assert_close(host_bf16_to_f64(dZ), ref["dZ"], what="dZ")
        assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)
        if with_z:
            assert_close(host_bf16_to_f64(Z), ref["Z"], what="Z")
    _status_ok(lay)


def test_bce_grad_stage(case, oracle_mod):
    """sg_bce_grad on a Z drawn by the generator (not produced by the GPU)."""
    w, engines, p, ref = case
    lay = _layout(p, SIMT)
    zbits = draw_bf16_matrix(1234, w.B, w.L, 3.0)
    want_dZ, want_loss = oracle_mod.bce(zbits, ref["srowptr"], ref["sslots"])
    d = dev_problem(p)
    dZ = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_bce_grad(lay, dev_bf16(zbits), w.B, d["rowptr"], d["labels"], p.nnz, dZ, loss)
    assert_close(host_bf16_to_f64(dZ), want_dZ, what="dZ")
    assert float(loss.item()) == pytest.approx(want_loss, rel=LOSS_RTOL)
    _status_ok(lay)


@pytest.mark.parametrize("engine", [SIMT, TC], ids=["simt", "tc"])
def test_bwd_stage(case, engine, oracle_mod):
    """sg_bwd / sg_bwd_dW / sg_bwd_dh on a dZ drawn by the generator."""
    w, engines, p, ref = case
    if engine not in engines:
        pytest.skip("engine not used for this shape")
    lay = _layout(p, engine)
    dzbits = draw_bf16_matrix(99, w.B, w.L, 0.5)
    want_dW = oracle_mod.weight_grad(p.h, dzbits, ref["idx_sorted"], w.G, w.F)
    want_dh = oracle_mod.feature_grad(p.W, dzbits, ref["idx_sorted"], w.G, w.H)
    d = dev_problem(p)
    dZ = dev_bf16(dzbits)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.full((w.B, w.H), float("nan"), dtype=torch.float32, device="cuda")
    _run(sg.sg_bwd_dW, lay, dZ, d["h"], dW)
    assert_close(host_bf16_to_f64(dW), want_dW, what="dW")
    _run(sg.sg_bwd_dh, lay, dZ, w.B, d["W"], dh)
    assert_close(dh.cpu().numpy(), want_dh, what="dh")
    dW.zero_()
    dh.fill_(7.0)
    _run(sg.sg_bwd, lay, dZ, d["h"], d["W"], dW, dh)
    assert_close(host_bf16_to_f64(dW), want_dW, what="dW")
    assert_close(dh.cpu().numpy(), want_dh, what="dh")
    _status_ok(lay)


@pytest.mark.parametrize("engine", [SIMT, TC], ids=["simt", "tc"])
def test_step_chain(case, engine):
    """The whole step from h, W and the positives."""
    w, engines, p, ref = case
    if engine not in engines:
        pytest.skip("engine not used for this shape")
    lay = _layout(p, engine)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    for _ in range(2):  # a second call must give the same answer (scratch reuse)
        _run(sg.sg_step, lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
        assert_close(host_bf16_to_f64(dW), ref["dW"], what="dW")
        assert_close(dh.cpu().numpy(), ref["dh"], what="dh")
        assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)
    _status_ok(lay)


# ------------------------------------------------------------------ edge cases
def test_empty_positive_lists(oracle_mod):
    w = _w("nopos", B=8, H=64, L=256, G=16, F=16, pos=0)
    p = generate(w)
    ref = oracle_mod.step(p)
    lay = build_layout(p, max_nnz=1)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], 0, dW, dh, loss)
    assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)
    assert_close(dh.cpu().numpy(), ref["dh"], what="dh")


_BY_NAME = {w.name: w for w, _ in CASES}


# kernels each workload shape launches: the fused forward + BCE + dW kernel
# and the dh kernel
_FUSED = ["like3m", "like670k", "like8p6m", "g64_b256", "g128_b256_sub", "g64_b200_f64",
          "g32_b150_f256", "g16_b256_f256", "g64_b256_f256", "g256_b256"]
_FUSED_KINDS = {n: {"prep", "fwd", "dh"} for n in _FUSED}


@pytest.mark.parametrize("name", _FUSED)
def test_step_fused_on_tensor_cores(name, oracle_mod):
    """The shapes of the three label-space workloads run the whole step on
    the tensor cores (engine pinned: a CUDA-core fallback would raise) through
    the fused forward + BCE + dW kernel (no separate dW launch) and the dh
    kernel."""
    w = _BY_NAME[name]
    p = generate(w)
    ref = oracle_mod.step(p)
    lay = _layout(p, TC)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_timing_start(lay, 64)
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
    rec = sg.sg_timing_stop(lay)
    _status_ok(lay)
    launched = {k for k, (ms, n) in rec.items() if n > 0}
    assert launched == _FUSED_KINDS[name], rec
    assert_close(host_bf16_to_f64(dW), ref["dW"], what="dW")
    assert_close(dh.cpu().numpy(), ref["dh"], what="dh")


# shapes of the single-kernel step (B <= 128, G in {16, 32, 64}, F % 16 == 0,
# F <= 128): one CTA per cluster (H within one TMEM band), two or three CTAs,
# a group count that is not a multiple of the cluster size, B = 1 and B <= 64
_SINGLE = ["tiny", "like3m", "like3m_oddK", "like8p6m", "g32_b100", "tc_b37_h320", "b1",
           "dense_F_eq_H", "clustered", "f16_h1000_c3"]
_BY_NAME["like3m_oddK"] = _w("like3m_oddK", B=128, H=768, L=32 * 301, G=32, F=128, pos=36, dist="zipf")
_BY_NAME["f16_h1000_c3"] = _w("f16_h1000_c3", B=96, H=1000, L=16 * 90, G=16, F=16, pos=3)


@pytest.mark.parametrize("name", _SINGLE)
def test_step_single_kernel(name, oracle_mod):
    """The whole step in one kernel on CTA clusters (engine SG_ENGINE_FUSED):
    dW, dh and the loss against the oracle, twice in a row (the layout's
    scratch and the kernel's shared-memory state must not leak between
    calls), and only the preparation kernels besides the step kernel run."""
    w = CONFIGS["tiny"] if name == "tiny" else _BY_NAME[name]
    p = generate(w)
    ref = oracle_mod.step(p)
    lay = build_layout(p)
    sg.sg_layout_set_engine(lay, sg.SG_ENGINE_FUSED)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    for _ in range(2):
        sg.sg_timing_start(lay, 64)
        sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
        rec = sg.sg_timing_stop(lay)
        _status_ok(lay)
        assert {k for k, (ms, n) in rec.items() if n > 0} == {"prep", "step"}, rec
        assert_close(host_bf16_to_f64(dW), ref["dW"], what="dW")
        assert_close(dh.cpu().numpy(), ref["dh"], what="dh")
        assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)


def test_step_single_kernel_large_weights(oracle_mod):
    """Weights beyond fp16's exact range (|W| ~ 2^16) in every third group,
    through the single-kernel step: those groups add their part of dh in fp32
    on CUDA cores, the rest on the tensor cores.  The large-weight groups read
    feature columns 320..447 (across the two CTAs' dh bands, so both take the
    fp32 path) where h >= 0, and their weights are positive: their logits are
    ~10^7, sigmoid is exactly 1 and dZ = 1 - y is exact, so dh is well
    conditioned in them.  (Inside the step dZ reaches dh as one fp16 plane:
    with O(1) logits and |W| ~ 2^16 its rounding alone moves dh by ~|W| 2^-12
    per term, beyond the tolerance wherever dh cancels to near zero.)"""
    w = _w("bigw1", B=128, H=768, L=32 * 40, G=32, F=128, pos=36, dist="zipf")
    p = generate(w)
    big = (np.arange(w.K) % 3) == 0
    cols = np.arange(320, 448, dtype=np.int32)
    idx = p.idx.copy()
    idx[big] = cols
    p.idx = idx
    hb = p.h.copy()
    hb[:, cols] &= np.uint16(0x7FFF)  # h >= 0 on the large-weight groups' columns
    p.h = hb
    # W is in slot order (slot s belongs to group s // G): positive and x 2^20
    # in the large-weight groups' rows
    slot_big = big[np.arange(w.L) // w.G]
    wb = p.W.astype(np.uint32)
    we = (wb >> 7) & 0xFF
    scaled = ((wb & 0x7FFF) + (20 << 7)).astype(np.uint32)
    p.W = np.where((we > 0) & (we < 0xFF - 20) & slot_big[:, None], scaled, wb).astype(np.uint16)
    assert np.abs(bf16_bits_to_f32(p.W)).max() > 2.0 ** 15
    ref = oracle_mod.step(p)
    lay = build_layout(p)
    sg.sg_layout_set_engine(lay, sg.SG_ENGINE_FUSED)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
    _status_ok(lay)
    assert_close(host_bf16_to_f64(dW), ref["dW"], what="dW")
    assert_close(dh.cpu().numpy(), ref["dh"], what="dh")
    assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)


@pytest.mark.parametrize("name", ["tiny", "like3m", "like670k", "like8p6m", "b256_f256", "g64_b256",
                                  "g64_b200_f64"])
def test_step_sgd_two_steps(name, oracle_mod):
    """sg_step_sgd against the oracle's step followed by its momentum-SGD update
    (Loss and training strategy), twice, each step from the library's own W and
    momentum of the step before.  The momentum may differ from the exact one by
    the gradient's tolerance, W by that times lr plus one bf16 rounding.
    Covers the fused path (dW never leaves the chip) and the unfused ones."""
    w = CONFIGS["tiny"] if name == "tiny" else _BY_NAME[name]
    p = generate(w)
    lay = build_layout(p)
    d = dev_problem(p)
    rng = np.random.default_rng(3)
    lr, mu = 0.05, 0.9
    m = (rng.standard_normal((w.L, w.F)) * 0.1).astype(np.float32)
    W_bits = p.W.copy()
    for step in range(2):
        p.W = W_bits
        ref = oracle_mod.step(p)
        W_ref, m_ref = oracle_mod.sgd_momentum(W_bits, ref["dW"], m.astype(np.float64), lr, mu)
        W_in = dev_bf16(W_bits)
        W_out = torch.empty_like(W_in)
        mom = torch.from_numpy(m.copy()).cuda()
        dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
        loss = torch.zeros(1, dtype=torch.float64, device="cuda")
        sg.sg_step_sgd(lay, d["h"], W_in, d["rowptr"], d["labels"], p.nnz, lr, mu, mom, W_out, dh, loss)
        _status_ok(lay)
        m_gpu = mom.cpu().numpy().astype(np.float64)
        W_gpu = W_out.cpu().numpy().view(np.uint16)
        m_tol = ZTOL * (1.0 + np.abs(ref["dW"])) + 1e-6 * (1.0 + np.abs(m_ref))
        assert np.all(np.abs(m_gpu - m_ref) <= m_tol), f"step {step}: momentum"
        Wg = bf16_bits_to_f32(W_gpu).astype(np.float64)
        Wr = bf16_bits_to_f32(W_ref).astype(np.float64)
        assert np.all(np.abs(Wg - Wr) <= 2.0 ** -7 * np.abs(Wr) + lr * m_tol), f"step {step}: W"
        assert_close(dh.cpu().numpy(), ref["dh"], what=f"step {step}: dh")
        assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)
        W_bits, m = W_gpu.copy(), mom.cpu().numpy()


def test_step_sgd_rejects_aliased_weights():
    w = CONFIGS["tiny"]
    p = generate(w)
    lay = build_layout(p)
    d = dev_problem(p)
    mom = torch.zeros((w.L, w.F), dtype=torch.float32, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    with pytest.raises(sg.SGError) as e:
        sg.sg_step_sgd(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, 0.1, 0.9, mom, d["W"], dh, loss)
    assert e.value.status == sg.SG_ERR_INVALID


def test_step_large_weights(oracle_mod):
    """|W| far above the fp16 range (W x 2^20, exact in bf16): inside the step
    dh multiplies fp16 copies of dZ and of W scaled by 2^-s, and scales the
    sums back by 2^s; the result must match the oracle as for ordinary W."""
    w = _w("bigw", B=128, H=768, L=32 * 40, G=32, F=128, pos=36, dist="zipf")
    p = generate(w)
    bits = p.W.astype(np.uint32)
    expo = (bits >> 7) & 0xFF
    scale = (expo > 0) & (expo < 0xFF - 20)
    p.W = np.where(scale, bits + (20 << 7), bits).astype(np.uint16)
    assert np.abs(bf16_bits_to_f32(p.W)).max() > 2.0 ** 16
    ref = oracle_mod.step(p)
    lay = build_layout(p)
    d = dev_problem(p)
    dW = torch.empty((w.L, w.F), dtype=torch.int16, device="cuda")
    dh = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_step(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dW, dh, loss)
    _status_ok(lay)
    assert_close(host_bf16_to_f64(dW), ref["dW"], what="dW")
    assert_close(dh.cpu().numpy(), ref["dh"], what="dh")
    assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)


def test_duplicate_positives_count_once(oracle_mod):
    w = CONFIGS["tiny"]
    p = generate(w)
    # repeat every positive of sample 0 three times
    row0 = p.pos_label[p.pos_rowptr[0]:p.pos_rowptr[1]]
    labels = np.concatenate([np.repeat(row0, 3), p.pos_label[p.pos_rowptr[1]:]]).astype(np.int32)
    rowptr = p.pos_rowptr.copy()
    rowptr[1:] += 2 * len(row0)
    p.pos_rowptr, p.pos_label = rowptr, labels
    ref = oracle_mod.step(p)
    lay = build_layout(p)
    d = dev_problem(p)
    dZ = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_fwd_bce(lay, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dZ, loss)
    assert_close(host_bf16_to_f64(dZ), ref["dZ"], what="dZ")
    assert float(loss.item()) == pytest.approx(ref["loss"], rel=LOSS_RTOL)


def test_layout_rejects_bad_data():
    w = CONFIGS["tiny"]
    p = generate(w)
    bad = p.groups.copy()
    bad[3] = w.K  # group id out of range
    with pytest.raises(sg.SGError) as e:
        sg.sg_layout_build(dev_i32(bad), w.L, w.G, dev_i32(p.idx.reshape(-1)), w.F, w.H, 4, 4)
    assert e.value.status == sg.SG_ERR_DATA
    bad = p.groups.copy()
    bad[0], bad[1] = bad[1], bad[1]  # one group too big, another too small
    if bad[0] != p.groups[0]:
        with pytest.raises(sg.SGError) as e:
            sg.sg_layout_build(dev_i32(bad), w.L, w.G, dev_i32(p.idx.reshape(-1)), w.F, w.H, 4, 4)
        assert e.value.status == sg.SG_ERR_DATA
    bidx = p.idx.copy()
    bidx[7, 3] = bidx[7, 4]  # duplicate index
    with pytest.raises(sg.SGError) as e:
        sg.sg_layout_build(dev_i32(p.groups), w.L, w.G, dev_i32(bidx.reshape(-1)), w.F, w.H, 4, 4)
    assert e.value.status == sg.SG_ERR_DATA
    bidx = p.idx.copy()
    bidx[9, 0] = w.H  # index out of range
    with pytest.raises(sg.SGError) as e:
        sg.sg_layout_build(dev_i32(p.groups), w.L, w.G, dev_i32(bidx.reshape(-1)), w.F, w.H, 4, 4)
    assert e.value.status == sg.SG_ERR_DATA


def test_bad_positive_label_sets_status():
    w = CONFIGS["tiny"]
    p = generate(w)
    lay = build_layout(p)
    d = dev_problem(p)
    labels = p.pos_label.copy()
    labels[2] = w.L + 5
    dZ = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_fwd_bce(lay, d["h"], d["W"], d["rowptr"], dev_i32(labels), p.nnz, dZ, loss)
    assert sg.sg_layout_status(lay) == sg.SG_ERR_DATA
    assert sg.sg_layout_status(lay) == 0  # cleared by the first read
    rp = p.pos_rowptr.copy()
    rp[3] = rp[4] + 1  # non-monotone row pointers
    sg.sg_fwd_bce(lay, d["h"], d["W"], dev_i32(rp), d["labels"], p.nnz, dZ, loss)
    assert sg.sg_layout_status(lay) == sg.SG_ERR_DATA
    lay.close()


def test_device_status_reports_a_layouts_word_without_clearing_it():
    gc.collect()  # free layouts other tests left to the collector
    if sg.sg_device_status() != 0:
        pytest.skip("another live layout on this device already holds an error")
    w = CONFIGS["tiny"]
    p = generate(w)
    good = build_layout(p)
    bad = build_layout(p)
    d = dev_problem(p)
    labels = p.pos_label.copy()
    labels[1] = w.L + 1
    dZ = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    sg.sg_fwd_bce(good, d["h"], d["W"], d["rowptr"], d["labels"], p.nnz, dZ, loss)
    assert sg.sg_device_status() == 0
    sg.sg_fwd_bce(bad, d["h"], d["W"], d["rowptr"], dev_i32(labels), p.nnz, dZ, loss)
    assert sg.sg_device_status() == sg.SG_ERR_DATA
    assert sg.sg_device_status() == sg.SG_ERR_DATA  # reading does not clear
    assert sg.sg_layout_status(good) == 0
    assert sg.sg_layout_status(bad) == sg.SG_ERR_DATA  # clears the word
    assert sg.sg_device_status() == 0
    sg.sg_fwd_bce(bad, d["h"], d["W"], d["rowptr"], dev_i32(labels), p.nnz, dZ, loss)
    bad.close()  # a freed layout no longer counts
    assert sg.sg_device_status() == 0
    good.close()


def test_call_argument_errors():
    w = CONFIGS["tiny"]
    p = generate(w)
    lay = build_layout(p, max_B=8, max_nnz=8)
    d = dev_problem(p)
    Z = torch.empty((w.B, w.L), dtype=torch.int16, device="cuda")
    with pytest.raises(sg.SGError) as e:  # B above max_B
        sg.sg_fwd(lay, d["h"], d["W"], Z)
    assert e.value.status == sg.SG_ERR_INVALID
    with pytest.raises(sg.SGError) as e:  # nnz above max_nnz
        sg.sg_bce_grad(lay, Z[:8].contiguous(), 8, d["rowptr"][:9].contiguous(),
                       d["labels"][:16].contiguous(), 16, Z[:8].contiguous(),
                       torch.zeros(1, dtype=torch.float64, device="cuda"))
    assert e.value.status == sg.SG_ERR_INVALID
    with pytest.raises(sg.SGError) as e:
        sg.sg_layout_set_engine(build_layout(generate(_w("g3", 4, 30, 30, 3, 5))), TC)
    assert e.value.status == sg.SG_ERR_UNSUPPORTED


# ------------------------------------------------------------------ engine range
# largest F (multiple of 16) at which all three phases of a step run on the
# tensor cores, by batch class and G (the table of include/sg.h)
_TC_MAX_F = {128: {16: 256, 32: 256, 64: 256, 128: 160, 192: 32, 256: 0},
             256: {16: 192, 32: 192, 64: 176, 128: 144, 192: 0, 256: 0}}
# F beyond that which the fused forward + BCE + dW kernel still takes (as
# subgroups of the group sharing I_k)
_TC_FUSED_EXTRA = {128: {128: {256}, 256: {64, 128}},
                   256: {16: {256}, 32: {256}, 64: {256}, 128: {256}, 256: {64, 128}}}


def test_step_plan_matches_documented_range():
    """sg_step_plan over G in {16, ..., 256}, F in {16, ..., 256} and B from 1
    to 256: the step runs every phase on the tensor cores exactly where the
    header's table says, and dh on the tensor cores everywhere."""
    for B in (1, 100, 128, 129, 256):
        cls = 128 if B <= 128 else 256
        for G in (16, 32, 64, 128, 192, 256):
            for F in range(16, 257, 16):
                L = G * 4
                groups = np.arange(L, dtype=np.int32) // G
                idx = np.tile(np.arange(F, dtype=np.int32), (4, 1))
                lay = sg.sg_layout_build(dev_i32(groups), L, G, dev_i32(idx.reshape(-1)), F, 256, B, 1)
                try:
                    path, f, w, h = sg.sg_step_plan(lay, B)
                finally:
                    lay.close()
                assert h, (B, G, F)
                want = F <= _TC_MAX_F[cls][G] or F in _TC_FUSED_EXTRA.get(cls, {}).get(G, set())
                assert (f and w and h) == want, (B, G, F, path, f, w, h)


@pytest.mark.parametrize("G,F", [(128, 128), (256, 64), (256, 256)])
def test_dh_stage_large_groups_tc(G, F, oracle_mod):
    """sg_bwd_dh on the tensor cores for groups of more than 64 labels (run as
    subgroups of 64 sharing I_k), against the oracle's dh."""
    w = _w(f"dh_g{G}_f{F}", B=96, H=512, L=G * 12, G=G, F=F, pos=3)
    p = generate(w)
    lay = build_layout(p)
    sg.sg_layout_set_engine(lay, TC)
    ids = sg.sg_layout_export(lay)[2].cpu().numpy().view(np.uint16)
    dzbits = draw_bf16_matrix(98, w.B, w.L, 0.5)
    want_dh = oracle_mod.feature_grad(p.W, dzbits, ids, w.G, w.H)
    dh = torch.full((w.B, w.H), float("nan"), dtype=torch.float32, device="cuda")
    sg.sg_bwd_dh(lay, dev_bf16(dzbits), w.B, dev_bf16(p.W), dh)
    torch.cuda.synchronize()
    assert_close(dh.cpu().numpy(), want_dh, what="dh")
    _status_ok(lay)
    lay.close()
