"""The seeded generators: deterministic, with the stated shapes and structure."""
import numpy as np
import pytest

from workloads import CONFIGS, generate, sweep_config, to_bf16_bits, bf16_bits_to_f32


def test_generate_is_deterministic_and_shaped():
    w = CONFIGS["tiny"]
    a, b = generate(w), generate(w)
    for name in ("groups", "idx", "h", "W", "pos_rowptr", "pos_label"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    assert a.h.shape == (w.B, w.H) and a.h.dtype == np.uint16
    assert a.W.shape == (w.L, w.F) and a.W.dtype == np.uint16
    assert a.idx.shape == (w.K, w.F)
    assert np.array_equal(np.bincount(a.groups, minlength=w.K), np.full(w.K, w.G))
    assert all(len(set(r)) == w.F for r in a.idx.tolist())
    assert a.idx.min() >= 0 and a.idx.max() < w.H
    assert np.all(np.diff(a.pos_rowptr) == w.pos)
    for r in range(w.B):
        row = a.pos_label[a.pos_rowptr[r]:a.pos_rowptr[r + 1]]
        assert len(set(row.tolist())) == len(row)


def test_clustered_idx_bands():
    w = sweep_config(16, "clustered").with_(L=4096)
    p = generate(w)
    band = w.H // 4
    lo = p.idx.min(axis=1) // band
    hi = p.idx.max(axis=1) // band
    assert np.array_equal(lo, hi)


def test_value_scales():
    w = CONFIGS["tiny"].with_(L=1 << 15)
    p = generate(w)
    Wf = bf16_bits_to_f32(p.W).astype(np.float64)
    assert abs(Wf.std() - (1 / w.F) ** 0.5) < 0.01
    hf = bf16_bits_to_f32(p.h).astype(np.float64)
    assert abs(hf.std() - 1.0) < 0.05


def test_zipf_positives_skew():
    w = CONFIGS["tiny"].with_(pos_dist="zipf", zipf_s=1.1, B=256)
    p = generate(w)
    counts = np.bincount(p.pos_label, minlength=w.L)
    assert counts[0] > counts[100:].max()


def test_bf16_rounding_is_rne():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8)], dtype=np.float32)
    assert to_bf16_bits(x).tolist() == [0x3F80, 0x3F82, 0xBF80]
