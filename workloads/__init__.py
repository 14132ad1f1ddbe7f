"""Seeded synthetic inputs for the group-shared fixed fan-in output layer.

This module only draws random inputs with the shapes and distributions of the
workloads in "HASTE: Hardware-Aware Dynamic Sparse Training for Large Output
Spaces" (main-experiment table: Amazon-670K, Amazon-3M, LF-Paper2Keywords-8.6M).
It holds none of the layer's arithmetic: no dot products, no sigmoid, no sorting
into the layout.  Both the CUDA library's tests/bench and the CPU oracle take
their inputs from here, so the two sides see bit-identical arrays.

The datasets themselves are not used; these draws stand in for them:
  * groups   : a seeded random balanced assignment, group(l) = pi(l) div G with
               pi a random permutation of [0, L).
  * idx      : per group, F distinct feature indices.  "uniform": the F smallest
               of H seeded uniform keys (an unordered F-subset of [0, H)).
               "clustered": the group picks one of 4 contiguous bands of H/4
               dims uniformly, then F distinct dims inside that band.
               The rows are left UNSORTED: sorting them is the layout's job.
  * h        : B x H, N(0, 1) drawn in fp64, rounded to fp32 then bf16 (RNE).
  * W        : L x F in slot order, N(0, 1/F), same rounding.
  * positives: per sample exactly `pos` distinct labels.  "zipf": rank r in
               1..L drawn with P(r) ~ r^-s by inverse CDF on a float64 table,
               label id = r - 1; "uniform": uniform over [0, L).  Draw order is
               kept (rows are unsorted, which the layer must handle).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

__all__ = ["Workload", "CONFIGS", "Problem", "generate", "to_bf16_bits",
           "bf16_bits_to_f32", "sweep_config", "draw_bf16_matrix", "draw_positives"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    G: int
    F: int
    pos: int            # positives per sample
    pos_dist: str       # "uniform" | "zipf"
    zipf_s: float
    idx_mode: str       # "uniform" | "clustered"
    seed: int = 0

    @property
    def K(self) -> int:
        return self.L // self.G

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


CONFIGS = {
    # tiny: B=32, H=256, L=4096 in K=256 groups of 16, F=32, 5 uniform positives
    "tiny": Workload("tiny", B=32, H=256, L=4096, G=16, F=32, pos=5,
                     pos_dist="uniform", zipf_s=0.0, idx_mode="uniform"),
    # Amazon-670K-shaped tail (top 3% labels already moved to the dense head)
    "amazon670k_tail": Workload("amazon670k_tail", B=256, H=768, L=650_000, G=16,
                                F=128, pos=5, pos_dist="zipf", zipf_s=1.1,
                                idx_mode="uniform"),
    # Amazon-3M-shaped tail: full fwd+BCE+bwd step (the headline workload)
    "amazon3m_tail": Workload("amazon3m_tail", B=128, H=768, L=2_900_000, G=32,
                              F=128, pos=36, pos_dist="zipf", zipf_s=1.1,
                              idx_mode="uniform"),
    # LF-Paper2Keywords-8.6M-shaped tail: fused-BCE path, no materialised Z
    "lf8p6m_tail": Workload("lf8p6m_tail", B=64, H=768, L=8_600_000, G=32, F=64,
                            pos=10, pos_dist="zipf", zipf_s=1.2,
                            idx_mode="uniform"),
}


def sweep_config(G: int, idx_mode: str = "uniform") -> Workload:
    """Group-size sweep point at L=2^20, H=768, F=128, B=256.

    The positives of the sweep are not specified; 5 Zipf(1.1) per sample (the
    670K-shaped draw) is the reading taken."""
    return Workload(f"sweep_g{G}_{idx_mode}", B=256, H=768, L=1 << 20, G=G,
                    F=128, pos=5, pos_dist="zipf", zipf_s=1.1, idx_mode=idx_mode)


for _g in (1, 16, 32, 64):
    for _m in ("uniform", "clustered"):
        _w = sweep_config(_g, _m)
        CONFIGS[_w.name] = _w


# ---------------------------------------------------------------- bf16 bits
def to_bf16_bits(x) -> np.ndarray:
    """fp64/fp32 values -> bf16 bit patterns (uint16), round-to-nearest-even
    (the fp64 value is first rounded to fp32, RNE)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- problem
@dataclass
class Problem:
    w: Workload
    groups: np.ndarray      # int32 [L]
    idx: np.ndarray         # int32 [K, F], unsorted rows
    h: np.ndarray           # uint16 bf16 bits [B, H]
    W: np.ndarray           # uint16 bf16 bits [L, F] (slot order)
    pos_rowptr: np.ndarray  # int32 [B+1]
    pos_label: np.ndarray   # int32 [nnz]

    @property
    def nnz(self) -> int:
        return int(self.pos_rowptr[-1])


def _rng(seq: np.random.SeedSequence) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seq))


def _draw_groups(rng, L: int, G: int) -> np.ndarray:
    perm = rng.permutation(L)
    return (perm // G).astype(np.int32)


def _draw_idx(rng, K: int, F: int, H: int, mode: str, chunk: int = 8192) -> np.ndarray:
    out = np.empty((K, F), dtype=np.int32)
    if mode == "uniform":
        for k0 in range(0, K, chunk):
            n = min(chunk, K - k0)
            keys = rng.random((n, H), dtype=np.float32)
            sel = np.argpartition(keys, F - 1, axis=1)[:, :F]
            out[k0:k0 + n] = sel
    elif mode == "clustered":
        if H % 4:
            raise ValueError("clustered idx needs H divisible by 4")
        band = H // 4
        if F > band:
            raise ValueError("clustered idx needs F <= H/4")
        bands = rng.integers(0, 4, size=K)
        for k0 in range(0, K, chunk):
            n = min(chunk, K - k0)
            keys = rng.random((n, band), dtype=np.float32)
            sel = np.argpartition(keys, F - 1, axis=1)[:, :F]
            out[k0:k0 + n] = sel + (bands[k0:k0 + n, None] * band)
    else:
        raise ValueError(f"unknown idx mode {mode!r}")
    return out


def _draw_normal_bf16(rng, rows: int, cols: int, scale: float,
                      chunk_rows: int = 1 << 18) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        n = min(chunk_rows, rows - r0)
        x = rng.standard_normal((n, cols))
        if scale != 1.0:
            x *= scale
        out[r0:r0 + n] = to_bf16_bits(x)
    return out


def _draw_positives(rng, B: int, L: int, n: int, dist: str, s: float):
    if n > L:
        raise ValueError("more positives per sample than labels")
    if dist == "zipf":
        ranks = np.arange(1, L + 1, dtype=np.float64)
        cdf = np.cumsum(ranks ** (-s))
        cdf /= cdf[-1]
    rows = []
    for _ in range(B):
        chosen: list[int] = []
        seen = set()
        while len(chosen) < n:
            m = 2 * (n - len(chosen)) + 8
            if dist == "zipf":
                u = rng.random(m)
                cand = np.searchsorted(cdf, u, side="right")
                cand = np.minimum(cand, L - 1)
            elif dist == "uniform":
                cand = rng.integers(0, L, size=m)
            else:
                raise ValueError(f"unknown positive distribution {dist!r}")
            for c in cand.tolist():
                if c not in seen:
                    seen.add(c)
                    chosen.append(c)
                    if len(chosen) == n:
                        break
        rows.append(chosen)
    rowptr = np.zeros(B + 1, dtype=np.int32)
    rowptr[1:] = np.cumsum([len(r) for r in rows])
    labels = np.array([c for r in rows for c in r], dtype=np.int32)
    return rowptr, labels


def generate(w: Workload, *, B: Optional[int] = None, shard: int = 0) -> Problem:
    """Draw one problem instance for workload `w` (deterministic in w.seed).

    `B` overrides the batch size (used for bounded samples); the other draws do
    not depend on it except h and the positives.  `shard` > 0 draws another
    label shard of the same batch: groups, idx, W and positives come from their
    own streams, h is the shard-0 h (the samples are shared)."""
    if w.L % w.G:
        raise ValueError("L must be a multiple of G")
    B = w.B if B is None else B
    s_groups, s_idx, s_h, s_W, s_pos = np.random.SeedSequence(w.seed).spawn(5)
    if shard:
        s_groups, s_idx, _, s_W, s_pos = np.random.SeedSequence([w.seed, shard]).spawn(5)
    groups = _draw_groups(_rng(s_groups), w.L, w.G)
    idx = _draw_idx(_rng(s_idx), w.K, w.F, w.H, w.idx_mode)
    h = _draw_normal_bf16(_rng(s_h), B, w.H, 1.0)
    W = _draw_normal_bf16(_rng(s_W), w.L, w.F, float(np.sqrt(1.0 / w.F)))
    rowptr, labels = _draw_positives(_rng(s_pos), B, w.L, w.pos, w.pos_dist, w.zipf_s)
    return Problem(w, groups, idx, h, W, rowptr, labels)


def draw_bf16_matrix(seed: int, rows: int, cols: int, scale: float) -> np.ndarray:
    """Stand-alone N(0, scale^2) bf16 matrix (stage inputs such as Z or dZ)."""
    return _draw_normal_bf16(_rng(np.random.SeedSequence(seed)), rows, cols, scale)


def draw_positives(seed: int, B: int, L: int, n: int, dist: str = "zipf", s: float = 1.1):
    """Stand-alone positive lists: B rows of n distinct labels in [0, L)
    ("zipf": rank r with P ~ r^-s, label r - 1; "uniform").  -> (rowptr, labels)."""
    return _draw_positives(_rng(np.random.SeedSequence(seed)), B, L, n, dist, s)

