"""CPU oracle for the group-shared fixed fan-in sparse output layer.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg may import this package; the product library never does.  The
arithmetic lives in `sg_oracle.c` (plain C, double precision); this module only
compiles it, marshals numpy arrays through ctypes and returns numpy results.

Inputs h, W, Z and dZ are accepted either as float64 arrays or as uint16 arrays
of bf16 bit patterns; the C side widens bf16 exactly to double.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "sg_oracle.c"
_LIB_PATH = _HERE / "libsg_oracle.so"
_lock = threading.Lock()
_lib = None

OR_OK, OR_ERR_INVALID, OR_ERR_DATA = 0, -1, -6


def build(force: bool = False) -> Path:
    """Compile sg_oracle.c into libsg_oracle.so (gcc, -O2, OpenMP)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", str(tmp), str(_SRC), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(str(_LIB_PATH))
            P = C.c_void_p
            i32, i64 = C.c_int32, C.c_int64
            lib.or_layout_build.argtypes = [i64, i32, P, P, i32, i32, P, P, P]
            lib.or_layout_build.restype = C.c_int
            lib.or_pos_slots.argtypes = [i32, P, P, i64, P, P, P]
            lib.or_pos_slots.restype = C.c_int
            lib.or_forward.argtypes = [i32, i32, i64, i32, i32, P, C.c_int, P, C.c_int, P, P]
            lib.or_forward_at.argtypes = [i32, i32, i32, P, C.c_int, P, C.c_int, P, i64, P, P, P]
            lib.or_bce.argtypes = [i32, i64, P, C.c_int, P, P, P, P]
            lib.or_weight_grad.argtypes = [i32, i32, i64, i32, i32, P, C.c_int, P, C.c_int, P, P]
            lib.or_feature_grad.argtypes = [i32, i32, i64, i32, i32, P, C.c_int, P, C.c_int, P, P]
            lib.or_weight_grad_rows.argtypes = [i32, i32, i64, i32, i32, P, C.c_int, P, C.c_int,
                                                P, P, P, i64, P, P]
            lib.or_feature_grad_rows.argtypes = [i32, i32, i64, i32, i32, P, C.c_int, P, C.c_int,
                                                 P, P, P, i64, P, P, P]
            lib.or_sgd_momentum.argtypes = [i64, P, P, P, C.c_double, C.c_double, P]
            lib.or_sigmoid.argtypes = [C.c_double]
            lib.or_sigmoid.restype = C.c_double
            lib.or_bce_term.argtypes = [C.c_double, C.c_int]
            lib.or_bce_term.restype = C.c_double
            lib.or_bf16_value.argtypes = [C.c_uint16]
            lib.or_bf16_value.restype = C.c_double
            lib.or_num_threads.restype = C.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return C.c_void_p(a.ctypes.data)


def _fp_in(a):
    """(contiguous array, is_bf16 flag) for an h/W/Z/dZ input."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), 1
    return np.ascontiguousarray(a, dtype=np.float64), 0


def num_threads() -> int:
    return int(_load().or_num_threads())


def sigmoid(z: float) -> float:
    return float(_load().or_sigmoid(float(z)))


def bce_term(z: float, y: int) -> float:
    return float(_load().or_bce_term(float(z), int(y)))


def bf16_value(bits: int) -> float:
    return float(_load().or_bf16_value(int(bits)))


# ------------------------------------------------------------------ O1, O2
def layout_build(groups, idx, L: int, G: int, F: int, H: int):
    """-> (status, slot_of_label[L], label_of_slot[L], idx_sorted[K, F] uint16)"""
    groups = np.ascontiguousarray(groups, dtype=np.int32)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    K = L // G if G > 0 else 0
    sol = np.full(L, -1, dtype=np.int32)
    los = np.full(L, -1, dtype=np.int32)
    ids = np.zeros((max(K, 0), F), dtype=np.uint16)
    st = _load().or_layout_build(L, G, _ptr(groups), _ptr(idx), F, H,
                                 _ptr(sol), _ptr(los), _ptr(ids))
    return int(st), sol, los, ids


def pos_slots(rowptr, labels, L: int, slot_of_label):
    """-> (status, out_rowptr[B+1], out_slots[n]) canonical slot lists."""
    rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    sol = np.ascontiguousarray(slot_of_label, dtype=np.int32)
    B = len(rowptr) - 1
    orp = np.zeros(B + 1, dtype=np.int32)
    osl = np.zeros(max(len(labels), 1), dtype=np.int32)
    st = _load().or_pos_slots(B, _ptr(rowptr), _ptr(labels if len(labels) else osl),
                              L, _ptr(sol), _ptr(orp), _ptr(osl))
    return int(st), orp, osl[:orp[-1]].copy()


# ------------------------------------------------------------------ O3..O6
def forward(h, W, idx_sorted, G: int) -> np.ndarray:
    """Z[B, L] (double) = the logits of every (sample, slot)."""
    h, hb = _fp_in(h)
    W, Wb = _fp_in(W)
    ids = np.ascontiguousarray(idx_sorted, dtype=np.uint16)
    B, H = h.shape
    L, F = W.shape
    Z = np.empty((B, L), dtype=np.float64)
    _load().or_forward(B, H, L, G, F, _ptr(h), hb, _ptr(W), Wb, _ptr(ids), _ptr(Z))
    return Z


def forward_at(h, W, idx_sorted, G: int, bs, ss) -> np.ndarray:
    h, hb = _fp_in(h)
    W, Wb = _fp_in(W)
    ids = np.ascontiguousarray(idx_sorted, dtype=np.uint16)
    bs = np.ascontiguousarray(bs, dtype=np.int32)
    ss = np.ascontiguousarray(ss, dtype=np.int64)
    out = np.empty(len(bs), dtype=np.float64)
    _load().or_forward_at(h.shape[1], G, W.shape[1], _ptr(h), hb, _ptr(W), Wb,
                          _ptr(ids), len(bs), _ptr(bs), _ptr(ss), _ptr(out))
    return out


def bce(Z, srowptr, sslots):
    """-> (dZ[B, L] double, loss = sum of the BCE terms)"""
    Z, Zb = _fp_in(Z)
    srowptr = np.ascontiguousarray(srowptr, dtype=np.int32)
    sslots = np.ascontiguousarray(sslots, dtype=np.int32)
    if len(sslots) == 0:
        sslots = np.zeros(1, dtype=np.int32)
    B, L = Z.shape
    dZ = np.empty((B, L), dtype=np.float64)
    loss = np.zeros(1, dtype=np.float64)
    _load().or_bce(B, L, _ptr(Z), Zb, _ptr(srowptr), _ptr(sslots), _ptr(dZ), _ptr(loss))
    return dZ, float(loss[0])


def weight_grad(h, dZ, idx_sorted, G: int, F: int) -> np.ndarray:
    h, hb = _fp_in(h)
    dZ, db = _fp_in(dZ)
    ids = np.ascontiguousarray(idx_sorted, dtype=np.uint16)
    B, H = h.shape
    L = dZ.shape[1]
    dW = np.empty((L, F), dtype=np.float64)
    _load().or_weight_grad(B, H, L, G, F, _ptr(h), hb, _ptr(dZ), db, _ptr(ids), _ptr(dW))
    return dW


def feature_grad(W, dZ, idx_sorted, G: int, H: int) -> np.ndarray:
    W, Wb = _fp_in(W)
    dZ, db = _fp_in(dZ)
    ids = np.ascontiguousarray(idx_sorted, dtype=np.uint16)
    B, L = dZ.shape
    F = W.shape[1]
    dh = np.empty((B, H), dtype=np.float64)
    _load().or_feature_grad(B, H, L, G, F, _ptr(W), Wb, _ptr(dZ), db, _ptr(ids), _ptr(dh))
    return dh


def sgd_momentum(W_bits, dW, m, lr: float, mu: float):
    """One momentum-SGD update of the output layer's weights (O7):
    m <- mu m + dW, W <- bf16(W - lr m).  Returns (new W bits, new m); the
    inputs are not modified."""
    W_bits = np.ascontiguousarray(W_bits, dtype=np.uint16)
    dW = np.ascontiguousarray(dW, dtype=np.float64)
    m_new = np.array(m, dtype=np.float64, copy=True, order="C")
    assert W_bits.shape == dW.shape == m_new.shape
    W_out = np.empty_like(W_bits)
    _load().or_sgd_momentum(W_bits.size, _ptr(W_bits), _ptr(dW), _ptr(m_new), float(lr), float(mu), _ptr(W_out))
    return W_out, m_new


# ------------------------------------------------------------------ sampled
def weight_grad_rows(h, W, idx_sorted, G: int, srowptr, sslots, slots) -> np.ndarray:
    h, hb = _fp_in(h)
    W, Wb = _fp_in(W)
    ids = np.ascontiguousarray(idx_sorted, dtype=np.uint16)
    srowptr = np.ascontiguousarray(srowptr, dtype=np.int32)
    sslots = np.ascontiguousarray(sslots if len(sslots) else np.zeros(1), dtype=np.int32)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    B, H = h.shape
    L, F = W.shape
    out = np.empty((len(slots), F), dtype=np.float64)
    _load().or_weight_grad_rows(B, H, L, G, F, _ptr(h), hb, _ptr(W), Wb, _ptr(ids),
                                _ptr(srowptr), _ptr(sslots), len(slots), _ptr(slots),
                                _ptr(out))
    return out


def feature_grad_rows(h, W, idx_sorted, G: int, srowptr, sslots, rows, want_dh=True):
    """-> (dh rows [n, H] or None, per-row loss [n])"""
    h, hb = _fp_in(h)
    W, Wb = _fp_in(W)
    ids = np.ascontiguousarray(idx_sorted, dtype=np.uint16)
    srowptr = np.ascontiguousarray(srowptr, dtype=np.int32)
    sslots = np.ascontiguousarray(sslots if len(sslots) else np.zeros(1), dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    B, H = h.shape
    L, F = W.shape
    dh = np.empty((len(rows), H), dtype=np.float64) if want_dh else None
    rl = np.empty(len(rows), dtype=np.float64)
    _load().or_feature_grad_rows(B, H, L, G, F, _ptr(h), hb, _ptr(W), Wb, _ptr(ids),
                                 _ptr(srowptr), _ptr(sslots), len(rows), _ptr(rows),
                                 _ptr(dh) if want_dh else None, _ptr(rl))
    return dh, rl


# ------------------------------------------------------------------ chains
def step(problem, want_Z: bool = False) -> dict:
    """Whole step from a workloads.Problem, every output materialised.
    Only for sizes where B x L doubles fit comfortably in host memory."""
    w = problem.w
    st, sol, los, ids = layout_build(problem.groups, problem.idx, w.L, w.G, w.F, w.H)
    if st != OR_OK:
        raise ValueError(f"oracle layout rejected the problem ({st})")
    st, srp, ssl = pos_slots(problem.pos_rowptr, problem.pos_label, w.L, sol)
    if st != OR_OK:
        raise ValueError(f"oracle positives rejected the problem ({st})")
    Z = forward(problem.h, problem.W, ids, w.G)
    dZ, loss = bce(Z, srp, ssl)
    dW = weight_grad(problem.h, dZ, ids, w.G, w.F)
    dh = feature_grad(problem.W, dZ, ids, w.G, w.H)
    out = dict(slot_of_label=sol, label_of_slot=los, idx_sorted=ids,
               srowptr=srp, sslots=ssl, dZ=dZ, loss=loss, dW=dW, dh=dh)
    if want_Z:
        out["Z"] = Z
    return out
