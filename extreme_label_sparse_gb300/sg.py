"""Thin ctypes binding of libsg (include/sg.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes torch
CUDA tensors where the C call takes device pointers; shapes and dtypes are
checked, the current torch stream is passed, and a non-zero status raises
SGError with the library's message.  No arithmetic of the layer happens here.
If libsg.so has not been built the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import threading
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libsg.so"
_lock = threading.Lock()
_lib = None

SG_OK, SG_ERR_INVALID, SG_ERR_UNSUPPORTED, SG_ERR_CUDA = 0, -1, -2, -3
SG_ERR_OOM, SG_ERR_TIMEOUT, SG_ERR_DATA = -4, -5, -6
SG_ENGINE_AUTO, SG_ENGINE_SIMT, SG_ENGINE_TC, SG_ENGINE_FUSED = 0, 1, 2, 3
KIND_NAMES = ("prep", "fwd", "bce", "dW", "dh", "step")


class SGError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


def lib_path() -> Path:
    return _LIB_PATH


def load():
    """Load libsg.so (raises if it is missing: build it first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH} is not built; run "
                               "extreme_label_sparse_gb300.build() first")
        lib = C.CDLL(str(_LIB_PATH))
        P, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        sig = {
            "sg_layout_build": ([P, i64, i32, P, i32, i32, i32, i64, P, C.POINTER(P)], C.c_int),
            "sg_layout_export": ([P, P, P, P, P], C.c_int),
            "sg_layout_free": ([P], None),
            "sg_layout_set_engine": ([P, i32], C.c_int),
            "sg_layout_info": ([P, C.POINTER(i64), C.POINTER(i32), C.POINTER(i32),
                                C.POINTER(i32), C.POINTER(i64)], C.c_int),
            "sg_layout_status": ([P, C.POINTER(i32), i32], C.c_int),
            "sg_device_status": ([C.POINTER(i32)], C.c_int),
            "sg_pos_export": ([P, i32, P, P, i64, P, P, P, P, P], C.c_int),
            "sg_fwd": ([P, P, i32, P, P, P], C.c_int),
            "sg_bce_grad": ([P, P, i32, P, P, i64, P, P, P], C.c_int),
            "sg_fwd_bce": ([P, P, i32, P, P, P, i64, P, P, P, P], C.c_int),
            "sg_bwd": ([P, P, P, i32, P, P, P, P], C.c_int),
            "sg_bwd_dW": ([P, P, P, i32, P, P], C.c_int),
            "sg_bwd_dh": ([P, P, i32, P, P, P], C.c_int),
            "sg_step": ([P, P, i32, P, P, P, i64, P, P, P, P], C.c_int),
            "sg_step_sgd": ([P, P, i32, P, P, P, i64, C.c_float, C.c_float, P, P, P, P, P], C.c_int),
            "sg_bce_grad_noalloc": ([P, i32, i64, i32, P, P, i64, P, P, P], C.c_int),
            "sg_selftest_wait_timeout": ([C.POINTER(i32)], C.c_int),
            "sg_proj_fwd": ([P, i32, i32, P, i32, P, P], C.c_int),
            "sg_step_plan": ([P, i32, i32, C.POINTER(i32)], C.c_int),
            "sg_rewire": ([P, P, i32, P, P, i32, P, P, P], C.c_int),
            "sg_grouping_create": ([i64, i32, i32, i32, C.POINTER(P)], C.c_int),
            "sg_grouping_free": ([P], None),
            "sg_grouping_status": ([P, C.POINTER(i32)], C.c_int),
            "sg_grouping_embed": ([P, P, i32, P, P, i64, C.POINTER(i64), P], C.c_int),
            "sg_grouping_set_embeddings": ([P, P, P, P], C.c_int),
            "sg_grouping_kmeans_init": ([P, P, P], C.c_int),
            "sg_grouping_set_centroids": ([P, P, P, P], C.c_int),
            "sg_grouping_kmeans_batch": ([P, P, i32, P, P], C.c_int),
            "sg_grouping_groups": ([P, P, P, P], C.c_int),
            "sg_grouping_export": ([P, P, P, P, P, P], C.c_int),
            "sg_proj_bwd": ([P, i32, i32, P, i32, P, P, P, P, i32, P], C.c_int),
            "sg_headtail_step": ([P, P, P, i32, i32, P, P, P, P, P, i64, P, P, P, i64, P, P, P, P, P, P, P],
                                 C.c_int),
            "sg_timing_start": ([P, i32], C.c_int),
            "sg_timing_stop": ([P, P, P], C.c_int),
            "sg_last_error": ([], C.c_char_p),
            "sg_status_string": ([i32], C.c_char_p),
            "sg_abi_version": ([], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().sg_status_string(int(status)).decode()


def last_error() -> str:
    return load().sg_last_error().decode()


def _check(status: int):
    if status != SG_OK:
        raise SGError(status, last_error())


def _stream(device: torch.device):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dev(t: torch.Tensor, name: str, dtypes, numel=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return C.c_void_p(t.data_ptr())


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_I32 = (torch.int32,)


class Layout:
    """Owner of an sg_layout handle (freed on close / garbage collection)."""

    def __init__(self, handle: C.c_void_p, L, G, F, H, max_B, max_nnz, device):
        self.handle = handle
        self.L, self.G, self.F, self.H = int(L), int(G), int(F), int(H)
        self.K = self.L // self.G
        self.max_B, self.max_nnz = int(max_B), int(max_nnz)
        self.device = device

    def close(self):
        if self.handle is not None and _lib is not None:
            _lib.sg_layout_free(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def _as_parameter_(self):
        if self.handle is None:
            raise ValueError("layout is closed")
        return self.handle


# ---------------------------------------------------------------- layout
def sg_layout_build(groups: torch.Tensor, L: int, G: int, idx: torch.Tensor,
                    F: int, H: int, max_B: int, max_nnz: int) -> Layout:
    lib = load()
    g = _dev(groups, "groups", _I32, L)
    K = L // G if G > 0 else 0
    i = _dev(idx, "idx", _I32, K * F)
    out = C.c_void_p()
    _check(lib.sg_layout_build(g, L, G, i, F, H, max_B, max_nnz,
                               _stream(groups.device), C.byref(out)))
    return Layout(out, L, G, F, H, max_B, max_nnz, groups.device)


def sg_layout_export(layout: Layout):
    """-> (slot_of_label[L] int32, label_of_slot[L] int32, idx_sorted[K, F] int16 bits)"""
    lib = load()
    dev = layout.device
    sol = torch.empty(layout.L, dtype=torch.int32, device=dev)
    los = torch.empty(layout.L, dtype=torch.int32, device=dev)
    ids = torch.empty((layout.K, layout.F), dtype=torch.int16, device=dev)
    _check(lib.sg_layout_export(layout, C.c_void_p(sol.data_ptr()),
                                C.c_void_p(los.data_ptr()), C.c_void_p(ids.data_ptr()),
                                _stream(dev)))
    return sol, los, ids


def sg_layout_set_engine(layout: Layout, engine: int):
    _check(load().sg_layout_set_engine(layout, int(engine)))


def sg_layout_status(layout: Layout, clear: bool = True) -> int:
    code = C.c_int32(0)
    _check(load().sg_layout_status(layout, C.byref(code), int(bool(clear))))
    return int(code.value)


def sg_device_status() -> int:
    """First non-zero status word among the live layouts of the current
    device (0 if none); reads without clearing."""
    code = C.c_int32(0)
    _check(load().sg_device_status(C.byref(code)))
    return int(code.value)


# ---------------------------------------------------------------- positives
def sg_pos_export(layout: Layout, B: int, pos_rowptr, pos_label, nnz: int):
    """-> (rowptr[B+1], slots[nnz], gptr[K+1], gentry[nnz]) device int32;
    rows of `slots` beyond rowptr[B] and entries beyond gptr[K] are unused."""
    lib = load()
    dev = layout.device
    rp = _dev(pos_rowptr, "pos_rowptr", _I32, B + 1)
    lb = _dev(pos_label, "pos_label", _I32, nnz) if nnz else C.c_void_p(0)
    orp = torch.empty(B + 1, dtype=torch.int32, device=dev)
    osl = torch.zeros(max(nnz, 1), dtype=torch.int32, device=dev)
    ogp = torch.empty(layout.K + 1, dtype=torch.int32, device=dev)
    oge = torch.zeros(max(nnz, 1), dtype=torch.int32, device=dev)
    _check(lib.sg_pos_export(layout, B, rp, lb, nnz, C.c_void_p(orp.data_ptr()),
                             C.c_void_p(osl.data_ptr()), C.c_void_p(ogp.data_ptr()),
                             C.c_void_p(oge.data_ptr()), _stream(dev)))
    return orp, osl, ogp, oge


# ---------------------------------------------------------------- compute
def _B_of(h: torch.Tensor, H: int) -> int:
    if h.dim() != 2 or h.shape[1] != H:
        raise ValueError(f"h must be [B, {H}]")
    return int(h.shape[0])


def sg_fwd(layout: Layout, h, W, Z):
    B = _B_of(h, layout.H)
    _check(load().sg_fwd(layout, _dev(h, "h", _BF16), B,
                         _dev(W, "W", _BF16, layout.L * layout.F),
                         _dev(Z, "Z", _BF16, B * layout.L), _stream(h.device)))


def sg_bce_grad(layout: Layout, Z, B: int, pos_rowptr, pos_label, nnz: int, dZ, loss):
    lb = _dev(pos_label, "pos_label", _I32, nnz) if nnz else C.c_void_p(0)
    _check(load().sg_bce_grad(layout, _dev(Z, "Z", _BF16, B * layout.L), B,
                              _dev(pos_rowptr, "pos_rowptr", _I32, B + 1), lb, nnz,
                              _dev(dZ, "dZ", _BF16, B * layout.L),
                              _dev(loss, "loss", (torch.float64,), 1), _stream(Z.device)))


def sg_fwd_bce(layout: Layout, h, W, pos_rowptr, pos_label, nnz: int, dZ, loss, Z=None):
    B = _B_of(h, layout.H)
    lb = _dev(pos_label, "pos_label", _I32, nnz) if nnz else C.c_void_p(0)
    zp = _dev(Z, "Z", _BF16, B * layout.L) if Z is not None else C.c_void_p(0)
    _check(load().sg_fwd_bce(layout, _dev(h, "h", _BF16), B,
                             _dev(W, "W", _BF16, layout.L * layout.F),
                             _dev(pos_rowptr, "pos_rowptr", _I32, B + 1), lb, nnz,
                             _dev(dZ, "dZ", _BF16, B * layout.L),
                             _dev(loss, "loss", (torch.float64,), 1), zp, _stream(h.device)))


def sg_bwd(layout: Layout, dZ, h, W, dW, dh):
    B = _B_of(h, layout.H)
    _check(load().sg_bwd(layout, _dev(dZ, "dZ", _BF16, B * layout.L), _dev(h, "h", _BF16), B,
                         _dev(W, "W", _BF16, layout.L * layout.F),
                         _dev(dW, "dW", _BF16, layout.L * layout.F),
                         _dev(dh, "dh", (torch.float32,), B * layout.H), _stream(h.device)))


def sg_bwd_dW(layout: Layout, dZ, h, dW):
    B = _B_of(h, layout.H)
    _check(load().sg_bwd_dW(layout, _dev(dZ, "dZ", _BF16, B * layout.L), _dev(h, "h", _BF16), B,
                            _dev(dW, "dW", _BF16, layout.L * layout.F), _stream(h.device)))


def sg_bwd_dh(layout: Layout, dZ, B: int, W, dh):
    _check(load().sg_bwd_dh(layout, _dev(dZ, "dZ", _BF16, B * layout.L), B,
                            _dev(W, "W", _BF16, layout.L * layout.F),
                            _dev(dh, "dh", (torch.float32,), B * layout.H), _stream(dZ.device)))


def sg_step(layout: Layout, h, W, pos_rowptr, pos_label, nnz: int, dW, dh, loss):
    B = _B_of(h, layout.H)
    lb = _dev(pos_label, "pos_label", _I32, nnz) if nnz else C.c_void_p(0)
    _check(load().sg_step(layout, _dev(h, "h", _BF16), B,
                          _dev(W, "W", _BF16, layout.L * layout.F),
                          _dev(pos_rowptr, "pos_rowptr", _I32, B + 1), lb, nnz,
                          _dev(dW, "dW", _BF16, layout.L * layout.F),
                          _dev(dh, "dh", (torch.float32,), B * layout.H),
                          _dev(loss, "loss", (torch.float64,), 1), _stream(h.device)))


def sg_step_sgd(layout: Layout, h, W_in, pos_rowptr, pos_label, nnz: int, lr: float, mu: float,
                mom, W_out, dh, loss):
    """The step, then the output layer's momentum-SGD update: mom <- mu mom + dW,
    W_out <- bf16(W_in - lr mom).  W_out must not overlap W_in."""
    B = _B_of(h, layout.H)
    n = layout.L * layout.F
    lb = _dev(pos_label, "pos_label", _I32, nnz) if nnz else C.c_void_p(0)
    _check(load().sg_step_sgd(layout, _dev(h, "h", _BF16), B, _dev(W_in, "W_in", _BF16, n),
                              _dev(pos_rowptr, "pos_rowptr", _I32, B + 1), lb, nnz,
                              float(lr), float(mu), _dev(mom, "mom", (torch.float32,), n),
                              _dev(W_out, "W_out", _BF16, n),
                              _dev(dh, "dh", (torch.float32,), B * layout.H),
                              _dev(loss, "loss", (torch.float64,), 1), _stream(h.device)))


# ---------------------------------------------------------------- timing
def sg_timing_start(layout: Layout, capacity: int):
    _check(load().sg_timing_start(layout, int(capacity)))


def sg_timing_stop(layout: Layout):
    """-> {kind: (total_ms, launches)} for the launches since sg_timing_start."""
    ms = (C.c_double * len(KIND_NAMES))()
    n = (C.c_int32 * len(KIND_NAMES))()
    _check(load().sg_timing_stop(layout, C.cast(ms, C.c_void_p), C.cast(n, C.c_void_p)))
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KIND_NAMES)}


# ---------------------------------------------------------------- no allocation
def sg_bce_grad_noalloc(Z, B: int, L: int, G: int, pos_rowptr, pos_slot, nnz: int, dZ, loss):
    """sg_bce_grad without a layout and without any device allocation: for
    callers whose device memory is owned by someone else.  Positives are slot
    ids.  Calls share one fixed working array: do not overlap them."""
    ps = _dev(pos_slot, "pos_slot", _I32, nnz) if nnz else C.c_void_p(0)
    _check(load().sg_bce_grad_noalloc(_dev(Z, "Z", _BF16, B * L), B, L, G,
                                      _dev(pos_rowptr, "pos_rowptr", _I32, B + 1), ps, nnz,
                                      _dev(dZ, "dZ", _BF16, B * L),
                                      _dev(loss, "loss", (torch.float64,), 1), _stream(Z.device)))


# ---------------------------------------------------------------- self-test
def sg_selftest_wait_timeout() -> int:
    """Run the bounded-wait self-test on the current device; returns the
    status the kernel recorded (SG_ERR_TIMEOUT when failure detection works)."""
    code = C.c_int32(0)
    _check(load().sg_selftest_wait_timeout(C.byref(code)))
    return int(code.value)


# ---------------------------------------------------------------- head-tail split
def sg_proj_fwd(h: torch.Tensor, P: torch.Tensor, out: torch.Tensor):
    """out[B][D] = bf16(h[B][E] P[D][E]^T) (bf16 tensors as int16/bfloat16)."""
    B, E = h.shape
    D = P.shape[0]
    _check(load().sg_proj_fwd(_dev(h, "h", _BF16, B * E), B, E, _dev(P, "P", _BF16, D * E), D,
                              _dev(out, "out", _BF16, B * D), _stream(h.device)))


def sg_proj_bwd(h: torch.Tensor, P: torch.Tensor, g: torch.Tensor, work: torch.Tensor, dP: torch.Tensor,
                dh: torch.Tensor, accumulate_dh: bool = False):
    """dP = g^T h, dh (+)= g P (fp32); work holds 2*B*D bf16."""
    B, E = h.shape
    D = P.shape[0]
    _check(load().sg_proj_bwd(_dev(h, "h", _BF16, B * E), B, E, _dev(P, "P", _BF16, D * E), D,
                              _dev(g, "g", (torch.float32,), B * D), _dev(work, "work", _BF16, 2 * B * D),
                              _dev(dP, "dP", (torch.float32,), D * E), _dev(dh, "dh", (torch.float32,), B * E),
                              int(bool(accumulate_dh)), _stream(h.device)))


def sg_headtail_step(head: "Layout", tail: "Layout", h, P_head, P_tail, W_head, head_rowptr, head_label,
                     head_nnz, W_tail, tail_rowptr, tail_label, tail_nnz, dW_head, dW_tail, dP_head, dP_tail,
                     dh, loss):
    B, E = h.shape
    Dh, H = head.H, tail.H
    _check(load().sg_headtail_step(
        head, tail, _dev(h, "h", _BF16, B * E), B, E, _dev(P_head, "P_head", _BF16, Dh * E),
        _dev(P_tail, "P_tail", _BF16, H * E), _dev(W_head, "W_head", _BF16, head.L * head.F),
        _dev(head_rowptr, "head_rowptr", _I32, B + 1), _dev(head_label, "head_label", _I32), int(head_nnz),
        _dev(W_tail, "W_tail", _BF16, tail.L * tail.F), _dev(tail_rowptr, "tail_rowptr", _I32, B + 1),
        _dev(tail_label, "tail_label", _I32), int(tail_nnz), _dev(dW_head, "dW_head", _BF16, head.L * head.F),
        _dev(dW_tail, "dW_tail", _BF16, tail.L * tail.F), _dev(dP_head, "dP_head", (torch.float32,), Dh * E),
        _dev(dP_tail, "dP_tail", (torch.float32,), H * E), _dev(dh, "dh", (torch.float32,), B * E),
        _dev(loss, "loss", (torch.float64,), 1), _stream(h.device)))


SG_PLAN_PER_PHASE, SG_PLAN_FUSED_FWDW, SG_PLAN_ONE_KERNEL = 0, 1, 2


def sg_step_plan(layout: "Layout", B: int, sgd: bool = False):
    """(path, forward on tensor cores, dW on tensor cores, dh on tensor cores)
    of a step of B samples on this layout."""
    plan = (C.c_int32 * 4)()
    _check(load().sg_step_plan(layout, int(B), int(bool(sgd)), plan))
    return int(plan[0]), bool(plan[1]), bool(plan[2]), bool(plan[3])


# ---------------------------------------------------------------- semantic grouping
class Grouping:
    """Owner of an sg_grouping handle (freed on close / garbage collection)."""

    def __init__(self, handle, L, D, G, C, device):
        self.handle = handle
        self.L, self.D, self.G, self.C = int(L), int(D), int(G), int(C)
        self.device = device

    def close(self):
        if self.handle is not None and _lib is not None:
            _lib.sg_grouping_free(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def _as_parameter_(self):
        if self.handle is None:
            raise ValueError("grouping is closed")
        return self.handle


def sg_grouping_create(L: int, D: int, G: int, n_clusters: int, device=None) -> Grouping:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        out = C.c_void_p()
        _check(load().sg_grouping_create(int(L), int(D), int(G), int(n_clusters), C.byref(out)))
    return Grouping(out, L, D, G, n_clusters, dev)


def sg_grouping_status(g: Grouping) -> int:
    code = C.c_int32(0)
    _check(load().sg_grouping_status(g, C.byref(code)))
    return int(code.value)


def sg_grouping_embed(g: Grouping, h, rowptr, labels, nnz: int) -> int:
    N = h.shape[0]
    n = C.c_int64(0)
    lb = _dev(labels, "labels", _I32) if nnz else C.c_void_p(0)
    _check(load().sg_grouping_embed(g, _dev(h, "h", _BF16, N * g.D), N, _dev(rowptr, "rowptr", _I32, N + 1), lb,
                                    int(nnz), C.byref(n), _stream(h.device)))
    return int(n.value)


def sg_grouping_set_embeddings(g: Grouping, E, has):
    _check(load().sg_grouping_set_embeddings(g, _dev(E, "E", _BF16, g.L * g.D), _dev(has, "has", (torch.uint8,), g.L),
                                             _stream(E.device)))


def sg_grouping_kmeans_init(g: Grouping, init_labels):
    _check(load().sg_grouping_kmeans_init(g, _dev(init_labels, "init_labels", _I32, g.C),
                                          _stream(init_labels.device)))


def sg_grouping_set_centroids(g: Grouping, centroids, counts=None):
    cp = _dev(counts, "counts", (torch.int64,), g.C) if counts is not None else C.c_void_p(0)
    _check(load().sg_grouping_set_centroids(g, _dev(centroids, "centroids", (torch.float32,), g.C * g.D), cp,
                                            _stream(centroids.device)))


def sg_grouping_kmeans_batch(g: Grouping, batch, assign_out=None):
    M = batch.numel()
    ap = _dev(assign_out, "assign_out", _I32, M) if assign_out is not None else C.c_void_p(0)
    _check(load().sg_grouping_kmeans_batch(g, _dev(batch, "batch", _I32, M), M, ap, _stream(batch.device)))


def sg_grouping_groups(g: Grouping, groups, cluster_out=None):
    cp = _dev(cluster_out, "cluster_out", _I32, g.L) if cluster_out is not None else C.c_void_p(0)
    _check(load().sg_grouping_groups(g, _dev(groups, "groups", _I32, g.L), cp, _stream(groups.device)))


def sg_grouping_export(g: Grouping, E=None, has=None, centroids=None, counts=None):
    dev = g.device

    def ptr(t, name, dt, n):
        return _dev(t, name, dt, n) if t is not None else C.c_void_p(0)

    _check(load().sg_grouping_export(g, ptr(E, "E", _BF16, g.L * g.D), ptr(has, "has", (torch.uint8,), g.L),
                                     ptr(centroids, "centroids", (torch.float32,), g.C * g.D),
                                     ptr(counts, "counts", (torch.int64,), g.C), _stream(dev)))


# ---------------------------------------------------------------- rewiring
def sg_rewire(layout: Layout, h, dZ, W, n_drop: int, idx_out, W_out):
    """One RigL-style re-selection of every group's fan-in set (see sg.h)."""
    B = h.shape[0]
    _check(load().sg_rewire(layout, _dev(h, "h", _BF16, B * layout.H), B, _dev(dZ, "dZ", _BF16, B * layout.L),
                            _dev(W, "W", _BF16, layout.L * layout.F), int(n_drop),
                            _dev(idx_out, "idx_out", _I32, layout.K * layout.F),
                            _dev(W_out, "W_out", _BF16, layout.L * layout.F), _stream(h.device)))
