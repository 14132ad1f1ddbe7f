"""CPU-only checks of the C ABI: the library loads without a GPU, exports every
entry point include/sg.h declares, and rejects bad arguments before launching
anything."""
import ctypes as C
import re
from pathlib import Path

import pytest

import extreme_label_sparse_gb300 as sgpkg

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    sgpkg.build()
    return sgpkg.load()


def _declared():
    text = (ROOT / "include" / "sg.h").read_text()
    return sorted(set(re.findall(r"^SG_API\s+[\w\s\*]+?\b(sg_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ("sg_layout_build", "sg_fwd", "sg_bce_grad", "sg_bwd", "sg_fwd_bce",
                 "sg_bwd_dW", "sg_bwd_dh", "sg_step", "sg_pos_export", "sg_layout_export",
                 "sg_device_status", "sg_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_abi_version_and_strings(lib):
    assert lib.sg_abi_version() == 1
    assert sgpkg.status_string(0) == "SG_OK"
    assert sgpkg.status_string(-6) == "SG_ERR_DATA"
    assert sgpkg.status_string(12345) == "SG_ERR_UNKNOWN"


def test_layout_build_validates_before_any_cuda_call(lib):
    out = C.c_void_p(123)
    fake = C.c_void_p(16)  # never dereferenced: validation fails first
    cases = [
        ((fake, 30, 4, fake, 3, 10, 1, 0), sgpkg.SG_ERR_INVALID),    # L % G
        ((fake, 32, 4, fake, 11, 10, 1, 0), sgpkg.SG_ERR_INVALID),   # F > H
        ((fake, 32, 0, fake, 3, 10, 1, 0), sgpkg.SG_ERR_INVALID),    # G < 1
        ((fake, 32, 4, fake, 3, 10, 0, 0), sgpkg.SG_ERR_INVALID),    # max_B < 1
        ((fake, 32, 4, fake, 3, 10, 1, -1), sgpkg.SG_ERR_INVALID),   # max_nnz < 0
        ((None, 32, 4, fake, 3, 10, 1, 0), sgpkg.SG_ERR_INVALID),    # null groups
        ((fake, 512, 512, fake, 3, 10, 1, 0), sgpkg.SG_ERR_UNSUPPORTED),  # G > 256
        ((fake, 32, 4, fake, 3, 65536, 1, 0), sgpkg.SG_ERR_UNSUPPORTED),  # H above u16 idx
        ((fake, 32, 4, fake, 3, 10, 300, 0), sgpkg.SG_ERR_UNSUPPORTED),   # max_B
    ]
    for args, want in cases:
        rc = lib.sg_layout_build(*args, None, C.byref(out))
        assert rc == want, (args, rc, sgpkg.last_error())
        assert out.value is None
        assert sgpkg.last_error()


def test_compute_calls_reject_null_layout(lib):
    P = C.c_void_p(16)
    assert lib.sg_fwd(None, P, 4, P, P, None) == sgpkg.SG_ERR_INVALID
    assert "layout is NULL" in sgpkg.last_error()
    assert lib.sg_step(None, P, 4, P, P, P, 0, P, P, P, None) == sgpkg.SG_ERR_INVALID
    assert lib.sg_bwd(None, P, P, 4, P, P, P, None) == sgpkg.SG_ERR_INVALID
    assert lib.sg_bce_grad(None, P, 4, P, P, 0, P, P, None) == sgpkg.SG_ERR_INVALID
    assert lib.sg_layout_set_engine(None, 0) == sgpkg.SG_ERR_INVALID
    lib.sg_layout_free(None)  # no-op
