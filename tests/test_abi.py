"""CPU checks of the C ABI: the library loads, exports every entry point the header
declares, and rejects bad arguments before touching the GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mnb.h")


@pytest.fixture(scope="module")
def lib():
    from gemm_mnb_gemv_gb300 import _build
    try:
        _build.build()
    except RuntimeError as e:  # no nvcc in this environment
        pytest.skip(str(e))
    import gemm_mnb_gemv_gb300 as mnb
    return mnb.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MNB_API\s+[\w\s\*]+?\b(mnb_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["mnb_dequant", "mnb_repack", "mnb_repacked_bytes", "mnb_gemv", "mnb_gemm",
                     "mnb_workspace_bytes", "mnb_gemv_gate_up_swiglu", "mnb_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_initial_error(lib):
    import gemm_mnb_gemv_gb300 as mnb
    assert "sm_103a" in mnb.mnb_version()
    assert isinstance(mnb.mnb_last_error(), str)


def test_repacked_bytes(lib):
    import gemm_mnb_gemv_gb300 as mnb
    from oracle import mnb_oracle as orc
    for K, N, bs in [(4096, 14336, 128), (64, 1, 16), (96, 130, 32), (256, 128, 64), (4096, 4096, 32)]:
        assert mnb.mnb_repacked_bytes(K, N, bs) == orc.repacked_bytes(K, N)
    assert mnb.mnb_repacked_bytes(100, 10, 32) == 0      # K not a multiple of bs
    assert mnb.mnb_repacked_bytes(64, 10, 48) == 0       # bad block size
    assert mnb.mnb_repacked_bytes(0, 10, 32) == 0


def test_workspace_bytes_is_defined(lib):
    import gemm_mnb_gemv_gb300 as mnb
    for M in (1, 2, 16, 17, 2048):
        assert mnb.mnb_workspace_bytes(M, 4096, 4096, 64) >= 0


def _w(packed=16, scales=16, dtype=0, zp=None):
    import gemm_mnb_gemv_gb300 as mnb
    return mnb.MnbWeight(packed, scales, dtype, zp)


@pytest.mark.parametrize("case,expect", [
    (dict(bs=48), 1),            # block size not in {16, 32, 64, 128}
    (dict(bs=8), 1),
    (dict(K=0), 1),
    (dict(N=-3), 1),
    (dict(K=100, bs=32), 2),     # partial last block: valid format, not handled here
    (dict(A=None), 1),
    (dict(A=24), 3),             # misaligned activation pointer
    (dict(Y=8), 3),
    (dict(w=dict(packed=None)), 1),
    (dict(w=dict(scales=4)), 3),
    (dict(w=dict(dtype=7)), 1),
    (dict(w=dict(zp=9)), 3),
])
def test_gemv_validation_without_gpu(lib, case, expect):
    import gemm_mnb_gemv_gb300 as mnb
    K, N, bs = case.get("K", 256), case.get("N", 128), case.get("bs", 32)
    A = case.get("A", 4096)
    Y = case.get("Y", 8192)
    wkw = dict(packed=16, scales=32, dtype=0, zp=None)
    wkw.update(case.get("w", {}))
    w = _w(**wkw)
    st = lib.mnb_gemv(ctypes.c_void_p(A) if A else None, w, K, N, bs,
                      ctypes.c_void_p(Y) if Y else None, None)
    assert st == expect, mnb.mnb_last_error()
    assert mnb.mnb_last_error().startswith("mnb_gemv")


def test_gemm_needs_repacked_above_16_rows(lib):
    import gemm_mnb_gemv_gb300 as mnb
    w = _w(16, 32, 0, None)
    st = lib.mnb_gemm(ctypes.c_void_p(4096), 17, w, None, 256, 128, 32, None, 0,
                      ctypes.c_void_p(8192), None)
    assert st == mnb.MNB_ERR_INVALID_ARG
    assert "repacked" in mnb.mnb_last_error()
    st = lib.mnb_gemm(ctypes.c_void_p(4096), 0, w, None, 256, 128, 32, None, 0,
                      ctypes.c_void_p(8192), None)
    assert st == mnb.MNB_ERR_INVALID_ARG


def test_swiglu_and_dequant_and_repack_validation(lib):
    import gemm_mnb_gemv_gb300 as mnb
    w = _w(16, 32, 1, None)
    bad = _w(None, 32, 1, None)
    assert lib.mnb_gemv_gate_up_swiglu(ctypes.c_void_p(64), w, bad, 256, 128, 32,
                                       ctypes.c_void_p(128), None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_dequant(w, 256, 128, 33, ctypes.c_void_p(64), None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_dequant(w, 256, 128, 32, ctypes.c_void_p(66), None) == mnb.MNB_ERR_MISALIGNED
    assert lib.mnb_repack(None, 256, 128, 32, ctypes.c_void_p(64), None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_repack(ctypes.c_void_p(64), 250, 128, 32, ctypes.c_void_p(64), None) == mnb.MNB_ERR_UNSUPPORTED
