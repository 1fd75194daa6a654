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


def test_workspace_bytes_f32_layout(lib):
    """fp32 workspace = split activation (4 M K) + exponents (4 M, rounded to 16) + the
    K-slice partials of the 2 M split rows when those run on the small-M kernel."""
    import gemm_mnb_gemv_gb300 as mnb
    assert mnb.mnb_workspace_bytes_f32(1, 4096, 4096, 32) == 0
    for M, K, N, bs in [(2, 4096, 4096, 64), (4, 14336, 256, 32), (8, 12288, 96, 128), (9, 4096, 512, 32),
                        (300, 1024, 200, 32)]:
        head = 4 * M * K + (4 * M + 15) // 16 * 16
        assert mnb.mnb_workspace_bytes_f32(M, K, N, bs) == head + mnb.mnb_workspace_bytes(2 * M, K, N, bs)
    # one shared-memory pass: no partials; K well beyond it: partials of every slice
    assert mnb.mnb_workspace_bytes(8, 4096, 4096, 64) == 0
    assert mnb.mnb_workspace_bytes(8, 14336, 256, 32) % (8 * 256 * 4) == 0
    assert mnb.mnb_workspace_bytes(8, 14336, 256, 32) >= 2 * 8 * 256 * 4
    # M > 16: partials for a K split over the SMs when the output has few tiles, none when
    # it has enough tiles for every SM
    assert mnb.mnb_workspace_bytes(17, 4096, 4096, 64) == 5 * 17 * 4096 * 4
    assert mnb.mnb_workspace_bytes(2048, 4096, 14336, 128) == 0
    assert mnb.mnb_workspace_bytes(300, 1000, 200, 8) == 0  # invalid block size: no split


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


# ---------------------------------------------------------------------------
# Act-order: the planning step is host code, so it runs here against the oracle.
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("kind,K,bs", [("act_order", 4096, 128), ("uneven", 1024, 32), ("identity", 512, 64),
                                       ("uneven", 256, 16), ("act_order", 14336, 32)])
def test_act_order_plan_matches_oracle(lib, kind, K, bs):
    import numpy as np
    import gemm_mnb_gemv_gb300 as mnb
    import mnb_synth as syn
    from oracle import mnb_oracle as orc
    wl = syn.custom(f"abi_plan_{kind}_{K}_{bs}", 1, K, 8, bs)
    g_idx = syn.make_g_idx(wl, kind)
    kp, perm, bg = mnb.mnb_act_order_plan(g_idx, K, bs)
    kp_ref, perm_ref, bg_ref = orc.act_order_plan(g_idx, K, bs)
    assert kp == kp_ref and K <= kp <= 2 * K
    np.testing.assert_array_equal(perm, perm_ref)
    np.testing.assert_array_equal(bg, bg_ref)


def test_act_order_plan_worst_case_and_errors(lib):
    import numpy as np
    import gemm_mnb_gemv_gb300 as mnb
    K, bs = 256, 16
    g_idx = np.arange(K, dtype=np.int32) % (K // bs)   # 16 groups of 16, interleaved: K' = K
    assert mnb.mnb_act_order_plan(g_idx, K, bs)[0] == K
    g_idx = np.zeros(K, dtype=np.int32)
    g_idx[: K // bs] = np.arange(K // bs)               # every group gets 1 member, group 0 gets 241
    kp, perm, bg = mnb.mnb_act_order_plan(g_idx, K, bs)
    assert kp == 16 * 16 + 15 * 16 and kp <= 2 * K
    bad = np.zeros(K, dtype=np.int32)
    bad[77] = K // bs
    with pytest.raises(mnb.MnbError, match=r"g_idx\[77\]=16 is outside 0..16"):
        mnb.mnb_act_order_plan(bad, K, bs)
    bad[77] = -2
    with pytest.raises(mnb.MnbError, match=r"g_idx\[77\]=-2"):
        mnb.mnb_act_order_plan(bad, K, bs)
    kp = ctypes.c_int32(0)
    assert lib.mnb_act_order_plan(None, K, bs, ctypes.byref(kp), None, None) == mnb.MNB_ERR_INVALID_ARG
    gp = g_idx.ctypes.data_as(ctypes.c_void_p)
    assert lib.mnb_act_order_plan(gp, K, bs, None, None, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_act_order_plan(gp, 250, bs, ctypes.byref(kp), None, None) == mnb.MNB_ERR_UNSUPPORTED


def test_act_order_entry_validation_without_gpu(lib):
    import gemm_mnb_gemv_gb300 as mnb
    w = _w(16, 32, 0, None)
    p = ctypes.c_void_p
    # K' outside [K, 2K]
    assert lib.mnb_gemm_act_order(p(64), 1, w, None, p(64), 256, 544, 128, 32, None, 0, p(64), 1 << 20,
                                  p(64), None) == mnb.MNB_ERR_INVALID_ARG
    assert "K_prepared" in mnb.mnb_last_error()
    # workspace too small
    assert lib.mnb_gemm_act_order(p(64), 4, w, None, p(64), 256, 256, 128, 32, None, 0, p(64), 100,
                                  p(64), None) == mnb.MNB_ERR_INVALID_ARG
    assert "workspace" in mnb.mnb_last_error()
    assert mnb.mnb_act_order_workspace_bytes(4, 256) == 4 * 256 * 2
    # perm NULL / misaligned
    assert lib.mnb_gemm_act_order(p(64), 1, w, None, None, 256, 256, 128, 32, None, 0, p(64), 512,
                                  p(64), None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_act_order_gather(p(64), 1, 256, p(68), 256, p(64), None) == mnb.MNB_ERR_MISALIGNED
    assert lib.mnb_act_order_gather(p(64), 1, 256, p(64), 260, p(64), None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_dequant_gidx(w, None, 256, 128, 32, p(64), None) == mnb.MNB_ERR_INVALID_ARG
    # prepare needs zero_points_out when the weight has zero points
    wz = _w(16, 32, 0, 48)
    assert lib.mnb_act_order_prepare(wz, 256, 128, 32, p(64), p(64), 256, p(64), p(64), None,
                                     None) == mnb.MNB_ERR_INVALID_ARG
    assert "zero_points_out" in mnb.mnb_last_error()
