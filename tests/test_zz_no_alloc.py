"""The act-order entry point that allocates nothing, against the oracle.

mnb_gemm_act_order_noalloc is for callers that cannot allocate device memory: it keeps
its scratch (the gathered activation rows, then K-slice partials) in a static device
array inside the library instead of a caller workspace.  Calls in a row with different
shapes -- a small-M call, then a smaller small-M call that reads scratch the first one
left behind, then an M > 16 call on the tensor-core kernel whose K-split partials also
live in that scratch -- each match the fp64 oracle within the product tolerance
|y - y_ref| <= 2e-3 * sum_k |a_k w_nk| + 1e-5, element by element, and each agrees with
the workspace entry point mnb_gemm_act_order to the same bound.  An oversized call is
refused.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import mnb_synth as syn
from oracle import mnb_oracle as orc
from tests.helpers import TOL_ABS, TOL_REL, assert_within_bound, upload_act, upload_weight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import gemm_mnb_gemv_gb300 as mnb
    return mnb, torch, torch.device("cuda:0")


def _case(mnb, torch, dev, name, M, K, N, bs, kind):
    wl = syn.custom(name, M, K, N, bs)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, kind)
    kp, perm, bg = mnb.mnb_act_order_plan(g_idx, K, bs)
    perm_d = torch.from_numpy(perm).to(dev)
    prep = mnb.mnb_act_order_prepare(*upload_weight(w, dev), K, N, bs, perm_d, torch.from_numpy(bg).to(dev), kp)
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    return upload_act(A, dev), kp, perm_d, prep, Y, B


def _call_noalloc(mnb, torch, a, M, prep, perm_d, K, kp, N, bs, y, repacked_ptr=None):
    lib = mnb.load_library()
    pk, sc, zp = prep
    w = mnb.MnbWeight(pk.data_ptr(), sc.data_ptr(), mnb.MNB_F16, zp.data_ptr() if zp is not None else None)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.mnb_gemm_act_order_noalloc(ctypes.c_void_p(a.data_ptr()), M, w,
                                          ctypes.c_void_p(repacked_ptr) if repacked_ptr else None,
                                          ctypes.c_void_p(perm_d.data_ptr()), K, kp, N, bs, None, 0,
                                          ctypes.c_void_p(y.data_ptr()), stream)


def test_noalloc_matches_oracle_calls_in_a_row(env):
    mnb, torch, dev = env
    cases = [("noalloc_first", 8, 2048, 384, 64, "act_order"),
             ("noalloc_second", 4, 1024, 200, 32, "act_order"),
             ("noalloc_tc", 40, 1024, 300, 64, "uneven")]
    prepared = [_case(mnb, torch, dev, *c) for c in cases]
    # the second call gathers fewer rows than the first left in the scratch
    assert cases[1][1] * prepared[1][1] < cases[0][1] * prepared[0][1]
    outs, variants, reps = [], [], []
    for (name, M, K, N, bs, _), (a, kp, perm_d, prep, Y, B) in zip(cases, prepared):
        rep = mnb.mnb_repack(prep[0], kp, N, bs) if M > 16 else None
        reps.append(rep)
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        st = _call_noalloc(mnb, torch, a, M, prep, perm_d, K, kp, N, bs, y,
                           repacked_ptr=rep.data_ptr() if rep is not None else None)
        assert st == mnb.MNB_OK, mnb.mnb_last_error()
        variants.append(mnb.mnb_last_variant())
        outs.append(y)
    torch.cuda.synchronize()
    assert variants[0].startswith("gemm_smallm") and variants[1].startswith("gemm_smallm"), variants
    assert variants[2].startswith("gemm_tcgen05"), variants
    for (name, M, K, N, bs, _), (a, kp, perm_d, prep, Y, B), y, rep in zip(cases, prepared, outs, reps):
        assert_within_bound(y.double().cpu().numpy(), Y, B, name)
        ref = mnb.mnb_gemm_act_order(a, *prep, perm_d, K, kp, N, bs, repacked=rep)
        torch.cuda.synchronize()
        got = y.double().cpu().numpy()
        want = ref.double().cpu().numpy()
        assert np.all(np.abs(got - want) <= TOL_REL * B + TOL_ABS), name
    mnb.mnb_check_device_status()


def test_noalloc_refuses_more_than_its_scratch(env):
    mnb, torch, dev = env
    a, kp, perm_d, prep, _, _ = _case(mnb, torch, dev, "noalloc_big", 1, 4096, 64, 128, "act_order")
    y = torch.empty((1, 64), dtype=torch.float16, device=dev)
    big_m = (8 << 20) // (kp * 2) + 1   # one row more than the 8 MiB scratch holds
    a_big = torch.zeros((big_m, 4096), dtype=torch.float16, device=dev)
    y_big = torch.empty((big_m, 64), dtype=torch.float16, device=dev)
    # M > 16 needs a repacked operand; the call is refused before anything reads it.
    st = _call_noalloc(mnb, torch, a_big, big_m, prep, perm_d, 4096, kp, 64, 128, y_big,
                       repacked_ptr=y_big.data_ptr())
    assert st == mnb.MNB_ERR_UNSUPPORTED and "static" in mnb.mnb_last_error()
    assert _call_noalloc(mnb, torch, a, 1, prep, perm_d, 4096, kp, 64, 128, y) == mnb.MNB_OK
