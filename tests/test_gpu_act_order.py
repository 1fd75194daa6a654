"""GPU parity of the act-order (g_idx) entry points against the fp64 oracle.

Bit-exact: the g_idx dequantisation (including out-of-range groups, which give 0),
the prepared weight and the activation gather.  Within |y - y_ref| <= 2e-3 * B + 1e-5
(B = sum_k |a_k w_nk| over the g_idx weights): the act-order product at every M
regime (GEMV, small M, tcgen05), for balanced act-order groups and uneven groups with
padding, with and without bias.  Also: graph capture, refusal of the one-time
preparation under capture, and the index bit of the device status word.
"""
from __future__ import annotations

import numpy as np
import pytest

import mnb_synth as syn
from oracle import mnb_oracle as orc
from tests.helpers import assert_within_bound, tc_variant, upload_act, upload_weight

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


def _i32(torch, x, dev):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev)


def _prepare(mnb, torch, dev, wl, w, g_idx):
    """Plan on the host, prepare on the device; returns the device pieces and the plan."""
    kp, perm, bg = mnb.mnb_act_order_plan(g_idx, wl.K, wl.block_size)
    perm_d, bg_d = _i32(torch, perm, dev), _i32(torch, bg, dev)
    prep = mnb.mnb_act_order_prepare(*upload_weight(w, dev), wl.K, wl.N, wl.block_size, perm_d, bg_d, kp)
    return kp, perm, bg, perm_d, prep


@pytest.mark.parametrize("kind,K,N,bs,sdt,zp", [
    ("act_order", 512, 130, 32, "f16", True),
    ("uneven", 1024, 64, 64, "f32", True),
    ("uneven", 256, 200, 16, "f16", False),
    ("identity", 384, 96, 128, "f32", False),
])
def test_dequant_gidx_bit_exact(env, kind, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"dqg_{kind}_{K}_{N}", 1, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    g_idx = syn.make_g_idx(wl, kind)
    out = mnb.mnb_dequant_gidx(*upload_weight(w, dev), _i32(torch, g_idx, dev), K, N, bs)
    ref = orc.dequant_kn_f32(w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    mnb.mnb_check_device_status()


def test_dequant_gidx_out_of_range_gives_zero_and_sets_index_bit(env):
    mnb, torch, dev = env
    K, N, bs = 256, 64, 32
    wl = syn.custom("dqg_oob", 1, K, N, bs)
    w = syn.make_weight(wl)
    g_idx = syn.make_g_idx(wl, "uneven").copy()
    g_idx[[3, 100, 255]] = [-1, K // bs, 1 << 30]
    out = mnb.mnb_dequant_gidx(*upload_weight(w, dev), _i32(torch, g_idx, dev), K, N, bs)
    ref = orc.dequant_kn_f32(w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.all(got[[3, 100, 255]] == 0)
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_check_device_status()
    assert e.value.status == mnb.MNB_ERR_INVALID_ARG and "index" in str(e.value)
    mnb.mnb_check_device_status()  # read-and-clear: clean again


@pytest.mark.parametrize("kind,K,N,bs,sdt,zp", [
    ("act_order", 1024, 130, 32, "f16", True),
    ("uneven", 1024, 77, 64, "f32", True),
    ("uneven", 512, 256, 16, "f16", False),
    ("identity", 256, 40, 128, "f16", True),
])
def test_prepare_bit_exact(env, kind, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"prep_{kind}_{K}_{N}", 1, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    g_idx = syn.make_g_idx(wl, kind)
    kp, perm, bg, _, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    rpk, rsc, rzp = orc.act_order_prepare(w.packed, w.scales, w.zero_points, K, N, bs, perm, bg)
    torch.cuda.synchronize()
    assert np.array_equal(pk.cpu().numpy(), rpk)
    assert np.array_equal(sc.cpu().numpy().view(np.uint8), rsc.view(np.uint8))
    if zp:
        assert np.array_equal(zpp.cpu().numpy(), rzp)
    else:
        assert zpp is None and rzp is None
    mnb.mnb_check_device_status()


@pytest.mark.parametrize("M,K,kind,bs", [(1, 4096, "act_order", 128), (3, 1024, "uneven", 32),
                                         (37, 512, "uneven", 16)])
def test_gather_bit_exact(env, M, K, kind, bs):
    mnb, torch, dev = env
    wl = syn.custom(f"gather_{M}_{K}", M, K, 8, bs)
    A = syn.make_activation(wl)
    A[0, :5] = -0.0  # signed zeros are copied as they are
    g_idx = syn.make_g_idx(wl, kind)
    kp, perm, _ = mnb.mnb_act_order_plan(g_idx, K, bs)
    out = mnb.mnb_act_order_gather(upload_act(A, dev), K, _i32(torch, perm, dev), kp)
    ref = orc.act_order_gather(A, perm)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.view(np.uint16))
    mnb.mnb_check_device_status()


ACT_ORDER_CASES = [
    # name, M, K, N, bs, sdt, zp, kind
    ("ao_gemv_bal", 1, 4096, 512, 128, "f16", True, "act_order"),
    ("ao_gemv_uneven", 1, 1024, 320, 32, "f32", False, "uneven"),
    ("ao_gemv_uneven16", 1, 512, 129, 16, "f16", True, "uneven"),
    ("ao_gemv_bigk", 1, 16384, 256, 128, "f16", True, "act_order"),  # K' > 8192: gather pass
    ("ao_small_bal", 4, 2048, 384, 64, "f16", True, "act_order"),
    ("ao_small_uneven", 13, 1024, 200, 32, "f32", True, "uneven"),
    ("ao_tc_bal", 300, 1024, 384, 128, "f16", True, "act_order"),
    ("ao_tc_uneven", 77, 1024, 256, 64, "f16", False, "uneven"),
    # K' beyond one shared-memory pass: K slices with partials after the gathered rows
    ("ao_small_bigk", 4, 12288, 160, 64, "f16", True, "act_order"),
    ("ao_small_bigk_pairs", 12, 8192, 96, 128, "f32", True, "act_order"),
]


@pytest.mark.parametrize("name,M,K,N,bs,sdt,zp,kind", ACT_ORDER_CASES)
def test_gemm_act_order_parity(env, name, M, K, N, bs, sdt, zp, kind):
    mnb, torch, dev = env
    wl = syn.custom(name, M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, kind)
    kp, perm, _, perm_d, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    rep = mnb.mnb_repack(pk, kp, N, bs) if M > 16 else None
    y = mnb.mnb_gemm_act_order(upload_act(A, dev), pk, sc, zpp, perm_d, K, kp, N, bs, repacked=rep)
    torch.cuda.synchronize()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    assert_within_bound(y.float().cpu().numpy(), Y, B, name)
    variant = mnb.mnb_last_variant()
    assert variant != "act_order_gather", variant  # the product kernel's name is reported
    if name == "ao_gemv_bal":
        assert variant == "gemv_tma_ring_gather", variant  # gather fused into the GEMV
    if name == "ao_gemv_bigk":
        assert variant == "gemv_tma_ring", variant  # separate gather, then the GEMV
    if M > 16:
        assert variant.startswith(tc_variant(N)), variant
    if name.startswith("ao_small_bigk"):
        assert variant == "gemm_smallm_mma16816_splitk", variant
    mnb.mnb_check_device_status()


def test_gemm_act_order_bigk_without_room_for_partials_still_correct(env):
    """A workspace of exactly mnb_act_order_workspace_bytes: the K-sliced product has no
    room for its partials and the call takes the generic kernel, with the same bound."""
    mnb, torch, dev = env
    wl = syn.custom("ao_bigk_tight", 3, 12288, 96, 64, scales_dtype="f16", has_zp=True)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, "act_order")
    kp, perm, _, perm_d, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    ws = torch.empty(mnb.mnb_act_order_workspace_bytes(3, kp), dtype=torch.uint8, device=dev)
    y = mnb.mnb_gemm_act_order(upload_act(A, dev), pk, sc, zpp, perm_d, wl.K, kp, wl.N, 64, workspace=ws)
    torch.cuda.synchronize()
    assert mnb.mnb_last_variant() == "generic"
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, 64, g_idx)
    assert_within_bound(y.float().cpu().numpy(), Y, B, wl.name)
    mnb.mnb_check_device_status()


def test_gemm_act_order_bias_modes(env):
    mnb, torch, dev = env
    M, K, N, bs = 5, 1024, 192, 32
    wl = syn.custom("ao_bias", M, K, N, bs)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, "act_order")
    bias = (syn.normal(syn.fnv1a64("ao_bias/bias"), N) * 0.5).astype(np.float16)
    kp, perm, _, perm_d, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    a = upload_act(A, dev)
    b = upload_act(bias, dev)
    y0 = mnb.mnb_gemm_act_order(a, pk, sc, zpp, perm_d, K, kp, N, bs)
    y2 = mnb.mnb_gemm_act_order(a, pk, sc, zpp, perm_d, K, kp, N, bs, bias=b, bias_mode=mnb.MNB_BIAS_AFTER_ROUND)
    y1 = mnb.mnb_gemm_act_order(a, pk, sc, zpp, perm_d, K, kp, N, bs, bias=b, bias_mode=mnb.MNB_BIAS_FUSED)
    torch.cuda.synchronize()
    assert torch.equal(y2, (y0.float() + b.float()).half())
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    ref = Y + bias.astype(np.float64)[None, :]
    err = np.abs(y1.double().cpu().numpy() - ref)
    assert np.all(err <= 2e-3 * B + 2.0 ** -11 * np.abs(ref) + 1e-5)


def test_act_order_full_size_gemv_attnproj(env):
    """Act-order weight of the attention-projection GEMV shape (K = N = 4096, bs 32)."""
    mnb, torch, dev = env
    wl = syn.WORKLOADS["gemv_attnproj_k4096_n4096"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, "act_order")
    kp, perm, _, perm_d, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    assert kp == wl.K
    y = mnb.mnb_gemm_act_order(upload_act(A, dev), pk, sc, zpp, perm_d, wl.K, kp, wl.N, wl.block_size)
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, g_idx)
    assert_within_bound(y.float().cpu().numpy(), Y, B, "act-order attnproj")
    assert mnb.mnb_last_variant().startswith("gemv_tma")


def test_act_order_full_size_prefill_every_output(env):
    """M = 2048, K = 4096, N = 14336, bs 128, act-order groups: every output against the
    fp64 oracle evaluated with g_idx directly."""
    mnb, torch, dev = env
    wl = syn.WORKLOADS["prefill_m2048_k4096_n14336"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, "act_order")
    kp, perm, _, perm_d, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    rep = mnb.mnb_repack(pk, kp, wl.N, wl.block_size)
    y = mnb.mnb_gemm_act_order(upload_act(A, dev), pk, sc, zpp, perm_d, wl.K, kp, wl.N, wl.block_size,
                               repacked=rep).cpu().numpy()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, g_idx)
    assert_within_bound(y.astype(np.float64), Y, B, "act-order prefill, every output")


def test_act_order_graph_capture_and_prepare_refusal(env):
    mnb, torch, dev = env
    M, K, N, bs = 1, 2048, 256, 64
    wl = syn.custom("ao_graph", M, K, N, bs)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g_idx = syn.make_g_idx(wl, "uneven")
    kp, perm, bg, perm_d, (pk, sc, zpp) = _prepare(mnb, torch, dev, wl, w, g_idx)
    a = upload_act(A, dev)
    wt = upload_weight(w, dev)
    bg_d = _i32(torch, bg, dev)
    ws = torch.empty(mnb.mnb_act_order_workspace_bytes(M, kp), dtype=torch.uint8, device=dev)
    eager = mnb.mnb_gemm_act_order(a, pk, sc, zpp, perm_d, K, kp, N, bs, workspace=ws).clone()
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    refused = None
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mnb.mnb_gemm_act_order(a, pk, sc, zpp, perm_d, K, kp, N, bs, workspace=ws, out=y)
            try:
                mnb.mnb_act_order_prepare(*wt, K, N, bs, perm_d, bg_d, kp,
                                          packed_out=pk, scales_out=sc, zero_points_out=zpp)
            except mnb.MnbError as e:
                refused = e.status
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert refused == mnb.MNB_ERR_CAPTURE
    assert torch.equal(y, eager)
