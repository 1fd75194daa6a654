"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact for the dequantised weights and the repacked operand; within
|y - y_ref| <= 2e-3 * sum_k |a_k w_nk| + 1e-5 per element for every product.  Shapes
cover the measured workloads at full size, ragged tails (N not a multiple of the
column tile, M not a multiple of the row tile), every block size, both scale dtypes,
with and without zero points, and each kernel variant the dispatcher can pick.
"""
from __future__ import annotations

import time

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


DEQUANT_CASES = [
    ("dq_tiny", 256, 128, 32, "f16", True),
    ("dq_ragged16", 96, 130, 16, "f32", True),
    ("dq_ragged64", 192, 200, 64, "f16", False),
    ("dq_f32_128", 512, 77, 128, "f32", True),
    ("dq_attnproj", 4096, 4096, 32, "f16", True),
]


@pytest.mark.parametrize("name,K,N,bs,sdt,zp", DEQUANT_CASES)
def test_dequant_bit_exact(env, name, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(name, 1, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    out = mnb.mnb_dequant(*upload_weight(w, dev), K, N, bs)
    torch.cuda.synchronize()
    ref = orc.dequant_kn_f32(w.packed, w.scales, w.zero_points, K, N, bs)
    got = out.cpu().numpy()
    assert got.shape == (K, N)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_prefill_weight_bit_exact(env):
    mnb, torch, dev = env
    wl = syn.WORKLOADS["prefill_m2048_k4096_n14336"]
    w = syn.make_weight(wl)
    out = mnb.mnb_dequant(*upload_weight(w, dev), wl.K, wl.N, wl.block_size)
    ref = orc.dequant_kn_f32(w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("K,N,bs", [(64, 1, 16), (96, 130, 32), (256, 128, 64), (192, 257, 64),
                                    (4096, 14336, 128)])
def test_repack_bit_exact(env, K, N, bs):
    mnb, torch, dev = env
    packed = syn.random_bytes(syn.fnv1a64(f"repack/{K}/{N}"), N * K // 2).reshape(N, K // 2)
    out = mnb.mnb_repack(torch.from_numpy(packed).to(dev), K, N, bs)
    ref = orc.repack(packed, K, N, bs)
    assert np.array_equal(out.cpu().numpy(), ref)


GEMV_CASES = [
    # name, K, N, bs, scales, zp, act, expected kernel (None: not asserted) -- chosen to hit
    # every M = 1 geometry: the tensor-core streaming kernel (K % 256 == 0, bs >= 32; half-SM
    # CTAs with all stages in flight, whole-K stages on a full SM, K slices), the bulk-copy
    # ring kernel, the register-pipelined kernel and the generic kernel
    ("gv_one_col", 64, 1, 16, "f16", True, "normal", "gemv_f16acc32"),
    ("gv_ragged32", 96, 130, 32, "f16", True, "normal", "gemv_f16acc32"),
    ("gv_ragged64", 192, 200, 64, "f32", False, "normal", None),
    ("gv_bs128", 384, 333, 128, "f32", True, "normal", None),
    ("gv_bs16_mid", 2048, 301, 16, "f16", True, "normal", "gemv_tma_ring"),
    ("gv_k8192", 8192, 300, 64, "f16", True, "normal", "gemv_mma"),
    ("gv_k16384", 16384, 100, 32, "f32", True, "normal", "gemv_tma_ring"),  # zero points, no K slices
    ("gv_k32768", 32768, 70, 128, "f16", False, "normal", "gemv_mma"),  # K slices, one CTA per SM
    ("gv_generic_k48", 48, 5, 16, "f16", True, "normal", "generic"),
    ("gv_generic_k65536", 65536, 9, 64, "f16", True, "normal", "generic"),
    # zero-point rows that are not 16-byte multiples (4, 28, 56 bytes)
    ("gv_zrow4", 1024, 150, 128, "f16", True, "normal", "gemv_tma_ring"),  # read from global
    ("gv_zrow28", 3584, 200, 64, "f32", True, "normal", "gemv_mma"),  # 16-row tiles copy whole
    ("gv_zrow56_down", 14336, 1000, 128, "f16", True, "normal", "gemv_tma_ring"),
    # the tensor-core kernel: ragged last tile with zero points, fp32 scales, several tiles
    # per CTA, K slices on the down-projection shape
    ("gv_mma_ragged_zp", 1024, 1000, 32, "f16", True, "normal", "gemv_mma"),
    ("gv_mma_bs64_f32", 2048, 333, 64, "f32", False, "normal", "gemv_mma"),
    ("gv_mma_bs128_multi", 4096, 3001, 128, "f16", True, "normal", "gemv_mma"),
    ("gv_mma_sliced_f32", 14336, 517, 32, "f32", False, "normal", "gemv_mma"),
    ("gv_mma_one_tile", 256, 16, 32, "f16", True, "normal", "gemv_mma"),
    # more tiles per CTA than ring slots + 1: stages reuse slots and each tile is summed by
    # the last warp to post it (two CTAs of the call per SM, 7 tiles each)
    ("gv_mma_many_tiles", 4096, 32768, 32, "f16", True, "normal", "gemv_mma"),
]


@pytest.mark.parametrize("name,K,N,bs,sdt,zp,act,kernel", GEMV_CASES)
def test_gemv_parity(env, name, K, N, bs, sdt, zp, act, kernel):
    mnb, torch, dev = env
    wl = syn.custom(name, 1, K, N, bs, scales_dtype=sdt, has_zp=zp, act=act)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemv(upload_act(A.reshape(-1), dev), *upload_weight(w, dev), K, N, bs)
    variant = mnb.mnb_last_variant()
    torch.cuda.synchronize()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy()[None, :], Y, B, name)
    if kernel is not None:
        assert variant == kernel or (kernel == "generic" and variant.startswith("generic")), variant


def rows_mapping_takes(M, K, bs):
    """Shapes the row mapping of the GEMV kernel takes (M <= 2 at block size 32, <= 4 at 64)."""
    return bs in (32, 64) and 2 <= M <= 2 * (bs // 32) and K % 256 == 0 and M * K * 2 <= 32768


# The row mapping: both block sizes, every M it takes, ragged N, fp32 scales, no zero points
# with K slices, a single tile, and more tiles than fit two CTAs per SM (small-M kernel).
ROWS_CASES = [
    (2, 4096, 4096, 32, "f16", True, "gemm_rows_mma"),
    (2, 1024, 333, 32, "f32", False, "gemm_rows_mma"),
    (3, 2048, 1000, 64, "f16", True, "gemm_rows_mma"),
    (4, 4096, 517, 64, "f32", True, "gemm_rows_mma"),
    (2, 8192, 700, 64, "f16", False, "gemm_rows_mma"),   # whole-K stage too large: K slices
    (4, 512, 16, 64, "f16", True, "gemm_rows_mma"),      # one tile, two blocks
    (4, 4096, 14336, 64, "f16", True, "gemm_smallm_mma16816"),  # 6 tiles per CTA: small-M kernel
    (3, 4096, 300, 32, "f16", True, "gemm_smallm_mma16816"),    # M > 2 at block size 32
]


@pytest.mark.parametrize("M,K,N,bs,sdt,zp,kernel", ROWS_CASES)
def test_gemm_rows_mapping(env, M, K, N, bs, sdt, zp, kernel):
    mnb, torch, dev = env
    wl = syn.custom(f"rows_{M}_{K}_{N}_{bs}_{sdt}_{zp}", M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemm(upload_act(A, dev), *upload_weight(w, dev), K, N, bs)
    assert mnb.mnb_last_variant() == kernel
    torch.cuda.synchronize()
    mnb.mnb_check_device_status()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)


@pytest.mark.parametrize("wname", ["tiny_gemv_k256_n128", "gemv_attnproj_k4096_n4096",
                                   "mlp_down_k14336_n4096"])
def test_gemv_workloads_full_size(env, wname):
    mnb, torch, dev = env
    wl = syn.WORKLOADS[wname]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemv(upload_act(A.reshape(-1), dev), *upload_weight(w, dev), wl.K, wl.N, wl.block_size)
    torch.cuda.synchronize()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    assert_within_bound(y.cpu().numpy()[None, :], Y, B, wname)


def _swiglu_case(env, wl, kernel=None):
    mnb, torch, dev = env
    wg = syn.make_weight(wl, "gate")
    wu = syn.make_weight(wl, "up")
    A = syn.make_activation(wl)
    out = mnb.mnb_gemv_gate_up_swiglu(upload_act(A.reshape(-1), dev), upload_weight(wg, dev),
                                      upload_weight(wu, dev), wl.K, wl.N, wl.block_size)
    variant = mnb.mnb_last_variant()
    torch.cuda.synchronize()
    ref, g, bg, u, bu = orc.gate_up_swiglu(A, (wg.packed, wg.scales, wg.zero_points),
                                           (wu.packed, wu.scales, wu.zero_points),
                                           wl.K, wl.N, wl.block_size)
    if kernel is not None:
        assert variant == kernel, variant
    tol = orc.swiglu_tolerance(g, bg, u, bu, ref)
    got = out.cpu().numpy().astype(np.float64)[None, :]
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"worst excess {float(np.max(err - tol)):.3e}"


def test_gate_up_swiglu_workload_full_size(env):
    _swiglu_case(env, syn.WORKLOADS["mlp_gate_up_k4096_n14336"])


@pytest.mark.parametrize("K,N,bs,sdt,zp,kernel", [
    (256, 130, 32, "f16", True, None), (1024, 77, 16, "f32", False, None),
    (8192, 65, 64, "f16", True, None), (48, 9, 16, "f16", True, None),
    # the tensor-core pair kernel: half-SM CTAs, zero points with a ragged tile, K slices
    (2048, 333, 64, "f32", False, "gemv_pair_swiglu_mma"),
    (4096, 1000, 128, "f16", True, "gemv_pair_swiglu_mma"),
    (14336, 100, 32, "f32", False, "gemv_pair_swiglu_mma"),
    # more tiles per CTA than ring slots + 1 (the last warp to post a tile sums it)
    (4096, 28672, 128, "f32", False, "gemv_pair_swiglu_mma")])
def test_gate_up_swiglu_ragged(env, K, N, bs, sdt, zp, kernel):
    _swiglu_case(env, syn.custom(f"sw_{K}_{N}_{bs}", 1, K, N, bs, scales_dtype=sdt, has_zp=zp), kernel)


@pytest.mark.parametrize("M", [2, 4, 8, 16])
def test_gemm_small_m_workloads_full_size(env, M):
    mnb, torch, dev = env
    wl = syn.WORKLOADS[f"verify_m{M}_k4096_n4096"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemm(upload_act(A, dev), *upload_weight(w, dev), wl.K, wl.N, wl.block_size)
    # M <= 4 at block size 64: the row mapping of the GEMV kernel; larger M: the small-M kernel
    assert mnb.mnb_last_variant() == ("gemm_rows_mma" if M <= 4 else "gemm_smallm_mma16816")
    torch.cuda.synchronize()
    mnb.mnb_check_device_status()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)


@pytest.mark.parametrize("M,K,N,bs,sdt,zp", [(3, 96, 130, 32, "f16", True), (5, 192, 200, 64, "f16", True),
                                             (13, 384, 77, 128, "f16", True), (7, 48, 33, 16, "f16", True),
                                             (16, 1024, 129, 16, "f16", True),
                                             (2, 1024, 300, 32, "f16", True), (9, 2048, 131, 64, "f32", False),
                                             (16, 4096, 48, 128, "f32", True), (8, 8192, 100, 256 // 2, "f16", False)])
def test_gemm_small_m_ragged(env, M, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"sm_{M}_{K}_{N}_{bs}", M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemm(upload_act(A, dev), *upload_weight(w, dev), K, N, bs)
    torch.cuda.synchronize()
    mnb.mnb_check_device_status()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)


# Every block size the small-M kernel specialises on (1, 2 or 4 chunks of 32 k per group, or
# two groups per chunk for block size 16),
# both scale dtypes, with and without zero points, fewer groups than K-splitting warps, and
# partial last tiles.
@pytest.mark.parametrize("M,K,N,bs,sdt,zp", [(2, 512, 64, 32, "f32", True), (6, 1536, 48, 64, "f32", False),
                                             (11, 1024, 160, 128, "f16", False), (4, 512, 16, 128, "f32", True),
                                             (16, 2048, 33, 32, "f16", True), (3, 4096, 40, 64, "f16", False),
                                             (9, 640, 72, 32, "f32", False), (8, 3072, 32, 128, "f32", True),
                                             # block size 16: two groups per 32-k chunk
                                             (5, 1024, 129, 16, "f16", True), (12, 2048, 48, 16, "f32", False),
                                             (2, 4096, 64, 16, "f32", True), (16, 512, 80, 16, "f16", True)])
def test_gemm_small_m_block_sizes(env, M, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"smb_{M}_{K}_{N}_{bs}_{sdt}_{zp}", M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemm(upload_act(A, dev), *upload_weight(w, dev), K, N, bs)
    expected = "gemm_rows_mma" if rows_mapping_takes(M, K, bs) else "gemm_smallm_mma16816"
    assert mnb.mnb_last_variant() == expected
    torch.cuda.synchronize()
    mnb.mnb_check_device_status()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)


@pytest.mark.parametrize("M,K,N,bs,sdt,zp", [(256, 128, 128, 128, "f16", True),
                                             (17, 128, 130, 32, "f16", True),
                                             (64, 256, 256, 128, "f16", True),
                                             (200, 320, 384, 64, "f32", False),
                                             (300, 1024, 520, 16, "f16", True),
                                             (100, 96, 200, 32, "f32", True),
                                             (513, 4096, 512, 128, "f16", True)])
def test_gemm_large_m_ragged(env, M, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"lm_{M}_{K}_{N}_{bs}", M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    packed, scales, zpt = upload_weight(w, dev)
    rp = mnb.mnb_repack(packed, K, N, bs)
    y = mnb.mnb_gemm(upload_act(A, dev), packed, scales, zpt, K, N, bs, repacked=rp)
    assert mnb.mnb_last_variant().startswith(tc_variant(N))
    torch.cuda.synchronize()
    mnb.mnb_check_device_status()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)


def test_gemm_prefill_full_size_every_output(env):
    """Full-size prefill (M=2048, K=4096, N=14336, bs=128): all 29,360,128 outputs against
    the fp64 oracle, element by element."""
    mnb, torch, dev = env
    wl = syn.WORKLOADS["prefill_m2048_k4096_n14336"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    packed, scales, zpt = upload_weight(w, dev)
    rp = mnb.mnb_repack(packed, wl.K, wl.N, wl.block_size)
    y = mnb.mnb_gemm(upload_act(A, dev), packed, scales, zpt, wl.K, wl.N, wl.block_size, repacked=rp)
    assert mnb.mnb_last_variant() == tc_variant(wl.N)
    yc = y.cpu().numpy()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    assert_within_bound(yc, Y, B, "prefill, every output")


def test_all_codes_equal_zero_point_gives_exact_zero(env):
    mnb, torch, dev = env
    K, N, bs = 512, 96, 32
    G = K // bs
    rng = np.random.default_rng(11)
    zp_ng = rng.integers(0, 16, size=(N, G))
    codes = np.repeat(zp_ng, bs, axis=1).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    zp = np.zeros((N, G // 2), dtype=np.uint8)
    zp |= zp_ng[:, 0::2].astype(np.uint8)
    zp |= (zp_ng[:, 1::2].astype(np.uint8) << 4)
    scales = rng.uniform(0.01, 2, size=(N, G)).astype(np.float16)
    A = rng.standard_normal((4, K)).astype(np.float16)
    t = lambda x: torch.from_numpy(x).to(dev)
    y1 = mnb.mnb_gemv(t(A[0]), t(packed), t(scales), t(zp), K, N, bs)
    y4 = mnb.mnb_gemm(t(A), t(packed), t(scales), t(zp), K, N, bs)
    torch.cuda.synchronize()
    assert np.all(y1.cpu().numpy() == 0) and np.all(y4.cpu().numpy() == 0)


def test_adversarial_extremes(env):
    """|a| = 4 everywhere and codes at 0/15 against zero points 15/0: the largest terms."""
    mnb, torch, dev = env
    K, N, bs = 4096, 64, 32
    G = K // bs
    rng = np.random.default_rng(12)
    codes = np.where(rng.random((N, K)) < 0.5, 0, 15).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    zp_ng = np.where(rng.random((N, G)) < 0.5, 0, 15).astype(np.uint8)
    zp = (zp_ng[:, 0::2] | (zp_ng[:, 1::2] << 4)).astype(np.uint8)
    scales = np.full((N, G), 0.02, dtype=np.float16)
    A = np.where(rng.random((1, K)) < 0.5, -4.0, 4.0).astype(np.float16)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    y = mnb.mnb_gemv(t(A[0]), t(packed), t(scales), t(zp), K, N, bs)
    torch.cuda.synchronize()
    Y, B = orc.matmul(A, packed, scales, zp, K, N, bs)
    assert_within_bound(y.cpu().numpy()[None, :], Y, B, "extremes")


def test_results_are_deterministic(env):
    mnb, torch, dev = env
    wl = syn.WORKLOADS["verify_m8_k4096_n4096"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    wt = upload_weight(w, dev)
    a = upload_act(A, dev)
    r1 = mnb.mnb_gemm(a, *wt, wl.K, wl.N, wl.block_size).clone()
    r2 = mnb.mnb_gemm(a, *wt, wl.K, wl.N, wl.block_size).clone()
    g1 = mnb.mnb_gemv(a[0].contiguous(), *wt, wl.K, wl.N, wl.block_size).clone()
    g2 = mnb.mnb_gemv(a[0].contiguous(), *wt, wl.K, wl.N, wl.block_size).clone()
    torch.cuda.synchronize()
    assert torch.equal(r1, r2) and torch.equal(g1, g2)


def test_graph_capture_replay_matches_eager(env):
    mnb, torch, dev = env
    wl = syn.WORKLOADS["gemv_attnproj_k4096_n4096"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl, rows=4)
    wt = upload_weight(w, dev)
    a = upload_act(A, dev)
    y1 = torch.empty(wl.N, dtype=torch.float16, device=dev)
    y2 = torch.empty((2, wl.N), dtype=torch.float16, device=dev)
    y4 = torch.empty((4, wl.N), dtype=torch.float16, device=dev)
    a0, a2 = a[0].contiguous(), a[:2].contiguous()
    e1 = mnb.mnb_gemv(a0, *wt, wl.K, wl.N, wl.block_size).clone()
    e2 = mnb.mnb_gemm(a2, *wt, wl.K, wl.N, wl.block_size).clone()
    assert mnb.mnb_last_variant() == "gemm_rows_mma"
    e4 = mnb.mnb_gemm(a, *wt, wl.K, wl.N, wl.block_size).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mnb.mnb_gemv(a0, *wt, wl.K, wl.N, wl.block_size, out=y1)
            mnb.mnb_gemm(a2, *wt, wl.K, wl.N, wl.block_size, out=y2)
            mnb.mnb_gemm(a, *wt, wl.K, wl.N, wl.block_size, out=y4)
            mnb.mnb_gemm(a2, *wt, wl.K, wl.N, wl.block_size, out=y2)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, e1) and torch.equal(y2, e2) and torch.equal(y4, e4)


# M > 16 with few output tiles: K split over the SMs (fp32 partials, summed in slice order).
@pytest.mark.parametrize("M,K,N,bs,sdt,zp", [(17, 4096, 512, 64, "f16", True), (40, 2048, 256, 128, "f32", False),
                                             (256, 4096, 384, 32, "f16", True), (100, 1024, 130, 16, "f16", True)])
def test_gemm_tc_split_k(env, M, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"tcsk_{M}_{K}_{N}_{bs}", M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    packed, scales, zpt = upload_weight(w, dev)
    rp = mnb.mnb_repack(packed, K, N, bs)
    a = upload_act(A, dev)
    y = mnb.mnb_gemm(a, packed, scales, zpt, K, N, bs, repacked=rp)
    torch.cuda.synchronize()
    assert mnb.mnb_last_variant() == "gemm_tcgen05_w128xa256_splitk"
    y2 = mnb.mnb_gemm(a, packed, scales, zpt, K, N, bs, repacked=rp)
    # without a workspace the same call runs unsplit
    y0 = mnb.mnb_gemm(a, packed, scales, zpt, K, N, bs, repacked=rp,
                      workspace=torch.empty(0, dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    assert mnb.mnb_last_variant() == "gemm_tcgen05_w128xa256"
    mnb.mnb_check_device_status()
    assert torch.equal(y, y2)  # deterministic
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)
    assert_within_bound(y0.cpu().numpy(), Y, B, wl.name + " unsplit")


def test_small_m_pairs_graph_and_programmatic_launch(env):
    """M > 8 runs as CTA pairs in a clustered launch: a chain of M = 16 GEMMs (each reading
    the previous output) gives the eager bits with programmatic dependent launch and when
    captured in a graph with it."""
    mnb, torch, dev = env
    wl = syn.WORKLOADS["verify_m16_k4096_n4096"]
    ws = [upload_weight(syn.make_weight(wl, f"pairs{i}"), dev) for i in range(3)]
    a = upload_act(syn.make_activation(wl), dev)

    def chain():
        x, outs = a, []
        for w in ws:
            x = mnb.mnb_gemm(x, *w, wl.K, wl.N, wl.block_size)
            outs.append(x)
        torch.cuda.synchronize()
        return [o.clone() for o in outs]

    eager = chain()
    assert mnb.mnb_last_variant() == "gemm_smallm_mma16816"
    mnb.mnb_set_programmatic_launch(True)
    try:
        pdl = chain()
    finally:
        mnb.mnb_set_programmatic_launch(False)
    assert all(torch.equal(x, y) for x, y in zip(pdl, eager))
    ys = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    mnb.mnb_set_programmatic_launch(True)
    try:
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                x = a
                for w, y in zip(ws, ys):
                    mnb.mnb_gemm(x, *w, wl.K, wl.N, wl.block_size, out=y)
                    x = y
    finally:
        mnb.mnb_set_programmatic_launch(False)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    mnb.mnb_check_device_status()
    assert all(torch.equal(x, y) for x, y in zip(ys, eager))
    assert all(bool(torch.isfinite(e).all()) for e in eager)


def test_repack_is_refused_during_capture(env):
    mnb, torch, dev = env
    K, N, bs = 256, 128, 32
    packed = torch.zeros((N, K // 2), dtype=torch.uint8, device=dev)
    out = torch.empty(mnb.mnb_repacked_bytes(K, N, bs), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    status = None
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            try:
                mnb.mnb_repack(packed, K, N, bs, out=out)
            except mnb.MnbError as e:
                status = e.status
    assert status == mnb.MNB_ERR_CAPTURE


def test_programmatic_launch_gives_same_bits(env):
    """A chain of GEMVs where each reads the previous output, with and without
    programmatic dependent launch: identical results."""
    mnb, torch, dev = env
    wl = syn.WORKLOADS["gemv_attnproj_k4096_n4096"]
    ws = [upload_weight(syn.make_weight(wl, f"chain{i}"), dev) for i in range(4)]
    a = upload_act(syn.make_activation(wl).reshape(-1), dev)

    def run():
        x = a
        outs = []
        for w in ws:
            x = mnb.mnb_gemv(x, *w, wl.K, wl.N, wl.block_size)
            outs.append(x)
        torch.cuda.synchronize()
        return [o.clone() for o in outs]

    base = run()
    mnb.mnb_set_programmatic_launch(True)
    try:
        pdl = run()
    finally:
        mnb.mnb_set_programmatic_launch(False)
    for b, p in zip(base, pdl):
        assert torch.equal(b, p)


# Every M = 1 workload runs on the tensor-core streaming kernel (tiny_gemv's 4-byte
# zero-point rows copy whole with its 16-row tiles).
@pytest.mark.parametrize("wname,variant", [("gemv_attnproj_k4096_n4096", "gemv_mma"),
                                           ("mlp_down_k14336_n4096", "gemv_mma"),
                                           ("tiny_gemv_k256_n128", "gemv_mma")])
def test_gemv_dispatch_picks_the_streaming_kernel(env, wname, variant):
    mnb, torch, dev = env
    wl = syn.WORKLOADS[wname]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    mnb.mnb_gemv(upload_act(A.reshape(-1), dev), *upload_weight(w, dev), wl.K, wl.N, wl.block_size)
    assert mnb.mnb_last_variant() == variant


def test_swiglu_dispatch_picks_the_streaming_kernel(env):
    mnb, torch, dev = env
    wl = syn.WORKLOADS["mlp_gate_up_k4096_n14336"]
    wg = upload_weight(syn.make_weight(wl, "gate"), dev)
    wu = upload_weight(syn.make_weight(wl, "up"), dev)
    a = upload_act(syn.make_activation(wl).reshape(-1), dev)
    mnb.mnb_gemv_gate_up_swiglu(a, wg, wu, wl.K, wl.N, wl.block_size)
    assert mnb.mnb_last_variant() == "gemv_pair_swiglu_mma"


def test_bounded_wait_gives_up_and_reports_timeout(env):
    """A kernel whose wait on a never-armed barrier has a 1 ms limit: the wait gives up, the
    kernel returns, the status word reports the timeout once, and the GPU stays usable."""
    mnb, torch, dev = env
    mnb.mnb_check_device_status()  # start from a clean word
    t0 = time.perf_counter()
    mnb.mnb_selftest_wait_timeout(1000)
    with pytest.raises(mnb.MnbError) as exc:
        mnb.mnb_check_device_status()
    elapsed = time.perf_counter() - t0
    assert exc.value.status == mnb.MNB_ERR_TIMEOUT
    assert "wait gave up" in str(exc.value)
    assert elapsed < 5.0  # the 1 ms limit, not the 500 ms default or a hang
    mnb.mnb_check_device_status()  # cleared by the read above
    with pytest.raises(mnb.MnbError) as bad:
        mnb.mnb_selftest_wait_timeout(0)
    assert bad.value.status == mnb.MNB_ERR_INVALID_ARG
    # the context still computes correctly
    wl = syn.WORKLOADS["tiny_gemv_k256_n128"]
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    y = mnb.mnb_gemv(upload_act(A.reshape(-1), dev), *upload_weight(w, dev), wl.K, wl.N, wl.block_size)
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    assert_within_bound(y.cpu().numpy()[None, :], Y, B, "after the wait self-test")
    mnb.mnb_check_device_status()


def test_device_status_is_clean_after_the_suite(env):
    mnb, torch, dev = env
    mnb.mnb_check_device_status()


def test_gate_up_swiglu_weights_with_different_storage(env):
    """Gate with fp16 scales and zero points, up with fp32 scales and none."""
    mnb, torch, dev = env
    wg_l = syn.custom("sw_mixed_gate", 1, 4096, 300, 64, scales_dtype="f16", has_zp=True)
    wu_l = syn.custom("sw_mixed_up", 1, 4096, 300, 64, scales_dtype="f32", has_zp=False)
    wg, wu = syn.make_weight(wg_l, "gate"), syn.make_weight(wu_l, "up")
    A = syn.make_activation(wg_l)
    out = mnb.mnb_gemv_gate_up_swiglu(upload_act(A.reshape(-1), dev), upload_weight(wg, dev),
                                      upload_weight(wu, dev), 4096, 300, 64)
    torch.cuda.synchronize()
    ref, g, bg, u, bu = orc.gate_up_swiglu(A, (wg.packed, wg.scales, wg.zero_points),
                                           (wu.packed, wu.scales, wu.zero_points), 4096, 300, 64)
    tol = orc.swiglu_tolerance(g, bg, u, bu, ref)
    got = out.cpu().numpy().astype(np.float64)[None, :]
    assert np.all(np.abs(got - ref) <= tol)


def test_mlp_chain_gate_up_then_down_full_size(env):
    """Decode MLP: the SwiGLU output (fp16, on the device) feeds the down GEMV directly,
    launched back to back with programmatic dependent launch.  Each step is checked
    against the oracle on the input it actually received."""
    mnb, torch, dev = env
    wgl = syn.WORKLOADS["mlp_gate_up_k4096_n14336"]
    wdl = syn.WORKLOADS["mlp_down_k14336_n4096"]
    wg, wu, wd = syn.make_weight(wgl, "gate"), syn.make_weight(wgl, "up"), syn.make_weight(wdl, "B")
    A = syn.make_activation(wgl)
    tg, tu, td = upload_weight(wg, dev), upload_weight(wu, dev), upload_weight(wd, dev)
    x = upload_act(A.reshape(-1), dev)
    mnb.mnb_set_programmatic_launch(True)
    try:
        h = mnb.mnb_gemv_gate_up_swiglu(x, tg, tu, wgl.K, wgl.N, wgl.block_size)
        y = mnb.mnb_gemv(h, *td, wdl.K, wdl.N, wdl.block_size)
    finally:
        mnb.mnb_set_programmatic_launch(False)
    torch.cuda.synchronize()
    ref, g, bg, u, bu = orc.gate_up_swiglu(A, (wg.packed, wg.scales, wg.zero_points),
                                           (wu.packed, wu.scales, wu.zero_points), wgl.K, wgl.N, wgl.block_size)
    hh = h.cpu().numpy()
    assert np.all(np.abs(hh.astype(np.float64)[None, :] - ref) <= orc.swiglu_tolerance(g, bg, u, bu, ref))
    Y, B = orc.matmul(hh[None, :], wd.packed, wd.scales, wd.zero_points, wdl.K, wdl.N, wdl.block_size)
    assert_within_bound(y.cpu().numpy()[None, :], Y, B, "down after swiglu")


BIAS_CASES = [  # (M, K, N, bs, expected variant prefix)
    (1, 4096, 4096, 32, "gemv_mma"),
    (1, 2048, 300, 16, "gemv_tma_ring"),
    (1, 96, 130, 32, "gemv_f16acc32"),
    (1, 48, 33, 16, "generic"),
    (4, 4096, 300, 64, "gemm_rows_mma"),
    (8, 4096, 300, 64, "gemm_smallm"),
    (3, 96, 77, 16, "generic"),
    (64, 256, 300, 128, "gemm_tcgen05"),
    (40, 256, 100, 64, "gemm_tcgen05"),
]


@pytest.mark.parametrize("M,K,N,bs,variant", BIAS_CASES)
def test_bias_epilogue_both_rounding_modes(env, M, K, N, bs, variant):
    """Mode 2 (round, then add) is bit-identical to mnb_gemm followed by a plain fp16 add;
    mode 1 (add, then round once) is within the product bound plus one fp16 rounding."""
    mnb, torch, dev = env
    wl = syn.custom(f"bias_{M}_{K}_{N}_{bs}", M, K, N, bs)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    bias_np = (syn.normal(syn.fnv1a64(f"{wl.name}/bias"), N) * 2.0).astype(np.float16)
    packed, scales, zpt = upload_weight(w, dev)
    a = upload_act(A, dev)
    rp = mnb.mnb_repack(packed, K, N, bs) if M > 16 else None
    bias = torch.from_numpy(bias_np).to(dev)
    y0 = mnb.mnb_gemm(a, packed, scales, zpt, K, N, bs, repacked=rp)
    y2 = mnb.mnb_gemm_bias(a, packed, scales, zpt, K, N, bs, bias, mnb.MNB_BIAS_AFTER_ROUND, repacked=rp)
    assert mnb.mnb_last_variant().startswith(variant)
    y1 = mnb.mnb_gemm_bias(a, packed, scales, zpt, K, N, bs, bias, mnb.MNB_BIAS_FUSED, repacked=rp)
    torch.cuda.synchronize()
    two_op = (y0.float() + bias.float()[None, :]).half()
    assert torch.equal(y2.view(torch.int16), two_op.view(torch.int16))
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    ref = Y + orc.f16_to_f64(bias_np)[None, :]
    got = y1.cpu().numpy().astype(np.float64)
    tol = 2e-3 * B + 2.0 ** -11 * np.abs(ref) + 1e-5
    assert np.all(np.abs(got - ref) <= tol)


def test_bias_mode_validation(env):
    mnb, torch, dev = env
    a = torch.zeros(64, dtype=torch.float16, device=dev)
    packed = torch.zeros((8, 32), dtype=torch.uint8, device=dev)
    scales = torch.ones((8, 2), dtype=torch.float16, device=dev)
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_gemm_bias(a, packed, scales, None, 64, 8, 32, torch.zeros(8, dtype=torch.float16, device=dev), 5)
    assert e.value.status == mnb.MNB_ERR_INVALID_ARG


# Small M with K beyond one shared-memory pass: K split into slices, fp32 partials in the
# workspace, summed in slice order.
SPLITK_CASES = [
    (2, 14336, 4096, 32, "f32", False),   # the down projection at speculative-verify M
    (5, 8192, 200, 64, "f16", True),
    (13, 12288, 96, 128, "f32", True),
    (3, 14336, 144, 128, "f16", True),    # last slice 2048 of 4096; zero-point rows of 56 bytes
    (16, 10240, 64, 32, "f16", False),
    (4, 16384, 64, 16, "f16", True),      # block size 16, four slices
]


@pytest.mark.parametrize("M,K,N,bs,sdt,zp", SPLITK_CASES)
def test_gemm_small_m_split_k(env, M, K, N, bs, sdt, zp):
    mnb, torch, dev = env
    wl = syn.custom(f"sk_{M}_{K}_{N}_{bs}", M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    need = mnb.mnb_workspace_bytes(M, K, N, bs)
    assert need > 0
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)  # stale contents must not matter
    y = mnb.mnb_gemm(upload_act(A, dev), *upload_weight(w, dev), K, N, bs, workspace=ws)
    torch.cuda.synchronize()
    assert mnb.mnb_last_variant() == "gemm_smallm_mma16816_splitk"
    mnb.mnb_check_device_status()
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert_within_bound(y.cpu().numpy(), Y, B, wl.name)


def test_gemm_small_m_split_k_bias_and_repeat(env):
    mnb, torch, dev = env
    M, K, N, bs = 4, 12288, 256, 64
    wl = syn.custom("sk_bias", M, K, N, bs)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    bias = (syn.normal(syn.fnv1a64("sk_bias/bias"), N) * 0.5).astype(np.float16)
    a, wt, b = upload_act(A, dev), upload_weight(w, dev), upload_act(bias, dev)
    ws = torch.empty(mnb.mnb_workspace_bytes(M, K, N, bs), dtype=torch.uint8, device=dev)
    y0 = mnb.mnb_gemm(a, *wt, K, N, bs, workspace=ws)
    y2 = mnb.mnb_gemm_bias(a, *wt, K, N, bs, b, mnb.MNB_BIAS_AFTER_ROUND, workspace=ws)
    y0b = mnb.mnb_gemm(a, *wt, K, N, bs, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y0, y0b)  # deterministic across calls
    assert torch.equal(y2, (y0.float() + b.float()).half())
    # a workspace smaller than stated is refused
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(mnb.MnbError):
        mnb.mnb_gemm(a, *wt, K, N, bs, workspace=small)
