"""GPU parity of the fp32-activation entry point against the fp64 oracle.

Every M regime (fp32 GEMV, split-activation small-M and tcgen05 kernels, the generic
fp32 kernel), both scale dtypes, with and without zero points and bias, ordinary and
very wide activation magnitudes (1e-6 .. 1e6, outside the fp16 range), full-size
shapes, and a case that fails if the activations were rounded to fp16 anywhere.
Bound: |y - y_ref| <= 2e-3 * sum_k |a_k w_nk| + 1e-5 (+ 2^-24 |bias| for the bias add).
"""
from __future__ import annotations

import numpy as np
import pytest

import mnb_synth as syn
from oracle import mnb_oracle as orc
from tests.helpers import assert_within_bound, upload_act, upload_weight

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


def _run(mnb, torch, dev, wl, w, A, bias=None):
    wt = upload_weight(w, dev)
    rep = mnb.mnb_repack(wt[0], wl.K, wl.N, wl.block_size) if wl.M > 8 else None
    b = None if bias is None else upload_act(bias, dev)
    y = mnb.mnb_gemm_f32(upload_act(A, dev), *wt, wl.K, wl.N, wl.block_size, repacked=rep, bias=b)
    torch.cuda.synchronize()
    return y.double().cpu().numpy(), mnb.mnb_last_variant()


F32_CASES = [
    # name, M, K, N, bs, sdt, zp, recipe, bias, expected variant
    ("f32_gemv", 1, 4096, 520, 32, "f16", True, "normal", False, "gemv_f32_tma_ring"),
    ("f32_gemv_wide", 1, 2048, 300, 128, "f32", False, "wide", True, "gemv_f32_tma_ring"),
    ("f32_gemv_cps2", 1, 12288, 160, 64, "f32", True, "normal", False, "gemv_f32_tma_ring"),
    ("f32_gemv_bs16", 1, 1024, 96, 16, "f16", True, "uniform1", True, "gemv_f32_tma_ring"),
    ("f32_gemv_k48", 1, 48, 40, 16, "f16", True, "normal", False, "generic_f32"),
    ("f32_m2", 2, 4096, 384, 64, "f16", True, "normal", False, "gemm_smallm_mma16816_f32split"),
    ("f32_m5_wide", 5, 2048, 200, 32, "f32", True, "wide", True, "gemm_smallm_mma16816_f32split"),
    ("f32_m8", 8, 1024, 130, 128, "f16", False, "normal", False, "gemm_smallm_mma16816_f32split"),
    ("f32_m3_bs16", 3, 512, 64, 16, "f16", True, "normal", False, "gemm_smallm_mma16816_f32split"),
    ("f32_m9", 9, 1024, 256, 64, "f16", True, "normal", True, "gemm_tcgen05_w128xa256_f32split"),
    ("f32_m40_wide", 40, 2048, 384, 128, "f32", True, "wide", False, "gemm_tcgen05_w128xa256_f32split"),
    ("f32_m300", 300, 1024, 200, 32, "f16", False, "normal", True, "gemm_tcgen05_w128xa256_f32split"),
    ("f32_m33_n96", 33, 512, 96, 32, "f16", True, "normal", True, "gemm_tcgen05_w128xa256_f32split"),
    # K beyond one shared-memory pass: K-slice partials of the split rows, then the combine
    ("f32_m4_k14336", 4, 14336, 256, 32, "f32", False, "normal", True, "gemm_smallm_mma16816_f32split_splitk"),
    ("f32_m2_k12288_wide", 2, 12288, 144, 128, "f16", True, "wide", False, "gemm_smallm_mma16816_f32split_splitk"),
    ("f32_m7_k8192", 7, 8192, 96, 64, "f32", True, "normal", True, "gemm_smallm_mma16816_f32split_splitk"),
    ("f32_m12_tc_splitk", 12, 2048, 256, 64, "f16", True, "wide", True, "gemm_tcgen05_w128xa256_f32split_splitk"),
]


@pytest.mark.parametrize("name,M,K,N,bs,sdt,zp,recipe,has_bias,variant", F32_CASES)
def test_gemm_f32_parity(env, name, M, K, N, bs, sdt, zp, recipe, has_bias, variant):
    mnb, torch, dev = env
    wl = syn.custom(name, M, K, N, bs, scales_dtype=sdt, has_zp=zp)
    w = syn.make_weight(wl)
    A = syn.make_activation_f32(wl, recipe=recipe)
    bias = (syn.normal(syn.fnv1a64(name + "/bias"), N) * 0.5).astype(np.float32) if has_bias else None
    y, got_variant = _run(mnb, torch, dev, wl, w, A, bias)
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    if bias is not None:
        Y = Y + bias.astype(np.float64)[None, :]
        B = B + 2.0 ** -24 / 2e-3 * np.abs(bias.astype(np.float64))[None, :]
    assert_within_bound(y, Y, B, name)
    # the tensor-core kernel splits K over the SMs when the output has few tiles
    assert got_variant == variant or (variant.startswith("gemm_tcgen05") and got_variant == variant + "_splitk")
    mnb.mnb_check_device_status()


@pytest.mark.parametrize("M", [1, 4, 20])
def test_gemm_f32_keeps_fp32_activations(env, M):
    """a = 1 + 2^-14 rounds to 1 in fp16 (spacing 2^-10), so any fp16 rounding of the
    activations would be off by 2^-14 * B; the fp32 path must be well inside half of that
    (fp32 accumulation of 2048 positive terms stays far below 2^-15)."""
    mnb, torch, dev = env
    K, N, bs = 2048, 256, 64
    wl = syn.custom(f"f32_exactness_{M}", M, K, N, bs, scale_lo=0.01, scale_hi=0.02, has_zp=False)
    w = syn.make_weight(wl)
    w.packed[:] = 0xFF  # every code 15, zero point 8: all weights positive
    A = np.full((M, K), 1.0 + 2.0 ** -14, dtype=np.float32)
    y, _ = _run(mnb, torch, dev, wl, w, A)
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    assert np.all(np.abs(y - Y) <= 2.0 ** -15 * B), np.max(np.abs(y - Y) / B)


def test_gemm_f32_full_size_attnproj_and_down(env):
    mnb, torch, dev = env
    for key in ("gemv_attnproj_k4096_n4096", "mlp_down_k14336_n4096"):
        wl = syn.WORKLOADS[key]
        w = syn.make_weight(wl)
        A = syn.make_activation_f32(wl)
        y, variant = _run(mnb, torch, dev, wl, w, A)
        Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
        assert_within_bound(y, Y, B, key)
        assert variant == "gemv_f32_tma_ring"


def test_gemm_f32_full_size_prefill_every_output(env):
    """fp32 activations at the prefill shape: every output against the fp64 oracle."""
    mnb, torch, dev = env
    wl = syn.WORKLOADS["prefill_m2048_k4096_n14336"]
    w = syn.make_weight(wl)
    A = syn.make_activation_f32(wl)
    y, variant = _run(mnb, torch, dev, wl, w, A)
    assert variant == "gemm_tcgen05_w128xa256_f32split"
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    assert_within_bound(y, Y, B, "f32 prefill, every output")


def test_gemm_f32_graph_replay(env):
    mnb, torch, dev = env
    wl = syn.custom("f32_graph", 4, 1024, 256, 32)
    w = syn.make_weight(wl)
    wt = upload_weight(w, dev)
    a = upload_act(syn.make_activation_f32(wl), dev)
    ws = torch.empty(mnb.mnb_workspace_bytes_f32(4, wl.K, wl.N, 32), dtype=torch.uint8, device=dev)
    eager = mnb.mnb_gemm_f32(a, *wt, wl.K, wl.N, 32, workspace=ws).clone()
    y = torch.empty((4, wl.N), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mnb.mnb_gemm_f32(a, *wt, wl.K, wl.N, 32, workspace=ws, out=y)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, eager)
