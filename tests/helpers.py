"""Shared test helpers: device upload of synthetic weights and the parity check."""
from __future__ import annotations

import numpy as np

TOL_REL = 2e-3
TOL_ABS = 1e-5


def upload_weight(w, device):
    import torch
    packed = torch.from_numpy(np.ascontiguousarray(w.packed)).to(device)
    scales = torch.from_numpy(np.ascontiguousarray(w.scales)).to(device)
    zp = None if w.zero_points is None else torch.from_numpy(np.ascontiguousarray(w.zero_points)).to(device)
    return packed, scales, zp


def upload_act(A, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(A)).to(device)


def assert_within_bound(y_gpu, Y_ref, B, what=""):
    """|y - Y| <= 2e-3 * sum|a w| + 1e-5 per element, and y finite."""
    y = np.asarray(y_gpu, dtype=np.float64).reshape(Y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    err = np.abs(y - Y_ref)
    tol = TOL_REL * B + TOL_ABS
    bad = err > tol
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside the bound; worst at {i}: "
            f"gpu {y[i]!r} ref {Y_ref[i]!r} err {err[i]:.3e} tol {tol[i]:.3e}")
    return float(np.max(err / tol))


def tc_variant(N: int, f32: bool = False) -> str:
    """Name of the tensor-core kernel the dispatcher picks for M > 16 (fp32: M > 8)."""
    return "gemm_tcgen05_w128xa256" + ("_f32split" if f32 else "")
