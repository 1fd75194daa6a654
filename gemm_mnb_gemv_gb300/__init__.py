"""Python binding of libmnb (block-quantized INT4 MatMulNBits GEMV/GEMM for sm_103a).

Argument marshalling only: every entry point forwards raw device pointers, sizes and
the current CUDA stream to the C ABI declared in ``include/mnb.h``; all arithmetic runs
in the library's CUDA kernels.  PyTorch supplies device memory and streams.  When an
output tensor is not passed, the binding allocates it with torch before the call (pass
``out=`` to keep a call free of allocations, e.g. under CUDA-graph capture).

The names match the C entry points: ``mnb_dequant``, ``mnb_repacked_bytes``,
``mnb_repack``, ``mnb_gemv``, ``mnb_workspace_bytes``, ``mnb_gemm``,
``mnb_gemm_bias``, ``mnb_gemv_gate_up_swiglu``, ``mnb_workspace_bytes_f32``, ``mnb_gemm_f32``,
``mnb_dequant_gidx``,
``mnb_act_order_plan``, ``mnb_act_order_prepare``, ``mnb_act_order_gather``,
``mnb_act_order_workspace_bytes``, ``mnb_gemm_act_order``, ``mnb_gemm_act_order_noalloc``,
``mnb_set_programmatic_launch``,
``mnb_check_device_status``,
``mnb_last_error``,
``mnb_last_variant``, ``mnb_version``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmnb.so")

MNB_OK, MNB_ERR_INVALID_ARG, MNB_ERR_UNSUPPORTED, MNB_ERR_MISALIGNED = 0, 1, 2, 3
MNB_ERR_CAPTURE, MNB_ERR_CUDA, MNB_ERR_TIMEOUT = 4, 5, 6
MNB_F16, MNB_F32 = 0, 1
STATUS_NAMES = {0: "MNB_OK", 1: "MNB_ERR_INVALID_ARG", 2: "MNB_ERR_UNSUPPORTED",
                3: "MNB_ERR_MISALIGNED", 4: "MNB_ERR_CAPTURE", 5: "MNB_ERR_CUDA",
                6: "MNB_ERR_TIMEOUT"}


class MnbError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class MnbWeight(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("scales_dtype", ctypes.c_int32), ("zero_points", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmnb.so (built in-tree by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m gemm_mnb_gemv_gb300._build` "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    c_int, c_size, vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    sigs = {
        "mnb_dequant": (c_int, [MnbWeight, c_int, c_int, c_int, vp, vp]),
        "mnb_repacked_bytes": (c_size, [c_int, c_int, c_int]),
        "mnb_repack": (c_int, [vp, c_int, c_int, c_int, vp, vp]),
        "mnb_gemv": (c_int, [vp, MnbWeight, c_int, c_int, c_int, vp, vp]),
        "mnb_workspace_bytes": (c_size, [c_int, c_int, c_int, c_int]),
        "mnb_gemm": (c_int, [vp, c_int, MnbWeight, vp, c_int, c_int, c_int, vp, c_size, vp, vp]),
        "mnb_gemv_gate_up_swiglu": (c_int, [vp, MnbWeight, MnbWeight, c_int, c_int, c_int, vp, vp]),
        "mnb_gemm_bias": (c_int, [vp, c_int, MnbWeight, vp, c_int, c_int, c_int, vp, c_int, vp, c_size, vp, vp]),
        "mnb_workspace_bytes_f32": (c_size, [c_int, c_int, c_int, c_int]),
        "mnb_gemm_f32": (c_int, [vp, c_int, MnbWeight, vp, c_int, c_int, c_int, vp, vp, c_size, vp, vp]),
        "mnb_dequant_gidx": (c_int, [MnbWeight, vp, c_int, c_int, c_int, vp, vp]),
        "mnb_act_order_plan": (c_int, [vp, c_int, c_int, vp, vp, vp]),
        "mnb_act_order_prepare": (c_int, [MnbWeight, c_int, c_int, c_int, vp, vp, c_int, vp, vp, vp, vp]),
        "mnb_act_order_gather": (c_int, [vp, c_int, c_int, vp, c_int, vp, vp]),
        "mnb_act_order_workspace_bytes": (c_size, [c_int, c_int]),
        "mnb_gemm_act_order": (c_int, [vp, c_int, MnbWeight, vp, vp, c_int, c_int, c_int, c_int, vp, c_int, vp,
                                       c_size, vp, vp]),
        "mnb_gemm_act_order_noalloc": (c_int, [vp, c_int, MnbWeight, vp, vp, c_int, c_int, c_int, c_int, vp,
                                               c_int, vp, vp]),
        "mnb_set_programmatic_launch": (None, [c_int]),
        "mnb_check_device_status": (c_int, []),
        "mnb_selftest_wait_timeout": (c_int, [ctypes.c_uint, vp]),
        "mnb_last_error": (ctypes.c_char_p, []),
        "mnb_last_variant": (ctypes.c_char_p, []),
        "mnb_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _torch():
    import torch
    return torch


def _stream_handle(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_dev(name, t, dtype=None):
    torch = _torch()
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _weight(packed, scales, zero_points) -> MnbWeight:
    torch = _torch()
    _check_dev("packed", packed, torch.uint8)
    _check_dev("scales", scales)
    _check_dev("zero_points", zero_points, torch.uint8)
    if scales.dtype == torch.float16:
        sd = MNB_F16
    elif scales.dtype == torch.float32:
        sd = MNB_F32
    else:
        raise TypeError("scales must be float16 or float32")
    return MnbWeight(packed.data_ptr(), scales.data_ptr(), sd,
                     zero_points.data_ptr() if zero_points is not None else None)


def _raise(status: int):
    if status != MNB_OK:
        raise MnbError(status, load_library().mnb_last_error().decode())


def mnb_last_error() -> str:
    return load_library().mnb_last_error().decode()


def mnb_last_variant() -> str:
    return load_library().mnb_last_variant().decode()


def mnb_version() -> str:
    return load_library().mnb_version().decode()


def mnb_set_programmatic_launch(enable: bool) -> None:
    load_library().mnb_set_programmatic_launch(1 if enable else 0)


def mnb_check_device_status() -> None:
    """Raises MnbError(MNB_ERR_TIMEOUT) if a device-side bounded wait gave up since the last check."""
    _raise(load_library().mnb_check_device_status())


def mnb_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launches the bounded-wait self-test kernel (its wait gives up after ``limit_us``)."""
    _raise(load_library().mnb_selftest_wait_timeout(limit_us, _stream_handle(stream)))


def mnb_repacked_bytes(K: int, N: int, block_size: int) -> int:
    return int(load_library().mnb_repacked_bytes(K, N, block_size))


def mnb_workspace_bytes(M: int, K: int, N: int, block_size: int) -> int:
    return int(load_library().mnb_workspace_bytes(M, K, N, block_size))


def mnb_dequant(packed, scales, zero_points, K: int, N: int, block_size: int, out=None, stream=None):
    """fp32 ``[K, N]`` dequantised weight (``out[k, n] = (code - zp) * scale``)."""
    torch = _torch()
    lib = load_library()
    w = _weight(packed, scales, zero_points)
    if out is None:
        out = torch.empty((K, N), dtype=torch.float32, device=packed.device)
    _check_dev("out", out, torch.float32)
    _raise(lib.mnb_dequant(w, K, N, block_size, _ptr(out), _stream_handle(stream)))
    return out


def mnb_repack(packed, K: int, N: int, block_size: int, out=None, stream=None):
    """uint8 repacked tensor-core operand (``mnb_repacked_bytes(K, N, bs)`` bytes)."""
    torch = _torch()
    lib = load_library()
    _check_dev("packed", packed, torch.uint8)
    if out is None:
        nbytes = mnb_repacked_bytes(K, N, block_size)
        if nbytes == 0:
            raise MnbError(MNB_ERR_INVALID_ARG, "mnb_repack: invalid shape")
        out = torch.empty(nbytes, dtype=torch.uint8, device=packed.device)
    _check_dev("out", out, torch.uint8)
    _raise(lib.mnb_repack(_ptr(packed), K, N, block_size, _ptr(out), _stream_handle(stream)))
    return out


def mnb_gemv(A, packed, scales, zero_points, K: int, N: int, block_size: int, out=None, stream=None):
    """fp16 ``[N]`` = A (fp16 ``[K]``) times the dequantised weight."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    w = _weight(packed, scales, zero_points)
    if out is None:
        out = torch.empty(N, dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_gemv(_ptr(A), w, K, N, block_size, _ptr(out), _stream_handle(stream)))
    return out


def mnb_gemm(A, packed, scales, zero_points, K: int, N: int, block_size: int, repacked=None,
             workspace=None, out=None, stream=None):
    """fp16 ``[M, N]`` = A (fp16 ``[M, K]``) times the dequantised weight."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    M = A.numel() // K
    w = _weight(packed, scales, zero_points)
    _check_dev("repacked", repacked, torch.uint8)
    need = mnb_workspace_bytes(M, K, N, block_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_gemm(_ptr(A), M, w, _ptr(repacked), K, N, block_size, _ptr(workspace), ws_bytes,
                        _ptr(out), _stream_handle(stream)))
    return out


MNB_BIAS_NONE, MNB_BIAS_FUSED, MNB_BIAS_AFTER_ROUND = 0, 1, 2


def mnb_gemm_bias(A, packed, scales, zero_points, K: int, N: int, block_size: int, bias, bias_mode: int,
                  repacked=None, workspace=None, out=None, stream=None):
    """``mnb_gemm`` plus a fp16 ``[N]`` bias: mode 1 = fp16(acc + b), mode 2 = fp16(fp16(acc) + b)."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    _check_dev("bias", bias, torch.float16)
    M = A.numel() // K
    w = _weight(packed, scales, zero_points)
    _check_dev("repacked", repacked, torch.uint8)
    need = mnb_workspace_bytes(M, K, N, block_size)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=A.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_gemm_bias(_ptr(A), M, w, _ptr(repacked), K, N, block_size, _ptr(bias), bias_mode,
                             _ptr(workspace), ws_bytes, _ptr(out), _stream_handle(stream)))
    return out


def mnb_gemv_gate_up_swiglu(A, gate, up, K: int, N: int, block_size: int, out=None, stream=None):
    """fp16 ``[N]`` = silu(A . gate^T) * (A . up^T); gate/up are (packed, scales, zero_points)."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    wg = _weight(*gate)
    wu = _weight(*up)
    if out is None:
        out = torch.empty(N, dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_gemv_gate_up_swiglu(_ptr(A), wg, wu, K, N, block_size, _ptr(out),
                                       _stream_handle(stream)))
    return out


# ---------------------------------------------------------------------------
# fp32 activations
# ---------------------------------------------------------------------------


def mnb_workspace_bytes_f32(M: int, K: int, N: int, block_size: int) -> int:
    return int(load_library().mnb_workspace_bytes_f32(M, K, N, block_size))


def mnb_gemm_f32(A, packed, scales, zero_points, K: int, N: int, block_size: int, repacked=None, bias=None,
                 workspace=None, out=None, stream=None):
    """fp32 ``[M, N]`` = A (fp32 ``[M, K]``) times the dequantised weight (+ fp32 bias ``[N]``)."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float32)
    _check_dev("bias", bias, torch.float32)
    _check_dev("repacked", repacked, torch.uint8)
    M = A.numel() // K
    w = _weight(packed, scales, zero_points)
    need = mnb_workspace_bytes_f32(M, K, N, block_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check_dev("out", out, torch.float32)
    _raise(lib.mnb_gemm_f32(_ptr(A), M, w, _ptr(repacked), K, N, block_size, _ptr(bias), _ptr(workspace),
                            ws_bytes, _ptr(out), _stream_handle(stream)))
    return out


# ---------------------------------------------------------------------------
# Act-order (g_idx) weights
# ---------------------------------------------------------------------------


def mnb_dequant_gidx(packed, scales, zero_points, g_idx, K: int, N: int, block_size: int, out=None,
                     stream=None):
    """fp32 ``[K, N]`` with the scale and zero point of group ``g_idx[k]`` at column ``k``."""
    torch = _torch()
    lib = load_library()
    w = _weight(packed, scales, zero_points)
    _check_dev("g_idx", g_idx, torch.int32)
    if out is None:
        out = torch.empty((K, N), dtype=torch.float32, device=packed.device)
    _check_dev("out", out, torch.float32)
    _raise(lib.mnb_dequant_gidx(w, _ptr(g_idx), K, N, block_size, _ptr(out), _stream_handle(stream)))
    return out


def mnb_act_order_plan(g_idx, K: int, block_size: int):
    """Host-only: ``(K_prepared, perm, block_group)`` as int / int32 numpy arrays.

    ``g_idx`` is any host int sequence of length ``K`` (numpy array, list or CPU tensor).
    """
    import numpy as np
    lib = load_library()
    g = np.ascontiguousarray(np.asarray(g_idx), dtype=np.int32).reshape(-1)
    if g.size != K:
        raise MnbError(MNB_ERR_INVALID_ARG, f"mnb_act_order_plan: g_idx has {g.size} entries, expected {K}")
    kp = ctypes.c_int32(0)
    gp = g.ctypes.data_as(ctypes.c_void_p)
    _raise(lib.mnb_act_order_plan(gp, K, block_size, ctypes.byref(kp), None, None))
    perm = np.empty(max(kp.value, 1), dtype=np.int32)
    bg = np.empty(max(kp.value // block_size, 1), dtype=np.int32)
    _raise(lib.mnb_act_order_plan(gp, K, block_size, ctypes.byref(kp), perm.ctypes.data_as(ctypes.c_void_p),
                                  bg.ctypes.data_as(ctypes.c_void_p)))
    return kp.value, perm[:kp.value], bg[:kp.value // block_size]


def mnb_act_order_prepare(packed, scales, zero_points, K: int, N: int, block_size: int, perm, block_group,
                          K_prepared: int, packed_out=None, scales_out=None, zero_points_out=None, stream=None):
    """Prepared block weight ``(packed', scales', zero_points')`` (device tensors)."""
    torch = _torch()
    lib = load_library()
    w = _weight(packed, scales, zero_points)
    _check_dev("perm", perm, torch.int32)
    _check_dev("block_group", block_group, torch.int32)
    Gp = K_prepared // block_size
    dev = packed.device
    if packed_out is None:
        packed_out = torch.empty((N, K_prepared // 2), dtype=torch.uint8, device=dev)
    if scales_out is None:
        scales_out = torch.empty((N, Gp), dtype=scales.dtype, device=dev)
    if zero_points is not None and zero_points_out is None:
        zero_points_out = torch.empty((N, (Gp + 1) // 2), dtype=torch.uint8, device=dev)
    if zero_points is None:
        zero_points_out = None
    _raise(lib.mnb_act_order_prepare(w, K, N, block_size, _ptr(perm), _ptr(block_group), K_prepared,
                                     _ptr(packed_out), _ptr(scales_out), _ptr(zero_points_out),
                                     _stream_handle(stream)))
    return packed_out, scales_out, zero_points_out


def mnb_act_order_gather(A, K: int, perm, K_prepared: int, out=None, stream=None):
    """fp16 ``[M, K']`` with ``out[m, k'] = A[m, perm[k']]`` (0 where ``perm = -1``)."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    _check_dev("perm", perm, torch.int32)
    M = A.numel() // K
    if out is None:
        out = torch.empty((M, K_prepared), dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_act_order_gather(_ptr(A), M, K, _ptr(perm), K_prepared, _ptr(out), _stream_handle(stream)))
    return out


def mnb_act_order_workspace_bytes(M: int, K_prepared: int) -> int:
    return int(load_library().mnb_act_order_workspace_bytes(M, K_prepared))


def mnb_gemm_act_order(A, packed, scales, zero_points, perm, K: int, K_prepared: int, N: int, block_size: int,
                       repacked=None, bias=None, bias_mode: int = MNB_BIAS_NONE, workspace=None, out=None,
                       stream=None):
    """fp16 ``[M, N]`` for an act-order weight; ``packed/scales/zero_points/repacked`` are the prepared ones."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    _check_dev("perm", perm, torch.int32)
    _check_dev("bias", bias, torch.float16)
    _check_dev("repacked", repacked, torch.uint8)
    M = A.numel() // K
    w = _weight(packed, scales, zero_points)
    if workspace is None:
        # the gathered activation, then room for the small-M kernel's K-slice partials
        head = (mnb_act_order_workspace_bytes(M, K_prepared) + 15) // 16 * 16
        workspace = torch.empty(head + mnb_workspace_bytes(M, K_prepared, N, block_size), dtype=torch.uint8,
                                device=A.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_gemm_act_order(_ptr(A), M, w, _ptr(repacked), _ptr(perm), K, K_prepared, N, block_size,
                                  _ptr(bias), bias_mode, _ptr(workspace), ws_bytes, _ptr(out),
                                  _stream_handle(stream)))
    return out


def mnb_gemm_act_order_noalloc(A, packed, scales, zero_points, perm, K: int, K_prepared: int, N: int,
                               block_size: int, repacked=None, bias=None, bias_mode: int = MNB_BIAS_NONE, out=None,
                               stream=None):
    """``mnb_gemm_act_order`` with the library's static scratch (M * K' * 2 <= 8 MiB) instead of a
    workspace; pass ``out`` to keep the call free of allocations."""
    torch = _torch()
    lib = load_library()
    _check_dev("A", A, torch.float16)
    _check_dev("perm", perm, torch.int32)
    _check_dev("bias", bias, torch.float16)
    _check_dev("repacked", repacked, torch.uint8)
    M = A.numel() // K
    w = _weight(packed, scales, zero_points)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_dev("out", out, torch.float16)
    _raise(lib.mnb_gemm_act_order_noalloc(_ptr(A), M, w, _ptr(repacked), _ptr(perm), K, K_prepared, N,
                                          block_size, _ptr(bias), bias_mode, _ptr(out), _stream_handle(stream)))
    return out
