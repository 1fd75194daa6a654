"""fp64 CPU oracle for block-quantized INT4 (MatMulNBits) products.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg import this module.  The library itself never calls it, shares no
code with it, and has no CPU fallback.

The arithmetic is plain C++ with fp64 loops (``oracle/mnb_oracle.cpp``, built by
``build_native`` with g++ into ``oracle/libmnb_oracle.so``); this module only
marshals numpy arrays to it and shapes the results.  What it computes:

    Y[m, n] = sum_k A[m, k] * (code[n, k] - zp[n, g(k)]) * scale[n, g(k)]

for a weight in the ONNX ``com.microsoft::MatMulNBits`` layout (onnx-runtime-ep-cuda
0.1.0-dev.6, ``src/kernels/marlin_gemm.rs``, module doc, section "ONNX MatMulNBits
int4 format"; onnx-runtime-ep-cuda 0.1.0-dev.3, ``src/kernels/matmul_nbits.rs``,
kernel ``matmul_nbits_dequant_f32``), summed in ascending ``k``, together with the
bound ``B[m, n] = sum_k |A[m, k] * w[n, k]|``; a device result ``y`` agrees when
``|y - Y| <= 2e-3 * B + 1e-5``.

The products split their output columns over the host's CPUs
(``os.sched_getaffinity``); each output is still one ascending-k sum, so the
thread count changes no result.  ``oracle/mnb_oracle_np.py`` is an earlier numpy
restatement of the same definition, kept as a cross-check.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "mnb_oracle.cpp")
_LIB_PATH = os.path.join(_DIR, "libmnb_oracle.so")
_CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]
_lock = threading.Lock()
_lib = None


def build_native(force: bool = False) -> str:
    """Compile ``mnb_oracle.cpp`` into ``libmnb_oracle.so`` when it is missing or older
    than its source (g++; the same flags on x86-64 and AArch64)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cxx = os.environ.get("CXX", "g++")
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    r = subprocess.run([cxx, *_CXXFLAGS, _SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_LL = ctypes.c_longlong
_I = ctypes.c_int
_SIGS = {
    "orc_k_blocks": (_LL, [_LL, _LL]),
    "orc_zp_row_bytes": (_LL, [_LL, _LL]),
    "orc_codes": (None, [_P, _LL, _LL, _LL, _P]),
    "orc_zero_points": (None, [_P, _LL, _LL, _LL, _P]),
    "orc_f16_to_f64": (None, [_P, _LL, _P]),
    "orc_weight_nk": (None, [_P, _P, _I, _P, _P, _LL, _LL, _LL, _P, _I]),
    "orc_dequant_kn_f32": (None, [_P, _P, _I, _P, _P, _LL, _LL, _LL, _P, _I]),
    "orc_matmul": (None, [_P, _I, _LL, _P, _P, _I, _P, _P, _LL, _LL, _LL, _P, _P, _I]),
    "orc_matmul_pairs": (None, [_P, _I, _P, _P, _I, _P, _P, _LL, _LL, _LL, _P, _P, _LL, _P, _P, _I]),
    "orc_silu": (None, [_P, _LL, _P]),
    "orc_swiglu": (None, [_P, _P, _LL, _P]),
    "orc_repacked_bytes": (_LL, [_LL, _LL]),
    "orc_repack": (None, [_P, _LL, _LL, _LL, _P]),
    "orc_unrepack_codes": (None, [_P, _LL, _LL, _P]),
    "orc_act_order_plan": (_LL, [_P, _LL, _LL, _P, _P, _P]),
    "orc_act_order_prepare": (None, [_P, _P, _I, _P, _LL, _LL, _LL, _P, _P, _LL, _P, _P, _P]),
    "orc_act_order_gather": (None, [_P, _LL, _LL, _I, _P, _LL, _P]),
}


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            build_native()
            h = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def threads() -> int:
    """CPUs this process may run on (the oracle's thread count for the products)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(a, count, what):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"{what} must be uint8, got {a.dtype}")
    if a.size != count:
        raise ValueError(f"{what} has {a.size} bytes, expected {count}")
    return a.reshape(-1)


# ---------------------------------------------------------------------------
# Storage decoding (layout only, integers)
# ---------------------------------------------------------------------------


def k_blocks(K: int, block_size: int) -> int:
    """Groups per weight row: ``ceil(K / block_size)``."""
    return int(lib().orc_k_blocks(K, block_size))


def zp_row_bytes(K: int, block_size: int) -> int:
    """Zero-point bytes per row: ``ceil(k_blocks / 2)``."""
    return int(lib().orc_zp_row_bytes(K, block_size))


def _packed(packed, K, N, block_size):
    return _u8(packed, N * k_blocks(K, block_size) * (block_size // 2), "packed")


def _zp(zp, K, N, block_size):
    return None if zp is None else _u8(zp, N * zp_row_bytes(K, block_size), "zero_points")


def _scales(scales, K, N, block_size):
    s = np.ascontiguousarray(scales).reshape(-1)
    G = k_blocks(K, block_size)
    if s.size != N * G:
        raise ValueError(f"scales has {s.size} values, expected {N * G}")
    if s.dtype == np.float16:
        return s, 1
    if s.dtype == np.float32:
        return s, 0
    raise TypeError(f"scales must be float16 or float32, got {s.dtype}")


def _g_idx(g_idx, K, block_size):
    """int32 ``[K]`` act-order groups (``[K]`` or ``[k_blocks * bs]`` accepted; entries past
    ``K`` are never read), or None."""
    if g_idx is None:
        return None
    g = np.asarray(g_idx).reshape(-1)
    if g.size not in (K, k_blocks(K, block_size) * block_size):
        raise ValueError(f"g_idx has {g.size} entries, expected {K} or the padded K")
    return np.ascontiguousarray(g[:K].astype(np.int32))


def codes(packed, K: int, N: int, block_size: int) -> np.ndarray:
    """int64 ``[N, K]`` codes in 0..15 (low nibble for the even ``k`` of a block)."""
    p = _packed(packed, K, N, block_size)
    out = np.empty((N, K), dtype=np.int8)
    lib().orc_codes(_ptr(p), K, N, block_size, _ptr(out))
    return out.astype(np.int64)


def zero_points(zp, K: int, N: int, block_size: int) -> np.ndarray:
    """int64 ``[N, k_blocks]`` zero points; ``None`` means the symmetric default 8."""
    z = _zp(zp, K, N, block_size)
    out = np.empty((N, k_blocks(K, block_size)), dtype=np.int8)
    lib().orc_zero_points(_ptr(z), K, N, block_size, _ptr(out))
    return out.astype(np.int64)


def f16_to_f64(h) -> np.ndarray:
    """Exact fp64 value of IEEE-754 binary16 numbers, decoded from their bits."""
    h = np.ascontiguousarray(h)
    bits = h.view(np.uint16).reshape(-1)
    out = np.empty(bits.size, dtype=np.float64)
    lib().orc_f16_to_f64(_ptr(bits), bits.size, _ptr(out))
    return out.reshape(h.shape)


def activations_f64(A) -> np.ndarray:
    """Exact fp64 value of fp16 activations (decoded from their bits) or fp32 ones
    (the operator's fp32 path, matmul_nbits.rs: A of type Float32, widened exactly)."""
    A = np.asarray(A)
    if A.dtype == np.float16:
        return f16_to_f64(A)
    if A.dtype == np.float32:
        return A.astype(np.float64)
    raise TypeError(f"activations are fp16 or fp32, got {A.dtype}")


def scales_f64(scales, K: int, N: int, block_size: int) -> np.ndarray:
    """``[N, k_blocks]`` scales as exact fp64 (fp16 or fp32 storage)."""
    s, f16 = _scales(scales, K, N, block_size)
    return (f16_to_f64(s) if f16 else s.astype(np.float64)).reshape(N, k_blocks(K, block_size))


# ---------------------------------------------------------------------------
# Weights and products
# ---------------------------------------------------------------------------


def weight_nk(packed, scales, zp, K: int, N: int, block_size: int, g_idx=None) -> np.ndarray:
    """Exact fp64 ``w[n, k] = (code[n, k] - zp[n, g]) * scale[n, g]``, ``g = g_idx[k]`` with
    act-order indices, else ``k // bs``; a group outside ``0 .. k_blocks-1`` gives 0."""
    p = _packed(packed, K, N, block_size)
    s, f16 = _scales(scales, K, N, block_size)
    z = _zp(zp, K, N, block_size)
    g = _g_idx(g_idx, K, block_size)
    out = np.empty((N, K), dtype=np.float64)
    lib().orc_weight_nk(_ptr(p), _ptr(s), f16, _ptr(z), _ptr(g), K, N, block_size, _ptr(out), threads())
    return out


def dequant_kn_f32(packed, scales, zp, K: int, N: int, block_size: int, g_idx=None) -> np.ndarray:
    """fp32 ``[K, N]``: each element is ``(code - zp) * scale`` rounded once to fp32,
    at ``depth * N + n`` as ``matmul_nbits_dequant_f32`` writes it."""
    p = _packed(packed, K, N, block_size)
    s, f16 = _scales(scales, K, N, block_size)
    z = _zp(zp, K, N, block_size)
    g = _g_idx(g_idx, K, block_size)
    out = np.empty((K, N), dtype=np.float32)
    lib().orc_dequant_kn_f32(_ptr(p), _ptr(s), f16, _ptr(z), _ptr(g), K, N, block_size, _ptr(out), threads())
    return out


def _acts(A, K):
    A = np.ascontiguousarray(A)
    if A.dtype == np.float16:
        a_f16 = 1
    elif A.dtype == np.float32:
        a_f16 = 0
    else:
        raise TypeError(f"activations are fp16 or fp32, got {A.dtype}")
    if A.size % K:
        raise ValueError(f"activations have {A.size} values, not a multiple of K = {K}")
    return A.reshape(-1, K), a_f16


def matmul(A, packed, scales, zp, K: int, N: int, block_size: int, g_idx=None, nthreads: int | None = None):
    """``(Y, B)``: fp64 ``Y = A . w^T`` and the bound ``B = |A| . |w|^T``, both ``[M, N]``.

    ``A`` is the fp16 (or fp32) activation ``[M, K]``, taken at its exact value (the pages'
    oracles consume the same fp16-rounded activations as the kernel).
    """
    a, a_f16 = _acts(A, K)
    M = a.shape[0]
    p = _packed(packed, K, N, block_size)
    s, f16 = _scales(scales, K, N, block_size)
    z = _zp(zp, K, N, block_size)
    g = _g_idx(g_idx, K, block_size)
    Y = np.empty((M, N), dtype=np.float64)
    B = np.empty((M, N), dtype=np.float64)
    lib().orc_matmul(_ptr(a), a_f16, M, _ptr(p), _ptr(s), f16, _ptr(z), _ptr(g), K, N, block_size,
                     _ptr(Y), _ptr(B), nthreads or threads())
    return Y, B


def matmul_rows(A, packed, scales, zp, K: int, N: int, block_size: int, rows, cols, g_idx=None):
    """``(Y, B)`` at the listed ``(rows[i], cols[i])`` pairs only (1-D, one per pair)."""
    a, a_f16 = _acts(A, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64).reshape(-1))
    if rows.size != cols.size:
        raise ValueError("rows and cols differ in length")
    if rows.size and (rows.min() < 0 or rows.max() >= a.shape[0] or cols.min() < 0 or cols.max() >= N):
        raise ValueError("a (row, col) pair is outside the output")
    p = _packed(packed, K, N, block_size)
    s, f16 = _scales(scales, K, N, block_size)
    z = _zp(zp, K, N, block_size)
    g = _g_idx(g_idx, K, block_size)
    Y = np.empty(rows.size, dtype=np.float64)
    B = np.empty(rows.size, dtype=np.float64)
    lib().orc_matmul_pairs(_ptr(a), a_f16, _ptr(p), _ptr(s), f16, _ptr(z), _ptr(g), K, N, block_size,
                           _ptr(rows), _ptr(cols), rows.size, _ptr(Y), _ptr(B), threads())
    return Y, B


def silu(x) -> np.ndarray:
    """``x / (1 + exp(-x))`` in fp64."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(x)
    lib().orc_silu(_ptr(x), x.size, _ptr(out))
    return out


def gate_up_swiglu(A, gate, up, K: int, N: int, block_size: int):
    """``(out, g, Bg, u, Bu)`` with ``out = silu(g) * u`` (paired gate/up projection).

    ``gate`` and ``up`` are ``(packed, scales, zero_points)`` triples sharing ``K, N, bs``.
    Follows ``matmul_nbits_gemv_f16_gate_up_swiglu`` (matmul_nbits.rs): two projections
    of one activation, then ``silu(gate) * up`` per output column.
    """
    g, bg = matmul(A, *gate, K, N, block_size)
    u, bu = matmul(A, *up, K, N, block_size)
    out = np.empty_like(g)
    lib().orc_swiglu(_ptr(g), _ptr(u), g.size, _ptr(out))
    return out, g, bg, u, bu


def swiglu_tolerance(g, bg, u, bu, out_ref):
    """Per-element tolerance for the fused SwiGLU output.

    The pages state none.  The projections each carry the product tolerance
    ``eps = 2e-3 * B + 1e-5``; it propagates through ``silu(g) * u`` with
    ``|silu'| <= 1.1`` and adds one fp16 rounding of the result (2^-10 covers the
    rounding of an intermediate and of the store).
    """
    eg = 2e-3 * bg + 1e-5
    eu = 2e-3 * bu + 1e-5
    sg = silu(g)
    return 1.1 * np.abs(u) * eg + np.abs(sg) * eu + eg * eu * 1.1 + 2.0 ** -10 * np.abs(out_ref) + 1e-5


# ---------------------------------------------------------------------------
# The repacked tensor-core operand layout (specification in mnb_oracle.cpp)
# ---------------------------------------------------------------------------


def repacked_bytes(K: int, N: int) -> int:
    return int(lib().orc_repacked_bytes(K, N))


def repack(packed, K: int, N: int, block_size: int) -> np.ndarray:
    """uint8 repacked buffer of ``repacked_bytes(K, N)`` bytes."""
    p = _packed(packed, K, N, block_size)
    out = np.empty(repacked_bytes(K, N), dtype=np.uint8)
    lib().orc_repack(_ptr(p), K, N, block_size, _ptr(out))
    return out


def unrepack_codes(repacked, K: int, N: int) -> np.ndarray:
    """int64 ``[N, K]`` codes read back from a repacked buffer."""
    r = _u8(repacked, repacked_bytes(K, N), "repacked")
    out = np.empty((N, K), dtype=np.int8)
    lib().orc_unrepack_codes(_ptr(r), K, N, _ptr(out))
    return out.astype(np.int64)


# ---------------------------------------------------------------------------
# Act-order weights prepared for the block kernels (plan in mnb_oracle.cpp)
# ---------------------------------------------------------------------------


def act_order_plan(g_idx, K: int, block_size: int):
    """``(K_prepared, perm, block_group)`` for a valid ``g_idx`` (int32 arrays).

    Raises ``ValueError`` for an entry outside ``0 .. k_blocks-1`` (the operator's own
    check on ``g_idx``, matmul_nbits.rs).
    """
    g = _g_idx(g_idx, K, block_size)
    G = k_blocks(K, block_size)
    cap = K + G * (block_size - 1)
    perm = np.empty(cap, dtype=np.int32)
    bg = np.empty(cap // block_size + 1, dtype=np.int32)
    bad = ctypes.c_longlong(-1)
    kp = int(lib().orc_act_order_plan(_ptr(g), K, block_size, _ptr(perm), _ptr(bg), ctypes.byref(bad)))
    if kp < 0:
        raise ValueError(f"g_idx[{bad.value}]={int(g[bad.value])} is outside 0..{G}")
    return kp, perm[:kp].copy(), bg[: kp // block_size].copy()


def act_order_prepare(packed, scales, zp, K: int, N: int, block_size: int, perm, block_group):
    """``(packed', scales', zero_points')`` of the prepared ``K' x N`` block weight.

    ``packed'`` is uint8 ``[N, K'/2]``, ``scales'`` keeps the scale dtype
    ``[N, K'/bs]``, ``zero_points'`` is uint8 ``[N, ceil(K'/bs/2)]`` (the unused high
    nibble of an odd count is 0), or ``None`` when the weight has none.
    """
    perm = np.ascontiguousarray(np.asarray(perm, dtype=np.int32).reshape(-1))
    bg = np.ascontiguousarray(np.asarray(block_group, dtype=np.int32).reshape(-1))
    Kp = perm.size
    if Kp % block_size or bg.size != Kp // block_size:
        raise ValueError("perm and block_group do not describe whole blocks")
    p = _packed(packed, K, N, block_size)
    s, _ = _scales(scales, K, N, block_size)
    z = _zp(zp, K, N, block_size)
    Gp = Kp // block_size
    pk = np.empty((N, Kp // 2), dtype=np.uint8)
    sp = np.empty((N, Gp), dtype=s.dtype)
    zpp = None if z is None else np.empty((N, (Gp + 1) // 2), dtype=np.uint8)
    lib().orc_act_order_prepare(_ptr(p), _ptr(s), s.itemsize, _ptr(z), K, N, block_size, _ptr(perm), _ptr(bg), Kp,
                                _ptr(pk), _ptr(sp), _ptr(zpp))
    return pk, sp, zpp


def act_order_gather(A, perm) -> np.ndarray:
    """``A'[m, k'] = A[m, perm[k']]``, and +0 where ``perm[k'] = -1`` (same dtype as A)."""
    A = np.ascontiguousarray(A)
    if A.ndim == 1:
        A = A.reshape(1, -1)
    perm = np.ascontiguousarray(np.asarray(perm, dtype=np.int32).reshape(-1))
    M, K = A.shape
    if perm.size and perm.max() >= K:
        raise ValueError("perm names a column past K")
    out = np.empty((M, perm.size), dtype=A.dtype)
    lib().orc_act_order_gather(_ptr(A), M, K, A.itemsize, _ptr(perm), perm.size, _ptr(out))
    return out
