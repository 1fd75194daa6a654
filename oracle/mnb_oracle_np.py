"""numpy restatement of the fp64 oracle, kept as a cross-check of the C++ oracle.

TEST INFRASTRUCTURE.  The oracle proper is ``mnb_oracle.cpp`` (loaded by
``mnb_oracle.py``); a CPU test compares the two on random inputs.  Only the tests
import this module.  The library itself never calls it, shares no code with it,
and has no CPU fallback.

What it computes is a plain definition, written out directly:

    Y[m, n] = sum_k A[m, k] * (code[n, k] - zp[n, k // bs]) * scale[n, k // bs]

with the weight stored in the ONNX ``com.microsoft::MatMulNBits`` layout.
Sources:

* onnx-runtime-ep-cuda 0.1.0-dev.6, ``src/kernels/marlin_gemm.rs``, module doc,
  section "ONNX MatMulNBits int4 format": the packed ``[N, k_blocks, bs/2]``
  byte layout, the low nibble holding the even ``k``, ``[N, k_blocks]`` scales
  in fp16 or fp32, nibble-packed zero points with ``ceil(k_blocks/2)`` bytes
  per row, low nibble for the even block, and the default zero point 8.
* onnx-runtime-ep-cuda 0.1.0-dev.3, ``src/kernels/matmul_nbits.rs``, kernel
  ``matmul_nbits_dequant_f32``: ``k_blocks = ceil(K/bs)``, the element
  ``(code - zp) * scale`` written to a ``[K, N]`` fp32 matrix indexed
  ``depth * N + n``.

Arithmetic is fp64.  Every quantity on the right-hand side is exact in fp64:
codes and zero points are small integers, fp16 and fp32 scales widen exactly,
and ``(code - zp) * scale`` has at most 4 + 24 significant bits.  The only
rounding in ``Y`` is the fp64 summation (done by a BLAS matmul, a library
primitive), far below the fp16 output precision.

The bound ``B[m, n] = sum_k |A[m, k] * w[n, k]|`` is returned with ``Y``; a
device result ``y`` agrees when ``|y - Y| <= 2e-3 * B + 1e-5``.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Storage decoding (layout only, integers)
# ---------------------------------------------------------------------------


def k_blocks(K: int, block_size: int) -> int:
    """Groups per weight row: ``ceil(K / block_size)`` (matmul_nbits.rs, attribute parsing)."""
    return -(-K // block_size)


def zp_row_bytes(K: int, block_size: int) -> int:
    """Zero-point bytes per row: ``ceil(k_blocks / 2)`` (marlin_gemm.rs module doc)."""
    return -(-k_blocks(K, block_size) // 2)


def codes(packed: np.ndarray, K: int, N: int, block_size: int) -> np.ndarray:
    """int64 ``[N, K]`` codes in 0..15.

    The byte for ``(n, k)`` sits at ``(n * k_blocks + k // bs) * (bs / 2) + (k % bs) / 2``;
    with ``within = k % bs``, an even ``within`` takes the low nibble and an odd one the
    high nibble (``matmul_nbits_dequant_f32``; marlin_gemm.rs module doc).  Positions of a
    partial last block beyond ``K`` are never read.
    """
    G = k_blocks(K, block_size)
    blob = block_size // 2
    flat = np.ascontiguousarray(packed).reshape(-1)
    if flat.size != N * G * blob:
        raise ValueError(f"packed has {flat.size} bytes, expected {N * G * blob}")
    n = np.arange(N, dtype=np.int64)[:, None]
    k = np.arange(K, dtype=np.int64)[None, :]
    block = k // block_size
    within = k - block * block_size
    byte = flat[(n * G + block) * blob + within // 2].astype(np.int64)
    return np.where((within & 1) == 1, byte >> 4, byte & 15)


def zero_points(zp: np.ndarray | None, K: int, N: int, block_size: int) -> np.ndarray:
    """int64 ``[N, k_blocks]`` zero points.

    ``None`` means the symmetric default 8.  Otherwise the nibble for ``(n, g)`` is in
    byte ``zp[n * zp_row_bytes + g / 2]``: low nibble for even ``g``, high for odd ``g``.
    """
    G = k_blocks(K, block_size)
    if zp is None:
        return np.full((N, G), 8, dtype=np.int64)
    zrb = zp_row_bytes(K, block_size)
    flat = np.ascontiguousarray(zp).reshape(-1)
    if flat.size != N * zrb:
        raise ValueError(f"zero_points has {flat.size} bytes, expected {N * zrb}")
    n = np.arange(N, dtype=np.int64)[:, None]
    g = np.arange(G, dtype=np.int64)[None, :]
    byte = flat[n * zrb + g // 2].astype(np.int64)
    return np.where((g & 1) == 1, byte >> 4, byte & 15)


def f16_to_f64(h: np.ndarray) -> np.ndarray:
    """Exact value of IEEE-754 binary16 numbers, decoded from their bits.

    Normal: (-1)^s * 2^(e-15) * (1 + m/1024); subnormal (e = 0): (-1)^s * 2^-14 * m/1024;
    e = 31: infinity (m = 0) or NaN.
    """
    bits = np.ascontiguousarray(h).view(np.uint16).astype(np.int64)
    sign = np.where(bits >> 15 == 1, -1.0, 1.0)
    e = (bits >> 10) & 0x1F
    m = (bits & 0x3FF).astype(np.float64)
    normal = np.ldexp(1.0 + m / 1024.0, (e - 15).astype(np.int32))
    sub = np.ldexp(m / 1024.0, -14)
    special = np.where(m == 0, np.inf, np.nan)
    val = np.where(e == 0, sub, np.where(e == 31, special, normal))
    return sign * val


def scales_f64(scales: np.ndarray, K: int, N: int, block_size: int) -> np.ndarray:
    """``[N, k_blocks]`` scales as exact fp64 (fp16 or fp32 storage)."""
    G = k_blocks(K, block_size)
    s = np.ascontiguousarray(scales).reshape(-1)
    if s.size != N * G:
        raise ValueError(f"scales has {s.size} values, expected {N * G}")
    if s.dtype == np.float16:
        out = f16_to_f64(s)
    elif s.dtype == np.float32:
        out = s.astype(np.float64)
    else:
        raise TypeError(f"scales must be float16 or float32, got {s.dtype}")
    return out.reshape(N, G)


# ---------------------------------------------------------------------------
# The product
# ---------------------------------------------------------------------------


def groups(K: int, block_size: int, g_idx=None) -> np.ndarray:
    """int64 ``[K]``: the group whose scale and zero point apply at each ``k``.

    Without ``g_idx`` it is the block ``k // bs``.  With the act-order input ``g_idx``
    (int32 ``[K]`` or ``[k_blocks * bs]``; entries past ``K`` are never read) it is
    ``g_idx[k]`` (``matmul_nbits_dequant_f32``: ``group = group_indices[depth]``).  The
    code itself is always read from block ``k // bs``.
    """
    if g_idx is None:
        return np.arange(K, dtype=np.int64) // block_size
    g = np.asarray(g_idx).reshape(-1).astype(np.int64)
    if g.size not in (K, k_blocks(K, block_size) * block_size):
        raise ValueError(f"g_idx has {g.size} entries, expected {K} or the padded K")
    return g[:K]


def weight_nk(packed, scales, zp, K: int, N: int, block_size: int, g_idx=None) -> np.ndarray:
    """Exact fp64 ``w[n, k] = (code[n, k] - zp[n, g]) * scale[n, g]``, ``g = groups(k)``.

    A group outside ``0 .. k_blocks-1`` gives ``w = 0`` (``matmul_nbits_dequant_f32``
    writes 0 for it; the operator's host check rejects such a ``g_idx`` outright).
    """
    c = codes(packed, K, N, block_size)
    z = zero_points(zp, K, N, block_size)
    s = scales_f64(scales, K, N, block_size)
    g = groups(K, block_size, g_idx)
    ok = (g >= 0) & (g < k_blocks(K, block_size))
    gc = np.where(ok, g, 0)
    w = (c - z[:, gc]).astype(np.float64) * s[:, gc]
    return np.where(ok[None, :], w, 0.0)


def dequant_kn_f32(packed, scales, zp, K: int, N: int, block_size: int, g_idx=None) -> np.ndarray:
    """fp32 ``[K, N]``: each element is ``(code - zp) * scale`` rounded once to fp32.

    ``matmul_nbits_dequant_f32`` writes this matrix at ``depth * N + n``.  The fp64
    product is exact, so one rounding gives the correctly rounded fp32 product; for
    fp16 scales the product is already representable in fp32 and the value is exact.
    """
    return weight_nk(packed, scales, zp, K, N, block_size, g_idx).T.astype(np.float32)


def activations_f64(A: np.ndarray) -> np.ndarray:
    """Exact fp64 value of fp16 activations (decoded from their bits) or fp32 ones
    (the operator's fp32 path, matmul_nbits.rs: A of type Float32, widened exactly)."""
    if A.dtype == np.float16:
        return f16_to_f64(A).reshape(A.shape)
    if A.dtype == np.float32:
        return A.astype(np.float64)
    raise TypeError(f"activations are fp16 or fp32, got {A.dtype}")


def matmul(A, packed, scales, zp, K: int, N: int, block_size: int, g_idx=None):
    """``(Y, B)``: fp64 ``Y = A . w^T`` and the bound ``B = |A| . |w|^T``, both ``[M, N]``.

    ``A`` is the fp16 activation ``[M, K]`` (taken at its fp16 value, as the pages'
    oracles consume the same fp16-rounded activations as the kernel).  ``g_idx``: see
    ``groups``.
    """
    a = activations_f64(A).reshape(-1, K)
    w = weight_nk(packed, scales, zp, K, N, block_size, g_idx)
    return a @ w.T, np.abs(a) @ np.abs(w).T


def matmul_rows(A, packed, scales, zp, K: int, N: int, block_size: int, rows, cols, g_idx=None):
    """``(Y, B)`` at the listed ``(row, col)`` pairs only (full-size spot checks)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a = activations_f64(A).reshape(-1, K)
    ucols, inv = np.unique(cols, return_inverse=True)
    G = k_blocks(K, block_size)
    blob = block_size // 2
    sub_packed = np.ascontiguousarray(packed).reshape(N, G * blob)[ucols]
    sub_scales = np.ascontiguousarray(scales).reshape(N, G)[ucols]
    sub_zp = None if zp is None else np.ascontiguousarray(zp).reshape(N, -1)[ucols]
    w = weight_nk(sub_packed, sub_scales, sub_zp, K, len(ucols), block_size, g_idx)
    ar = a[rows]
    wc = w[inv]
    return np.einsum("ik,ik->i", ar, wc), np.einsum("ik,ik->i", np.abs(ar), np.abs(wc))


def silu(x: np.ndarray) -> np.ndarray:
    """``x / (1 + exp(-x))`` in fp64."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def gate_up_swiglu(A, gate, up, K: int, N: int, block_size: int):
    """``(out, g, Bg, u, Bu)`` with ``out = silu(g) * u`` (paired gate/up projection).

    ``gate`` and ``up`` are ``(packed, scales, zero_points)`` triples sharing ``K, N, bs``.
    Follows ``matmul_nbits_gemv_f16_gate_up_swiglu`` (matmul_nbits.rs): two projections
    of one activation, then ``silu(gate) * up`` per output column.
    """
    g, bg = matmul(A, *gate, K, N, block_size)
    u, bu = matmul(A, *up, K, N, block_size)
    return silu(g) * u, g, bg, u, bu


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
# The repacked tensor-core operand layout
# ---------------------------------------------------------------------------
#
# This layout is this library's own (the pages repack for mma.sync fragments; the
# layout here is built for 1-D bulk copies and shared-memory dequantisation):
#
#   Np = ceil(N / 128) * 128, Kp = ceil(K / 64) * 64, size = Np * Kp / 2 bytes.
#   Tile t (128 rows) and k-block b (64 k) form one 4096-byte block at byte
#   (t * (Kp / 64) + b) * 4096.  Inside it, the 16 bytes at q * 2048 + r * 16
#   (q in 0..1, r in 0..127) hold the 32 codes of row n = 128 t + r for
#   k = 64 b + 32 q + i, i in 0..31.  Those 16 bytes are four little-endian 32-bit
#   words; word j = i // 8 holds i at nibble position p (bits 4p..4p+3) where
#   i = 8 j + 2 (p % 4) + p // 4.  Codes for n >= N or k >= K are 0.
#
# Nothing here is shared with the device code; this is an independent restatement
# of the same specification.

REPACK_TILE_N = 128
REPACK_TILE_K = 64


def repacked_bytes(K: int, N: int) -> int:
    np_ = -(-N // REPACK_TILE_N) * REPACK_TILE_N
    kp = -(-K // REPACK_TILE_K) * REPACK_TILE_K
    return np_ * kp // 2


def _repack_positions(K: int, N: int):
    """For every (n, k): destination byte and nibble half (0 low, 1 high)."""
    kp = -(-K // REPACK_TILE_K) * REPACK_TILE_K
    n = np.arange(N, dtype=np.int64)[:, None]
    k = np.arange(K, dtype=np.int64)[None, :]
    t, r = n // REPACK_TILE_N, n % REPACK_TILE_N
    b, kk = k // REPACK_TILE_K, k % REPACK_TILE_K
    q, i = kk // 32, kk % 32
    j, i8 = i // 8, i % 8
    # invert i8 = 2 (p % 4) + p // 4
    p = (i8 // 2) + 4 * (i8 % 2)
    byte = (t * (kp // REPACK_TILE_K) + b) * 4096 + q * 2048 + r * 16 + 4 * j + p // 2
    return byte, np.broadcast_to(p % 2, byte.shape)


def repack(packed, K: int, N: int, block_size: int) -> np.ndarray:
    """uint8 repacked buffer of ``repacked_bytes(K, N)`` bytes."""
    c = codes(packed, K, N, block_size)
    byte, half = _repack_positions(K, N)
    out = np.zeros(repacked_bytes(K, N), dtype=np.uint8)
    lo = half == 0
    out[byte[lo]] |= c[lo].astype(np.uint8)
    out[byte[~lo]] |= (c[~lo] << 4).astype(np.uint8)
    return out


def unrepack_codes(repacked: np.ndarray, K: int, N: int) -> np.ndarray:
    """int64 ``[N, K]`` codes read back from a repacked buffer."""
    byte, half = _repack_positions(K, N)
    v = np.asarray(repacked).reshape(-1)[byte].astype(np.int64)
    return np.where(half == 1, v >> 4, v & 15)


# ---------------------------------------------------------------------------
# Act-order weights prepared for the block kernels
# ---------------------------------------------------------------------------
#
# With ``g_idx`` the members of a group are scattered over K.  Reordering k so that
# each group's members sit together turns the weight into a plain block weight:
#
#   * groups in ascending order; inside a group, its members in ascending k;
#   * each group's run padded with empty slots (-1) to a whole number of blocks;
#   * ``perm[k']`` = the source k of prepared position k' (or -1), ``K' = len(perm)``,
#     ``block_group[j]`` = the group of prepared block j.
#
# The prepared weight has codes ``code[n, perm[k']]`` (the block's zero point at an
# empty slot, so its weight is 0), and the scale and zero point of ``block_group[j]``
# for block j.  The matching activation is ``A'[m, k'] = A[m, perm[k']]`` (0 at an
# empty slot), and ``A' . w'^T = A . w^T`` term by term.  This preparation is this
# library's own; the pages dequantise with ``g_idx`` directly.


def act_order_plan(g_idx, K: int, block_size: int):
    """``(K_prepared, perm, block_group)`` for a valid ``g_idx`` (int32 arrays).

    Raises ``ValueError`` for an entry outside ``0 .. k_blocks-1`` (the operator's own
    check on ``g_idx``, matmul_nbits.rs).
    """
    G = k_blocks(K, block_size)
    g = groups(K, block_size, g_idx)
    bad = np.nonzero((g < 0) | (g >= G))[0]
    if bad.size:
        raise ValueError(f"g_idx[{bad[0]}]={g[bad[0]]} is outside 0..{G}")
    perm, block_group = [], []
    for grp in range(G):
        members = np.nonzero(g == grp)[0].tolist()
        nblocks = -(-len(members) // block_size)
        perm += members + [-1] * (nblocks * block_size - len(members))
        block_group += [grp] * nblocks
    return len(perm), np.array(perm, dtype=np.int32), np.array(block_group, dtype=np.int32)


def _pack_nibbles(v: np.ndarray) -> np.ndarray:
    """uint8 rows from int rows of 4-bit values: low nibble from the even position."""
    v = np.asarray(v, dtype=np.int64)
    if v.shape[1] % 2:
        v = np.concatenate([v, np.zeros((v.shape[0], 1), dtype=np.int64)], axis=1)
    return (v[:, 0::2] | (v[:, 1::2] << 4)).astype(np.uint8)


def act_order_prepare(packed, scales, zp, K: int, N: int, block_size: int, perm, block_group):
    """``(packed', scales', zero_points')`` of the prepared ``K' x N`` block weight.

    ``packed'`` is uint8 ``[N, K'/2]``, ``scales'`` keeps the scale dtype
    ``[N, K'/bs]``, ``zero_points'`` is uint8 ``[N, ceil(K'/bs/2)]`` (the unused high
    nibble of an odd count is 0), or ``None`` when the weight has none.
    """
    perm = np.asarray(perm, dtype=np.int64)
    bg = np.asarray(block_group, dtype=np.int64)
    Kp = perm.size
    if Kp % block_size or bg.size != Kp // block_size:
        raise ValueError("perm and block_group do not describe whole blocks")
    c = codes(packed, K, N, block_size)
    z = zero_points(zp, K, N, block_size)
    zb = z[:, bg]                                         # [N, K'/bs]
    zk = zb[:, np.arange(Kp) // block_size]               # [N, K']
    cp = np.where(perm[None, :] >= 0, c[:, np.maximum(perm, 0)], zk)
    G = k_blocks(K, block_size)
    sp = np.ascontiguousarray(scales).reshape(N, G)[:, bg].copy()
    zpp = None if zp is None else _pack_nibbles(zb)
    return _pack_nibbles(cp), sp, zpp


def act_order_gather(A, perm) -> np.ndarray:
    """fp16 ``A'[m, k'] = A[m, perm[k']]``, and +0 where ``perm[k'] = -1``."""
    A = np.asarray(A)
    perm = np.asarray(perm, dtype=np.int64)
    out = np.zeros((A.shape[0], perm.size), dtype=A.dtype)
    ok = perm >= 0
    out[:, ok] = A[:, perm[ok]]
    return out
