"""Seeded synthetic inputs for block-quantized INT4 (MatMulNBits) products.

This module is shared by the tests, the benchmark and the smoke check.  It draws
random bytes and numbers only: it holds none of the product's arithmetic (no
nibble decoding, no dequantisation, no dot products), so neither the CUDA path
nor the fp64 oracle depends on the other through it.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based stream: element ``i``
of a tensor is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)``.  The seed of each
tensor is FNV-1a-64 of ``"<workload>/<tensor>"``.  Uniform doubles take the top
53 bits; normals come from the Box-Muller transform of consecutive pairs.

Because codes and zero-point nibbles are uniform over 0..15, a packed byte
(two nibbles) is uniform over 0..255, so packed weights and zero points are
drawn as raw random bytes.  That matches the MatMulNBits storage directly
(``packed`` is ``[N, k_blocks, block_size/2]`` bytes, ``zero_points`` is
``[N, ceil(k_blocks/2)]`` bytes) without any packing step here.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for b in text.encode("utf-8"):
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def splitmix64(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` outputs of the counter-based SplitMix64 stream, as uint64."""
    i = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, count: int) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits of each output."""
    return (splitmix64(seed, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, count: int) -> np.ndarray:
    pairs = (count + 1) // 2
    u = uniform01(seed, 2 * pairs)
    u1 = 1.0 - u[0::2]  # (0, 1], keeps log finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:count]


def random_bytes(seed: int, count: int) -> np.ndarray:
    words = splitmix64(seed, (count + 7) // 8)
    return words.astype("<u8").view(np.uint8)[:count].copy()


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MatMulNBits problem: shapes, storage dtypes and value recipes."""

    name: str
    M: int
    K: int
    N: int
    block_size: int
    scales_dtype: str          # "f16" or "f32"
    scale_lo: float
    scale_hi: float
    has_zp: bool
    act: str                   # "uniform1" (U[-1,1]), "normal", "normal_clip4"

    @property
    def k_blocks(self) -> int:
        return -(-self.K // self.block_size)

    @property
    def zp_row_bytes(self) -> int:
        return -(-self.k_blocks // 2)


def make_activation(wl: Workload, tag: str = "A", rows: int | None = None) -> np.ndarray:
    """fp16 activations ``[rows or M, K]`` drawn per the workload's recipe."""
    rows = wl.M if rows is None else rows
    seed = fnv1a64(f"{wl.name}/{tag}")
    n = rows * wl.K
    if wl.act == "uniform1":
        x = uniform01(seed, n) * 2.0 - 1.0
    elif wl.act == "normal":
        x = normal(seed, n)
    elif wl.act == "normal_clip4":
        x = np.clip(normal(seed, n), -4.0, 4.0)
    else:
        raise ValueError(wl.act)
    return x.astype(np.float16).reshape(rows, wl.K)


def make_activation_f32(wl: Workload, tag: str = "A", rows: int | None = None, recipe: str | None = None):
    """fp32 activations ``[rows or M, K]`` (not rounded to fp16).

    ``recipe`` defaults to the workload's; ``"wide"`` draws magnitudes log-uniform over
    1e-6 .. 1e6 with random signs (values far outside the fp16 range).
    """
    rows = wl.M if rows is None else rows
    recipe = wl.act if recipe is None else recipe
    seed = fnv1a64(f"{wl.name}/{tag}/f32")
    n = rows * wl.K
    if recipe == "wide":
        u = uniform01(seed, 2 * n)
        x = np.where(u[0::2] < 0.5, -1.0, 1.0) * 10.0 ** (12.0 * u[1::2] - 6.0)
    elif recipe == "uniform1":
        x = uniform01(seed, n) * 2.0 - 1.0
    elif recipe == "normal":
        x = normal(seed, n)
    elif recipe == "normal_clip4":
        x = np.clip(normal(seed, n), -4.0, 4.0)
    else:
        raise ValueError(recipe)
    return x.astype(np.float32).reshape(rows, wl.K)


@dataclasses.dataclass
class QuantWeight:
    """Host copy of one quantised weight in MatMulNBits storage."""

    packed: np.ndarray               # uint8 [N, k_blocks * block_size // 2]
    scales: np.ndarray               # float16 or float32 [N, k_blocks]
    zero_points: np.ndarray | None   # uint8 [N, zp_row_bytes] or None (zp = 8)


def make_weight(wl: Workload, tag: str = "B") -> QuantWeight:
    seed = fnv1a64(f"{wl.name}/{tag}/packed")
    blob = wl.block_size // 2
    packed = random_bytes(seed, wl.N * wl.k_blocks * blob).reshape(wl.N, wl.k_blocks * blob)
    u = uniform01(fnv1a64(f"{wl.name}/{tag}/scales"), wl.N * wl.k_blocks)
    s = wl.scale_lo + (wl.scale_hi - wl.scale_lo) * u
    sdt = np.float16 if wl.scales_dtype == "f16" else np.float32
    scales = s.astype(sdt).reshape(wl.N, wl.k_blocks)
    zp = None
    if wl.has_zp:
        zp = random_bytes(fnv1a64(f"{wl.name}/{tag}/zp"), wl.N * wl.zp_row_bytes)
        zp = zp.reshape(wl.N, wl.zp_row_bytes)
    return QuantWeight(packed=packed, scales=scales, zero_points=zp)


def make_g_idx(wl: Workload, kind: str = "act_order", tag: str = "g_idx") -> np.ndarray:
    """int32 ``[K]`` group indices, the optional act-order input of MatMulNBits.

    ``"act_order"``: the K columns are visited in a random order and each run of
    ``block_size`` consecutive visits is one group, so every group has ``block_size``
    members scattered over K (the structure act-order quantisation produces).
    ``"uneven"``: every k draws a uniform random group, so group sizes vary and some
    groups may be empty.  ``"identity"``: group ``k // block_size``, the plain layout.
    """
    seed = fnv1a64(f"{wl.name}/{tag}")
    G = wl.k_blocks
    if kind == "act_order":
        visit = np.argsort(uniform01(seed, wl.K), kind="stable")
        g = np.empty(wl.K, dtype=np.int64)
        g[visit] = np.arange(wl.K) // wl.block_size
    elif kind == "uneven":
        g = np.minimum((uniform01(seed, wl.K) * G).astype(np.int64), G - 1)
    elif kind == "identity":
        g = np.arange(wl.K) // wl.block_size
    else:
        raise ValueError(kind)
    return g.astype(np.int32)


# The five problem families this library is measured on.  Names say what they are.
WORKLOADS = {
    "tiny_gemv_k256_n128": Workload("tiny_gemv_k256_n128", 1, 256, 128, 32, "f16", 0.005, 0.02, True, "uniform1"),
    "gemv_attnproj_k4096_n4096": Workload("gemv_attnproj_k4096_n4096", 1, 4096, 4096, 32, "f16", 0.005, 0.02, True, "normal_clip4"),
    "mlp_gate_up_k4096_n14336": Workload("mlp_gate_up_k4096_n14336", 1, 4096, 14336, 128, "f32", 0.002, 0.01, False, "normal"),
    "mlp_down_k14336_n4096": Workload("mlp_down_k14336_n4096", 1, 14336, 4096, 32, "f32", 0.002, 0.01, False, "normal"),
    "verify_m2_k4096_n4096": Workload("verify_m2_k4096_n4096", 2, 4096, 4096, 64, "f16", 0.005, 0.02, True, "normal"),
    "verify_m4_k4096_n4096": Workload("verify_m4_k4096_n4096", 4, 4096, 4096, 64, "f16", 0.005, 0.02, True, "normal"),
    "verify_m8_k4096_n4096": Workload("verify_m8_k4096_n4096", 8, 4096, 4096, 64, "f16", 0.005, 0.02, True, "normal"),
    "verify_m16_k4096_n4096": Workload("verify_m16_k4096_n4096", 16, 4096, 4096, 64, "f16", 0.005, 0.02, True, "normal"),
    "prefill_m2048_k4096_n14336": Workload("prefill_m2048_k4096_n14336", 2048, 4096, 14336, 128, "f16", 0.002, 0.01, True, "normal"),
}


def custom(name: str, M: int, K: int, N: int, block_size: int, scales_dtype: str = "f16",
           has_zp: bool = True, act: str = "normal", scale_lo: float = 0.005,
           scale_hi: float = 0.02) -> Workload:
    """An ad-hoc workload (parity sweeps over ragged shapes)."""
    return Workload(name, M, K, N, block_size, scales_dtype, scale_lo, scale_hi, has_zp, act)
