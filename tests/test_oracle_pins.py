"""Pins for the fp64 oracle (C++ loops in oracle/mnb_oracle.cpp, loaded through
oracle/mnb_oracle.py): each checks it against something other than itself.

* a hand-decoded worked example of the storage (tests/golden),
* single-hot brute force on every block size (pins the (n, k) -> byte/nibble map),
* a second reading of the layout, from the fp16 GEMV kernel's 32-bit word loads,
* exact rational brute force on a tiny problem,
* the integer special case (zp 0, scale 1, integer activations) against int64 matmul,
* invariants: all codes equal to the zero point give Y = 0; scale linearity;
  the default zero point 8 equals an explicit 0x88 buffer,
* fp16 decoding against numpy's own conversion for all 65536 bit patterns,
* silu against ``x * scipy.special.expit(x)``,
* the repacked layout: a hand-placed code, and the round trip,
* fp32 activations are taken at their exact value (rational brute force with values
  that fp16 cannot hold),
* act-order ``g_idx``: the identity reduces to the plain layout; a weight built the
  act-order way (codes quantised in a visit order, stored in k order) dequantises to
  the same matrix; exact rational brute force with uneven and out-of-range groups;
  a hand-worked preparation plan; the prepared weight holds the same weights,
* the spot-check product at (row, col) pairs equals the full product there, with
  repeated and unsorted pairs, act-order groups and fp32 activations,
* the thread count changes no result,
* the C++ oracle agrees with an earlier numpy restatement (integers and fp32 dequant
  bitwise, Y to fp64 summation order).
"""
from __future__ import annotations

import fractions
import os

import numpy as np
import pytest

import mnb_synth as syn
from oracle import mnb_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_worked_example.txt")


def _read_golden(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def _pack_codes(codes_nk: np.ndarray) -> np.ndarray:
    """Test-side packer (the inverse direction): row n is K/2 bytes, low nibble = even k."""
    N, K = codes_nk.shape
    c = codes_nk.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _pack_zp(zp_ng: np.ndarray) -> np.ndarray:
    N, G = zp_ng.shape
    zrb = -(-G // 2)
    out = np.zeros((N, zrb), dtype=np.uint8)
    for g in range(G):
        if g % 2 == 0:
            out[:, g // 2] |= zp_ng[:, g].astype(np.uint8)
        else:
            out[:, g // 2] |= (zp_ng[:, g].astype(np.uint8) << 4)
    return out


def test_golden_worked_example():
    g = _read_golden(GOLDEN)
    K, N, bs = int(g["K"][0]), int(g["N"][0]), int(g["block_size"][0])
    packed = np.array([int(x, 16) for x in g["packed"]], dtype=np.uint8).reshape(N, -1)
    zp = np.array([int(x, 16) for x in g["zero_points"]], dtype=np.uint8).reshape(N, -1)
    scales = np.array([int(x, 16) for x in g["scales_f16_bits"]], dtype=np.uint16).view(np.float16).reshape(N, -1)
    W = orc.dequant_kn_f32(packed, scales, zp, K, N, bs)
    np.testing.assert_array_equal(W[:, 0], np.array(g["dequant_n0"], dtype=np.float32))
    np.testing.assert_array_equal(W[:, 1], np.array(g["dequant_n1"], dtype=np.float32))
    A = np.ones((1, K), dtype=np.float16)
    Y, B = orc.matmul(A, packed, scales, zp, K, N, bs)
    np.testing.assert_array_equal(Y[0], np.array(g["y_ones"], dtype=np.float64))
    np.testing.assert_array_equal(B[0], np.array(g["bound_ones"], dtype=np.float64))
    Y0, _ = orc.matmul(A, packed, scales, None, K, N, bs)
    np.testing.assert_array_equal(Y0[0], np.array(g["y_ones_no_zp"], dtype=np.float64))


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_single_hot_layout(bs):
    """One code differs from the zero point; A = e_k: only Y[n] is nonzero, exactly."""
    K, N = 3 * bs, 5
    G = K // bs
    rng = np.random.default_rng(bs)
    scales = (rng.uniform(0.25, 2.0, size=(N, G))).astype(np.float16)
    for (n, k, c) in [(0, 0, 3), (1, 1, 15), (4, K - 1, 0), (2, bs + 1, 12), (3, 2 * bs, 9)]:
        packed = np.full((N, K // 2), 0x88, dtype=np.uint8)   # every code 8 = default zp
        byte = n * (K // 2) + k // 2
        flat = packed.reshape(-1)
        flat[byte] = (flat[byte] & 0xF0) | c if k % 2 == 0 else (flat[byte] & 0x0F) | (c << 4)
        A = np.zeros((1, K), dtype=np.float16)
        A[0, k] = 1.0
        Y, B = orc.matmul(A, packed, scales, None, K, N, bs)
        expect = np.zeros(N)
        expect[n] = (c - 8) * float(scales[n, k // bs])
        np.testing.assert_array_equal(Y[0], expect)
        W = orc.dequant_kn_f32(packed, scales, None, K, N, bs)
        assert np.count_nonzero(W) == (1 if c != 8 else 0)
        assert W[k, n] == np.float32(expect[n])


@pytest.mark.parametrize("g", [0, 1, 2, 5])
def test_zero_point_nibble_order(g):
    """A single non-default zero point at an even or odd group shifts only that group."""
    bs, G, N = 16, 6, 3
    K = bs * G
    zp_ng = np.full((N, G), 8)
    zp_ng[1, g] = 3
    zp = _pack_zp(zp_ng)
    packed = np.full((N, K // 2), 0x88, dtype=np.uint8)
    scales = np.ones((N, G), dtype=np.float16)
    W = orc.dequant_kn_f32(packed, scales, zp, K, N, bs)
    expect = np.zeros((K, N), dtype=np.float32)
    expect[g * bs:(g + 1) * bs, 1] = 8 - 3
    np.testing.assert_array_equal(W, expect)
    # explicit nibble check by byte: low nibble for even g
    byte = zp[1, g // 2]
    assert ((byte & 15) if g % 2 == 0 else (byte >> 4)) == 3


def test_layout_second_reading_u32_words():
    """The fp16 GEMV kernel in matmul_nbits.rs loads aligned 32-bit words of a row and
    takes nibble i (bits 4i..4i+3) as k = depth + i.  Decoding that way must agree."""
    K, N, bs = 256, 7, 32
    packed = syn.random_bytes(1234, N * K // 2).reshape(N, K // 2)
    words = packed.reshape(-1).view("<u4").reshape(N, K // 8).astype(np.int64)
    by_words = np.empty((N, K), dtype=np.int64)
    for i in range(8):
        by_words[:, i::8] = (words >> (4 * i)) & 15
    np.testing.assert_array_equal(orc.codes(packed, K, N, bs), by_words)


def test_default_zero_point_is_8():
    wl = syn.custom("pin_default_zp", 3, 192, 40, 64, has_zp=False)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    explicit = np.full((wl.N, wl.zp_row_bytes), 0x88, dtype=np.uint8)
    Y0, B0 = orc.matmul(A, w.packed, w.scales, None, wl.K, wl.N, wl.block_size)
    Y1, B1 = orc.matmul(A, w.packed, w.scales, explicit, wl.K, wl.N, wl.block_size)
    np.testing.assert_array_equal(Y0, Y1)
    np.testing.assert_array_equal(B0, B1)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_all_codes_equal_zero_point_gives_zero(bs):
    K, N, M = 2 * bs, 9, 3
    G = K // bs
    rng = np.random.default_rng(7 + bs)
    zp_ng = rng.integers(0, 16, size=(N, G))
    codes_nk = np.repeat(zp_ng, bs, axis=1)
    packed = _pack_codes(codes_nk)
    zp = _pack_zp(zp_ng)
    scales = rng.uniform(0.001, 3.0, size=(N, G)).astype(np.float32)
    A = rng.standard_normal((M, K)).astype(np.float16)
    Y, B = orc.matmul(A, packed, scales, zp, K, N, bs)
    assert np.all(Y == 0.0) and np.all(B == 0.0)


def test_scale_linearity():
    """Doubling one group's scale doubles exactly that group's contribution."""
    wl = syn.custom("pin_linearity", 1, 128, 6, 32, scales_dtype="f16")
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    g = 2
    A_in = np.zeros_like(A)
    A_in[:, g * 32:(g + 1) * 32] = A[:, g * 32:(g + 1) * 32]
    A_out = A - A_in
    s2 = w.scales.copy()
    s2[:, g] = (s2[:, g].astype(np.float32) * 2).astype(np.float16)  # power of two: exact
    y_in, _ = orc.matmul(A_in, w.packed, w.scales, w.zero_points, wl.K, wl.N, 32)
    y_in2, _ = orc.matmul(A_in, w.packed, s2, w.zero_points, wl.K, wl.N, 32)
    y_out, _ = orc.matmul(A_out, w.packed, w.scales, w.zero_points, wl.K, wl.N, 32)
    y_out2, _ = orc.matmul(A_out, w.packed, s2, w.zero_points, wl.K, wl.N, 32)
    np.testing.assert_array_equal(y_in2, 2 * y_in)
    np.testing.assert_array_equal(y_out2, y_out)


def test_integer_special_case_matches_int64_matmul():
    """zp = 0, scale = 1, integer activations: Y is the integer product of A and the codes."""
    K, N, M, bs = 256, 33, 4, 64
    G = K // bs
    rng = np.random.default_rng(99)
    codes_nk = rng.integers(0, 16, size=(N, K))
    packed = _pack_codes(codes_nk)
    zp = np.zeros((N, -(-G // 2)), dtype=np.uint8)
    scales = np.ones((N, G), dtype=np.float16)
    A_int = rng.integers(-8, 9, size=(M, K))
    Y, B = orc.matmul(A_int.astype(np.float16), packed, scales, zp, K, N, bs)
    exact = A_int.astype(np.int64) @ codes_nk.astype(np.int64).T
    np.testing.assert_array_equal(Y, exact.astype(np.float64))
    np.testing.assert_array_equal(B, (np.abs(A_int) @ codes_nk.T).astype(np.float64))


def test_exact_rational_brute_force():
    """Tiny problem in exact rationals, decoding bytes the word way, summing in any order."""
    wl = syn.custom("pin_rational", 2, 64, 3, 16, scales_dtype="f32")
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    K, N, bs, G = wl.K, wl.N, wl.block_size, wl.k_blocks
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs)
    for m in range(wl.M):
        for n in range(N):
            acc = fractions.Fraction(0)
            row = w.packed[n].tobytes()
            for k in range(K):
                b = row[k // 2]
                code = (b >> 4) if k % 2 else (b & 15)
                zb = int(w.zero_points[n][(k // bs) // 2])
                zpv = (zb >> 4) if (k // bs) % 2 else (zb & 15)
                s = fractions.Fraction(float(w.scales[n, k // bs]))
                a = fractions.Fraction(float(A[m, k]))
                acc += a * (code - zpv) * s
            assert abs(Y[m, n] - float(acc)) <= 1e-12 * max(1.0, B[m, n])


def test_f16_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.f16_to_f64(bits.view(np.float16))
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_silu_against_expit():
    scipy_special = pytest.importorskip("scipy.special")
    x = np.linspace(-40, 40, 2001)
    np.testing.assert_allclose(orc.silu(x), x * scipy_special.expit(x), rtol=1e-14, atol=1e-300)
    assert orc.silu(np.array([0.0]))[0] == 0.0


def test_dequant_matches_product_definition():
    """Y equals A times the fp32 dequantised matrix when that matrix is exact (fp16 scales)."""
    wl = syn.custom("pin_compose", 3, 256, 20, 32, scales_dtype="f16")
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    W = orc.dequant_kn_f32(w.packed, w.scales, w.zero_points, wl.K, wl.N, 32).astype(np.float64)
    Y, _ = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, 32)
    np.testing.assert_allclose(orc.activations_f64(A) @ W, Y, rtol=0, atol=1e-12)


def test_partial_last_block():
    """K not a multiple of bs: k_blocks = ceil(K/bs); padding nibbles are never read."""
    K, N, bs = 40, 2, 16          # 3 blocks, the last one half used
    G = 3
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, size=(N, G * bs // 2)).astype(np.uint8)
    scales = np.ones((N, G), dtype=np.float16)
    c = orc.codes(packed, K, N, bs)
    assert c.shape == (N, K)
    # k = 32..39 live in block 2, bytes 16..19 of the row's 24
    np.testing.assert_array_equal(c[:, 32], packed[:, 16] & 15)
    np.testing.assert_array_equal(c[:, 39], packed[:, 19] >> 4)
    W = orc.dequant_kn_f32(packed, scales, None, K, N, bs)
    assert W.shape == (K, N)


def test_repack_hand_placed_code():
    """Code 7 at (n=1, k=3) lands in byte 18, high nibble (hand-derived from the layout).

    Tile 0, k-block 0, q = 0, r = 1 -> offset 16; i = 3 = 8*0 + 2*(p%4) + p//4 gives
    p = 5: word 0, byte 5//2 = 2, odd p -> high nibble.  Offset 16 + 2 = 18.
    """
    K, N, bs = 64, 2, 32
    codes_nk = np.zeros((N, K), dtype=np.int64)
    codes_nk[1, 3] = 7
    out = orc.repack(_pack_codes(codes_nk), K, N, bs)
    assert out.size == 128 * 64 // 2
    nz = np.nonzero(out)[0]
    assert list(nz) == [18] and out[18] == 0x70
    # and (n=130, k=70): tile 1, k-block 1 of Kp/64 = 2 -> block 3 at 12288; q = 0, r = 2,
    # i = 6 = 2*(p%4) + p//4 -> p = 3: byte 1, high nibble.  12288 + 32 + 1 = 12321.
    K, N = 128, 131
    codes_nk = np.zeros((N, K), dtype=np.int64)
    codes_nk[130, 70] = 5
    out = orc.repack(_pack_codes(codes_nk), K, N, 64)
    assert out.size == 256 * 128 // 2
    nz = np.nonzero(out)[0]
    assert list(nz) == [12321] and out[12321] == 0x50


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_repack_roundtrip_is_bijection(bs):
    K, N = 3 * max(bs, 64), 5 + 128
    packed = syn.random_bytes(77 + bs, N * K // 2).reshape(N, K // 2)
    rp = orc.repack(packed, K, N, bs)
    assert rp.size == orc.repacked_bytes(K, N)
    np.testing.assert_array_equal(orc.unrepack_codes(rp, K, N), orc.codes(packed, K, N, bs))
    # every stored nibble used exactly once, padding nibbles zero: with every code 15 the
    # buffer holds exactly N * K set nibbles (two codes sent to one nibble would leave
    # fewer), and each single-hot code lands alone
    full = orc.repack(np.full((N, K // 2), 0xFF, dtype=np.uint8), K, N, bs)
    nib = np.stack([full & 15, full >> 4], axis=1).reshape(-1)
    assert set(np.unique(nib).tolist()) <= {0, 15}
    assert int(np.count_nonzero(nib)) == N * K
    rng = np.random.default_rng(bs)
    seen = set()
    for _ in range(64):
        n, k = int(rng.integers(N)), int(rng.integers(K))
        c = np.zeros((N, K), dtype=np.int64)
        c[n, k] = 9
        one = orc.repack(_pack_codes(c), K, N, bs)
        nz = np.nonzero(one)[0]
        assert nz.size == 1 and one[nz[0]] in (0x09, 0x90)
        seen.add((int(nz[0]), int(one[nz[0]]), n, k))
    assert len({(b, v) for b, v, _, _ in seen}) == len({(n, k) for _, _, n, k in seen})


def test_synth_streams_are_deterministic():
    a = syn.splitmix64(42, 5)
    b = syn.splitmix64(42, 5)
    assert np.array_equal(a, b)
    # SplitMix64 reference outputs for seed 0 (first three values of the published generator)
    z = syn.splitmix64(0, 3)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


# ---------------------------------------------------------------------------
# Act-order g_idx (matmul_nbits.rs, matmul_nbits_dequant_f32 and the g_idx check)
# ---------------------------------------------------------------------------


def test_g_idx_identity_equals_plain_layout():
    wl = syn.custom("pin_gidx_identity", 2, 256, 9, 32)
    w = syn.make_weight(wl)
    g_idx = np.repeat(np.arange(wl.k_blocks, dtype=np.int32), wl.block_size)
    plain = orc.weight_nk(w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    act = orc.weight_nk(w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, g_idx)
    np.testing.assert_array_equal(act, plain)


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_g_idx_act_order_construction(bs):
    """Quantise in a visit order v (group = step // bs), store codes in k order: the
    g_idx weight at column v[j] equals the plain weight of the visit-ordered codes at j."""
    K, N = 8 * bs, 5
    G = K // bs
    rng = np.random.default_rng(bs)
    q = rng.integers(0, 16, size=(N, K))          # codes in visit order
    zp = rng.integers(0, 16, size=(N, G))
    scales = rng.uniform(0.01, 0.1, size=(N, G)).astype(np.float16)
    v = rng.permutation(K)                         # v[j] = the k visited at step j
    stored = np.empty_like(q)
    stored[:, v] = q
    g_idx = np.empty(K, dtype=np.int32)
    g_idx[v] = np.arange(K) // bs
    w_act = orc.weight_nk(_pack_codes(stored), scales, _pack_zp(zp), K, N, bs, g_idx)
    w_plain = orc.weight_nk(_pack_codes(q), scales, _pack_zp(zp), K, N, bs)
    np.testing.assert_array_equal(w_act[:, v], w_plain)


def test_g_idx_exact_rational_brute_force():
    """Uneven groups and two out-of-range entries (which contribute nothing)."""
    wl = syn.custom("pin_gidx_rational", 2, 64, 3, 16, scales_dtype="f32")
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    K, N, bs, G = wl.K, wl.N, wl.block_size, wl.k_blocks
    g_idx = syn.make_g_idx(wl, "uneven").copy()
    g_idx[5], g_idx[40] = -1, G
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    for m in range(wl.M):
        for n in range(N):
            acc = fractions.Fraction(0)
            row = w.packed[n].tobytes()
            for k in range(K):
                g = int(g_idx[k])
                if not 0 <= g < G:
                    continue
                b = row[k // 2]
                code = (b >> 4) if k % 2 else (b & 15)
                zb = int(w.zero_points[n][g // 2])
                zpv = (zb >> 4) if g % 2 else (zb & 15)
                s = fractions.Fraction(float(w.scales[n, g]))
                acc += fractions.Fraction(float(A[m, k])) * (code - zpv) * s
            assert abs(Y[m, n] - float(acc)) <= 1e-12 * max(1.0, B[m, n])


def test_act_order_plan_hand_worked():
    """K = 12, bs = 4, three groups of sizes 5, 1 and 6, worked out by hand:
    group 0 = k {1, 2, 6, 9, 10} -> 2 blocks, group 1 = {4} -> 1, group 2 =
    {0, 3, 5, 7, 8, 11} -> 2; empty slots close each group's last block."""
    g_idx = np.array([2, 0, 0, 2, 1, 2, 0, 2, 2, 0, 0, 2], dtype=np.int32)
    Kp, perm, bg = orc.act_order_plan(g_idx, 12, 4)
    assert Kp == 20
    assert perm.tolist() == [1, 2, 6, 9, 10, -1, -1, -1, 4, -1, -1, -1,
                             0, 3, 5, 7, 8, 11, -1, -1]
    assert bg.tolist() == [0, 0, 1, 2, 2]


def test_act_order_plan_balanced_keeps_k():
    wl = syn.custom("pin_plan_balanced", 1, 1024, 4, 128)
    g_idx = syn.make_g_idx(wl, "act_order")
    Kp, perm, bg = orc.act_order_plan(g_idx, wl.K, wl.block_size)
    assert Kp == wl.K
    assert sorted(perm.tolist()) == list(range(wl.K))
    np.testing.assert_array_equal(g_idx[perm], np.arange(wl.K) // wl.block_size)
    assert bg.tolist() == list(range(wl.k_blocks))


def test_act_order_plan_rejects_out_of_range():
    g_idx = np.zeros(64, dtype=np.int32)
    g_idx[7] = 4
    with pytest.raises(ValueError, match=r"g_idx\[7\]=4"):
        orc.act_order_plan(g_idx, 64, 16)
    g_idx[7] = -1
    with pytest.raises(ValueError):
        orc.act_order_plan(g_idx, 64, 16)


@pytest.mark.parametrize("kind,has_zp,sdt", [("act_order", True, "f16"), ("uneven", True, "f32"),
                                              ("uneven", False, "f16"), ("identity", True, "f16")])
def test_act_order_prepare_holds_the_same_weights(kind, has_zp, sdt):
    wl = syn.custom(f"pin_prepare_{kind}_{has_zp}_{sdt}", 1, 512, 7, 32, scales_dtype=sdt, has_zp=has_zp)
    w = syn.make_weight(wl)
    g_idx = syn.make_g_idx(wl, kind)
    Kp, perm, bg = orc.act_order_plan(g_idx, wl.K, wl.block_size)
    pk, sc, zp = orc.act_order_prepare(w.packed, w.scales, w.zero_points, wl.K, wl.N,
                                       wl.block_size, perm, bg)
    assert pk.shape == (wl.N, Kp // 2) and sc.shape == (wl.N, Kp // wl.block_size)
    assert sc.dtype == w.scales.dtype and (zp is None) == (not has_zp)
    w_prep = orc.weight_nk(pk, sc, zp, Kp, wl.N, wl.block_size)
    w_orig = orc.weight_nk(w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, g_idx)
    real = perm >= 0
    np.testing.assert_array_equal(w_prep[:, real], w_orig[:, perm[real]])
    np.testing.assert_array_equal(w_prep[:, ~real], 0.0)
    if kind == "identity":
        assert Kp == wl.K and perm.tolist() == list(range(wl.K))
        np.testing.assert_array_equal(pk, w.packed)


def test_act_order_product_equivalence_exact():
    """Integer activations and power-of-two scales: every sum is exact in fp64, so the
    gathered product over the prepared weight equals the g_idx product bit for bit."""
    K, N, M, bs = 256, 6, 3, 32
    G = K // bs
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    zp = rng.integers(0, 256, size=(N, -(-G // 2))).astype(np.uint8)
    scales = (2.0 ** rng.integers(-6, 0, size=(N, G))).astype(np.float16)
    A = rng.integers(-9, 10, size=(M, K)).astype(np.float16)
    g_idx = rng.integers(0, G, size=K).astype(np.int32)
    Y, _ = orc.matmul(A, packed, scales, zp, K, N, bs, g_idx)
    Kp, perm, bg = orc.act_order_plan(g_idx, K, bs)
    pk, sc, zpp = orc.act_order_prepare(packed, scales, zp, K, N, bs, perm, bg)
    Ag = orc.act_order_gather(A, perm)
    Y2, _ = orc.matmul(Ag, pk, sc, zpp, Kp, N, bs)
    np.testing.assert_array_equal(Y2, Y)
    assert np.all(Ag[:, perm < 0] == 0) and not np.any(np.signbit(Ag[:, perm < 0]))


def test_f32_activations_exact_rational():
    """fp32 activations enter at their own value, not rounded to fp16: 1 + 2^-20, 1e6 and
    3e-9 are not fp16 numbers, and the product equals the exact rational sum."""
    K, N, bs = 32, 2, 16
    rng = np.random.default_rng(3)
    codes_nk = rng.integers(0, 16, size=(N, K))
    packed = _pack_codes(codes_nk)
    zp = _pack_zp(rng.integers(0, 16, size=(N, K // bs)))
    scales = np.array([[0.25, 0.125], [0.5, 2.0]], dtype=np.float32)
    A = np.full((1, K), 1.0 + 2.0 ** -20, dtype=np.float32)
    A[0, 3], A[0, 17] = 1e6, 3e-9
    Y, _ = orc.matmul(A, packed, scales, zp, K, N, bs)
    zpn = orc.zero_points(zp, K, N, bs)
    for n in range(N):
        acc = fractions.Fraction(0)
        for k in range(K):
            acc += fractions.Fraction(float(A[0, k])) * int(codes_nk[n, k] - zpn[n, k // bs]) * \
                fractions.Fraction(float(scales[n, k // bs]))
        assert abs(Y[0, n] - float(acc)) <= 1e-12 * abs(float(acc)) + 1e-300
    # within the fp16 range, the fp16-rounded activation gives a different result
    A[0, 3] = 1.0
    Y32, _ = orc.matmul(A, packed, scales, zp, K, N, bs)
    Y16, _ = orc.matmul(A.astype(np.float16), packed, scales, zp, K, N, bs)
    assert not np.allclose(Y16, Y32, rtol=1e-9, atol=0)


# ---------------------------------------------------------------------------
# Spot-check products, thread-count invariance, and the numpy cross-check
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("case", ["zp_f16", "nozp_f32", "gidx_uneven", "gidx_act_order", "f32_act"])
def test_matmul_rows_equals_matmul_at_the_pairs(case):
    """The spot-check product at (row, col) pairs (the full-size referee) equals the full
    product there bit for bit, with repeated and unsorted columns and rows, with and
    without zero points, fp16 and fp32 scales, with act-order groups (uneven sizes, some
    empty) and fp32 activations."""
    sdt = "f32" if case == "nozp_f32" else "f16"
    wl = syn.custom(f"pin_rows_{case}", 5, 384, 37, 32, scales_dtype=sdt, has_zp=case != "nozp_f32")
    w = syn.make_weight(wl)
    A = syn.make_activation_f32(wl) if case == "f32_act" else syn.make_activation(wl)
    g_idx = None
    if case.startswith("gidx"):
        g_idx = syn.make_g_idx(wl, "uneven" if case == "gidx_uneven" else "act_order")
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, g_idx)
    rows = np.array([4, 0, 4, 2, 1, 3, 0, 4, 2, 2], dtype=np.int64)
    cols = np.array([36, 5, 5, 0, 36, 17, 17, 2, 2, 30], dtype=np.int64)
    y, b = orc.matmul_rows(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, rows, cols, g_idx)
    np.testing.assert_array_equal(y, Y[rows, cols])
    np.testing.assert_array_equal(b, B[rows, cols])


def test_matmul_rows_sees_the_column_of_each_pair():
    """Two pairs at one row and two columns with different weights give the two different
    full-product values (a mapping that sent every pair to one column would not)."""
    wl = syn.custom("pin_rows_cols", 2, 128, 4, 32)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    Y, _ = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size)
    y, _ = orc.matmul_rows(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, [1, 1, 0], [3, 0, 3])
    assert len({float(v) for v in Y[[1, 1, 0], [3, 0, 3]]}) == 3
    np.testing.assert_array_equal(y, Y[[1, 1, 0], [3, 0, 3]])


def test_matmul_thread_count_changes_nothing():
    wl = syn.custom("pin_threads", 3, 512, 67, 64)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    Y1, B1 = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, nthreads=1)
    Y7, B7 = orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, nthreads=7)
    np.testing.assert_array_equal(Y1, Y7)
    np.testing.assert_array_equal(B1, B7)


@pytest.mark.parametrize("bs,sdt,has_zp,gkind", [(16, "f16", True, None), (32, "f32", False, None),
                                                  (64, "f16", True, "uneven"), (128, "f32", True, "act_order")])
def test_cpp_oracle_agrees_with_numpy_restatement(bs, sdt, has_zp, gkind):
    """The C++ oracle and the earlier numpy restatement of the same definition: integer
    decodes, the fp32 dequant and the repack byte for byte; Y to fp64 summation order."""
    from oracle import mnb_oracle_np as onp
    wl = syn.custom(f"pin_xcheck_{bs}_{sdt}", 3, 4 * max(bs, 64), 29, bs, scales_dtype=sdt, has_zp=has_zp)
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    K, N = wl.K, wl.N
    g_idx = None if gkind is None else syn.make_g_idx(wl, gkind)
    np.testing.assert_array_equal(orc.codes(w.packed, K, N, bs), onp.codes(w.packed, K, N, bs))
    np.testing.assert_array_equal(orc.zero_points(w.zero_points, K, N, bs), onp.zero_points(w.zero_points, K, N, bs))
    np.testing.assert_array_equal(orc.weight_nk(w.packed, w.scales, w.zero_points, K, N, bs, g_idx),
                                  onp.weight_nk(w.packed, w.scales, w.zero_points, K, N, bs, g_idx))
    np.testing.assert_array_equal(orc.dequant_kn_f32(w.packed, w.scales, w.zero_points, K, N, bs, g_idx).view(np.uint32),
                                  onp.dequant_kn_f32(w.packed, w.scales, w.zero_points, K, N, bs, g_idx).view(np.uint32))
    np.testing.assert_array_equal(orc.repack(w.packed, K, N, bs), onp.repack(w.packed, K, N, bs))
    Y, B = orc.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    Yn, Bn = onp.matmul(A, w.packed, w.scales, w.zero_points, K, N, bs, g_idx)
    assert np.all(np.abs(Y - Yn) <= 1e-12 * B)
    np.testing.assert_allclose(B, Bn, rtol=1e-12, atol=0)
    if g_idx is not None:
        plan, plan_n = orc.act_order_plan(g_idx, K, bs), onp.act_order_plan(g_idx, K, bs)
        assert plan[0] == plan_n[0]
        np.testing.assert_array_equal(plan[1], plan_n[1])
        np.testing.assert_array_equal(plan[2], plan_n[2])
        prep = orc.act_order_prepare(w.packed, w.scales, w.zero_points, K, N, bs, plan[1], plan[2])
        prep_n = onp.act_order_prepare(w.packed, w.scales, w.zero_points, K, N, bs, plan[1], plan[2])
        for x, xn in zip(prep, prep_n):
            if x is None:
                assert xn is None
            else:
                np.testing.assert_array_equal(x.view(np.uint8), xn.view(np.uint8))
        np.testing.assert_array_equal(orc.act_order_gather(A, plan[1]).view(np.uint16),
                                      onp.act_order_gather(A, plan[1]).view(np.uint16))
