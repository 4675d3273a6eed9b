"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against exact rational arithmetic (brute force on
tiny inputs), closed forms and special cases that reduce to a library
routine, or hand-derived values from the definitions:

* quantizer -- "test_int4_quantized_gemm.py", _packed_with_dense
  (INT4, group 32, asymmetric min-max);
* dequant + matmul -- "test_int4_quantized_gemm.py", _dequant_matmul;
* W4A8 -- "test_int4_quantized_gemm.py", Int4QuantizedGemmPrecisionTest;
* W8 -- "gpt-fast issue #114", WeightOnlyInt8Linear.forward;
* packed layout -- this library's layout (the header include/w4q.h).
"""
import bisect
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GROUP = 32

# --------------------------------------------------------------------------
# exact bf16 helpers (independent of the oracle's C code)
# --------------------------------------------------------------------------


def bits_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def float_to_bits(v: float) -> int:
    """bf16 bits of a float that is exactly representable in bf16."""
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    assert u & 0xFFFF == 0, v
    return u >> 16


_POS = None


def positive_bf16():
    """Every finite positive bf16 as (Fraction value, bits), sorted."""
    global _POS
    if _POS is None:
        _POS = sorted((Fraction(bits_to_float(b)), b) for b in range(1, 0x7F80))
    return _POS


def ru_bf16_brute(v: Fraction) -> int:
    """Smallest bf16 >= v > 0, by search over every bf16 number."""
    table = positive_bf16()
    i = bisect.bisect_left(table, (v, -1))
    return table[i][1]


def clamp15(v):
    return min(15, max(0, v))


def brute_quant_group(wbits):
    """Exact-rational restatement of the quantizer on one group."""
    vals = [Fraction(bits_to_float(b)) for b in wbits]
    mx, mn = max(vals), min(vals)
    if mx == mn:
        c = abs(mx)
        sb = 0x3F80 if c == 0 else ru_bf16_brute(c / 15)
    else:
        sb = ru_bf16_brute((mx - mn) / 15)
    s = Fraction(bits_to_float(sb))
    z = clamp15(round(-mn / s))          # round(): half to even
    q = [clamp15(round(v / s) + z) for v in vals]
    return q, sb, z


def quant_rows(groups):
    """Run the oracle on a list of 32-element groups (one row each)."""
    W = np.array(groups, dtype=np.uint16).reshape(len(groups), GROUP)
    q, s, z = oracle.quantize_w4(W, len(groups), GROUP)
    return q, s, z


def randn_bits(shape, seed):
    return workloads.randn_bf16(shape, seed).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# quantizer
# --------------------------------------------------------------------------


def test_quantizer_matches_exact_rational_brute_force_on_randn():
    W = randn_bits((64, 128), seed=5)
    q, s, z = oracle.quantize_w4(W, 64, 128)
    for n in range(64):
        for g in range(128 // GROUP):
            bq, bs, bz = brute_quant_group(W[n, g * GROUP:(g + 1) * GROUP])
            assert s[n, g] == bs
            assert z[n, g] == bz
            assert list(q[n, g * GROUP:(g + 1) * GROUP]) == bq


def _group(values):
    vals = list(values) + [values[-1]] * (GROUP - len(values))
    return [float_to_bits(v) for v in vals]


ADVERSARIAL = {
    # range 15 -> s = 1 exactly, z = 1 (odd): w/s = 0.5 must give q = 0 + 1,
    # not rint(0.5 + 1) = 2 (the zero point is a separately rounded term).
    "tie_odd_zero": [-1.0, 14.0, 0.5, 1.5, 2.5, -0.5, 3.5, 12.5],
    # z = 2 (even).
    "tie_even_zero": [-2.0, 13.0, 0.5, 1.5, 2.5, -1.5, 4.5],
    "all_zero": [0.0],
    "negative_zero": [-0.0, 0.0, -0.0],
    "constant_pos": [3.0],
    "constant_neg": [-3.0],
    "same_sign_pos": [1.0, 1.25, 1.5, 2.0],
    "same_sign_neg": [-1.0, -1.25, -1.5, -2.0],
    # exact multiples of s = 0.5 around z = 4: dequant is exact.
    "exact_multiples": [-2.0, 5.5, -1.5, 0.0, 0.5, 3.0, 4.5],
    "tiny_subnormal_range": [bits_to_float(0x0001), bits_to_float(0x0003)],
    "huge_range": [bits_to_float(0xFF7F), bits_to_float(0x7F7F), bits_to_float(0x7E96)],
}


@pytest.mark.parametrize("name", sorted(ADVERSARIAL))
def test_quantizer_adversarial_groups(name):
    bits = _group(ADVERSARIAL[name])
    q, s, z = quant_rows([bits])
    bq, bs, bz = brute_quant_group(bits)
    assert (int(s[0, 0]), int(z[0, 0]), list(q[0])) == (bs, bz, bq)


def test_quantizer_hand_derived_values():
    # range 15 -> s = 1.0 (bf16 0x3F80), z = rint(1/1) = 1.
    q, s, z = quant_rows([_group([-1.0, 14.0, 0.5, 1.5, 2.5, -0.5])])
    assert s[0, 0] == 0x3F80 and z[0, 0] == 1
    # codes: -1 -> 0, 14 -> 15, 0.5 -> 0+1, 1.5 -> 2+1, 2.5 -> 2+1, -0.5 -> 0+1
    assert list(q[0, :6]) == [0, 15, 1, 3, 3, 1]
    # constant 3.0: s = RU_bf16(0.2) = 0.2001953125 (0x3E4D), z = 0, q = 15
    q, s, z = quant_rows([_group([3.0])])
    assert s[0, 0] == 0x3E4D and z[0, 0] == 0 and q[0, 0] == 15
    # constant -3.0: z = 15, q = 0
    q, s, z = quant_rows([_group([-3.0])])
    assert s[0, 0] == 0x3E4D and z[0, 0] == 15 and q[0, 0] == 0
    # all zeros: s = 1.0, z = 0, q = 0 -> dequant exactly 0
    q, s, z = quant_rows([_group([0.0])])
    assert s[0, 0] == 0x3F80 and z[0, 0] == 0 and q[0, 0] == 0


def test_quantizer_invariants_on_randn():
    N, K = 512, 1024
    W = randn_bits((N, K), seed=11)
    q, s, z = oracle.quantize_w4(W, N, K)
    assert q.max() <= 15 and z.max() <= 15
    w = oracle.bf16_bits_to_f64(W).reshape(N, K // GROUP, GROUP)
    sv = oracle.bf16_bits_to_f64(s)[:, :, None]
    deq = (q.reshape(N, K // GROUP, GROUP).astype(np.float64) - z[:, :, None]) * sv
    mx, mn = w.max(axis=2), w.min(axis=2)
    straddle = (mn <= 0) & (mx >= 0)
    assert straddle.mean() > 0.99
    err = np.abs(w - deq)
    assert np.all(err[straddle] <= sv[straddle] / 2)
    # s is the least bf16 >= (max - min) / 15 (exact in fp64 for these inputs)
    rng = (mx - mn) / 15.0
    assert np.all(sv[:, :, 0] >= rng)
    prev = oracle.bf16_bits_to_f64(s.astype(np.int64) - 1)
    assert np.all(prev < rng)


def test_dequant_is_q_minus_z_times_s():
    q = np.array([[0, 15, 7, 8] * 8], dtype=np.uint8)
    s = np.array([[float_to_bits(0.5)]], dtype=np.uint16)
    z = np.array([[7]], dtype=np.uint8)
    d = oracle.dequant_w4(q, s, z)
    assert list(d[0, :4]) == [-3.5, 4.0, 0.0, 0.5]


# --------------------------------------------------------------------------
# packed layout
# --------------------------------------------------------------------------


def decode_layout(packed, N, K):
    """Second, vectorised reading of the documented layout (independent of
    the oracle's scalar code): returns q [N,K], s [N,K/32], z [N,K/32]."""
    KB, G = K // 256, (N + 127) // 128
    T = 8 * G
    # tiles are ordered (128-row group, super-block, row tile in the group)
    tiles = packed.reshape(G, KB, 8, 2432).transpose(0, 2, 1, 3).reshape(T, KB, 2432)
    nib = tiles[:, :, :2048].reshape(T, KB, 4, 32, 4, 4)          # sb, lane, word, byte
    words = nib.astype(np.uint32)
    words = words[..., 0] | (words[..., 1] << 8) | (words[..., 2] << 16) | (words[..., 3] << 24)
    q = np.zeros((T * 16, K), np.uint8)
    for lane in range(32):
        r, c = lane // 4, 2 * (lane % 4)
        for a in range(2):          # row half
            for e in range(2):      # column half
                for h in range(2):
                    row = r + 8 * a
                    col = c + 8 * e + h
                    vals = (words[:, :, :, lane, :] >> (8 * a + 4 * e + 16 * h)) & 0xF
                    for sb in range(4):
                        for j in range(4):
                            k = np.arange(KB) * 256 + 64 * sb + 16 * j + col
                            q[np.arange(T)[:, None] * 16 + row, k[None, :]] = vals[:, :, sb, j]
    sc = tiles[:, :, 2048:2304].reshape(T, KB, 2, 8, 4, 2, 2)       # ghi, r, glo, half, byte
    sc = sc[..., 0].astype(np.uint16) | (sc[..., 1].astype(np.uint16) << 8)
    s = np.zeros((T * 16, K // 32), np.uint16)
    zr = tiles[:, :, 2304:2432].reshape(T, KB, 8, 8, 2)              # r, g, half
    z = np.zeros((T * 16, K // 32), np.uint8)
    for r in range(8):
        for half in range(2):
            rows = np.arange(T) * 16 + r + 8 * half
            for g in range(8):
                s[rows[:, None], np.arange(KB)[None, :] * 8 + g] = sc[:, :, g // 4, r, g % 4, half]
                z[rows[:, None], np.arange(KB)[None, :] * 8 + g] = zr[:, :, r, g, half]
    return q[:N], s[:N], z[:N], q[N:], s[N:], z[N:]


def test_packed_size():
    assert oracle.packed_bytes(256, 768) == 16 * 3 * 2432 == 116736
    assert oracle.packed_bytes(257, 256) == 3 * 8 * 2432      # rows padded to 3 * 128
    assert oracle.packed_bytes(16, 256) == 8 * 2432
    assert oracle.packed_bytes(39936, 6656) == 157827072
    assert oracle.packed_bytes(64, 288) == 0       # K % 256 != 0 is unsupported


@pytest.mark.parametrize("N,K", [(16, 256), (257, 512), (40, 768)])
def test_pack_matches_independent_layout_decoder(N, K):
    rng = np.random.default_rng(N * 7 + K)
    q = rng.integers(0, 16, (N, K), dtype=np.uint8)
    s = rng.integers(0, 0x7F80, (N, K // 32), dtype=np.uint16)
    z = rng.integers(0, 16, (N, K // 32), dtype=np.uint8)
    packed = oracle.pack_w4(q, s, z)
    dq, ds, dz, pq, ps, pz = decode_layout(packed, N, K)
    np.testing.assert_array_equal(dq, q)
    np.testing.assert_array_equal(ds, s)
    np.testing.assert_array_equal(dz, z)
    assert not pq.any() and not ps.any() and not pz.any()   # padded rows are zero
    uq, us, uz = oracle.unpack_w4(packed, N, K)
    np.testing.assert_array_equal(uq, q)
    np.testing.assert_array_equal(us, s)
    np.testing.assert_array_equal(uz, z)


def test_pack_hand_derived_positions():
    N, K = 16, 256
    cases = {  # (n, k) -> (byte, shift) derived by hand from the layout rule
        (0, 0): (0, 0),      # lane 0, word 0, bit 0
        (0, 1): (2, 0),      # h = 1 -> bit 16
        (8, 0): (1, 0),      # a = 1 (row + 8) -> bit 8
        (0, 8): (0, 4),      # e = 1 (col + 8) -> bit 4
        (8, 9): (3, 4),      # a = 1, e = 1, h = 1 -> bit 28
        (1, 0): (64, 0),     # r = 1 -> lane 4
        (0, 2): (16, 0),     # c = 2 -> lane 1
        (0, 16): (4, 0),     # word 1
        (0, 64): (512, 0),   # sub-block 1
        (15, 255): (512 * 3 + 16 * 31 + 12 + 3, 4),
    }
    for (n, k), (byte, shift) in cases.items():
        q = np.zeros((N, K), np.uint8)
        q[n, k] = 0xB
        packed = oracle.pack_w4(q, np.zeros((N, 8), np.uint16), np.zeros((N, 8), np.uint8))
        nz = np.flatnonzero(packed)
        assert list(nz) == [byte], (n, k)
        assert packed[byte] == 0xB << shift, (n, k)
    # tile order: (row 16*9 + 3, k 256*2 + 5) sits in group 1, super-block 2,
    # row tile 1 of the group -> tile index (1*KB + 2)*8 + 1 with KB = 3
    N2, K2 = 300, 768
    q2 = np.zeros((N2, K2), np.uint8)
    q2[16 * 9 + 3, 256 * 2 + 5] = 0x7
    packed2 = oracle.pack_w4(q2, np.zeros((N2, K2 // 32), np.uint16), np.zeros((N2, K2 // 32), np.uint8))
    tile = ((1 * 3 + 2) * 8 + 1) * 2432
    # r = 3, c = 4 (col 5 = c + h with h = 1) -> lane 14, word 0, bit 16
    assert list(np.flatnonzero(packed2)) == [tile + 16 * 14 + 2]
    # scale of (row 9, group 5): r = 1, half = 1 -> 2048 + 128 + 16 + 4 + 2
    s = np.zeros((N, 8), np.uint16)
    s[9, 5] = 0x1234
    z = np.zeros((N, 8), np.uint8)
    z[9, 5] = 7
    packed = oracle.pack_w4(np.zeros((N, K), np.uint8), s, z)
    assert packed[2048 + 128 + 16 + 4 + 2] == 0x34 and packed[2048 + 128 + 16 + 4 + 3] == 0x12
    assert packed[2304 + 16 + 10 + 1] == 7
    assert np.count_nonzero(packed) == 3


# --------------------------------------------------------------------------
# W4A16 matmul
# --------------------------------------------------------------------------


def _quantized(N, K, seed):
    W = randn_bits((N, K), seed)
    q, s, z = oracle.quantize_w4(W, N, K)
    return W, q, s, z


def test_w4a16_exact_rational_brute_force_tiny():
    N, K, M = 3, 64, 2
    _, q, s, z = _quantized(N, K, 21)
    x = randn_bits((M, K), 22)
    out = oracle.w4a16(x, q, s, z)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(bits_to_float(x[m, k])) *
                        (int(q[n, k]) - int(z[n, k // 32])) *
                        Fraction(bits_to_float(s[n, k // 32])) for k in range(K))
            assert abs(Fraction(out[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 60)


def test_w4a16_one_hot_selects_a_dequantized_column():
    N, K = 40, 512
    _, q, s, z = _quantized(N, K, 31)
    for k in (0, 31, 32, 255, 256, 511):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80                                  # 1.0
        out = oracle.w4a16(x, q, s, z)[0]
        col = (q[:, k].astype(np.float64) - z[:, k // 32]) * oracle.bf16_bits_to_f64(s[:, k // 32])
        np.testing.assert_array_equal(out, col)


def test_w4a16_matches_library_matmul():
    N, K, M = 256, 768, 4
    _, q, s, z = _quantized(N, K, 41)
    x = randn_bits((M, K), 42)
    ref = oracle.bf16_bits_to_f64(x) @ oracle.dequant_w4(q, s, z).T
    np.testing.assert_allclose(oracle.w4a16(x, q, s, z), ref, rtol=1e-12, atol=1e-12)
    # a row window gives the same numbers
    np.testing.assert_allclose(oracle.w4a16(x, q, s, z, 16, 48), ref[:, 16:48], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# W4A8
# --------------------------------------------------------------------------


def test_act_quant_hand_derived():
    # one scale per (row, group of 32); K = 64 is two groups
    K = 64
    g_sx1 = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.0, -127.0] + [0.0] * 24   # sx = 1 exactly
    g_sx2 = [254.0, 1.0, 3.0, -1.0, 5.0, 0.0, -254.0, 2.0] + [0.0] * 24    # sx = 2: x/2 = .5 ties
    g_zero = [0.0] * 32                                                    # all zero -> sx = 0
    rows = [g_sx1 + g_sx2, g_zero + g_zero, g_zero + g_sx1]
    x = np.array([[float_to_bits(v) for v in r] for r in rows], np.uint16)
    xq, sx = oracle.act_quant(x, K)
    assert sx.shape == (3, 2)
    assert sx.tolist() == [[1.0, 2.0], [0.0, 0.0], [0.0, 1.0]]
    assert list(xq[0, :8]) == [127, 0, 2, 2, 0, -2, 3, -127]
    assert list(xq[0, 32:40]) == [127, 0, 2, 0, 2, 0, -127, 1]
    assert not xq[1].any()
    assert not xq[2, :32].any() and list(xq[2, 32:40]) == [127, 0, 2, 2, 0, -2, 3, -127]


def test_act_quant_scale_is_per_group():
    # a large value in one group leaves the codes of the others untouched
    K = 96
    base = randn_bits((1, K), 52)[0]
    big = base.copy()
    big[40] = float_to_bits(500.0)
    x = np.stack([base, big])
    xq, sx = oracle.act_quant(x, K)
    assert sx[1, 1] > 100 * sx[0, 1]                       # group 1 holds the outlier
    assert np.array_equal(xq[0, :32], xq[1, :32]) and np.array_equal(xq[0, 64:], xq[1, 64:])
    assert sx[0, 0] == sx[1, 0] and sx[0, 2] == sx[1, 2]


def test_act_quant_matches_exact_rounding_away_from_ties():
    M, K = 4, 4096
    x = randn_bits((M, K), 51)
    xq, sx = oracle.act_quant(x, K)
    xf = x.astype(np.uint32) << 16
    xf = xf.view(np.float32)
    amax = np.abs(xf).reshape(M, K // 32, 32).max(axis=2)
    # sx is the fp32 rounding of the group's absmax / 127
    assert np.array_equal(sx, (amax / np.float32(127)).astype(np.float32))
    near = 0
    for m in range(M):
        for k in range(0, K, 7):
            v = Fraction(float(xf[m, k])) / Fraction(float(sx[m, k // 32]))
            frac = v - int(v)
            if abs(abs(frac) - Fraction(1, 2)) < Fraction(1, 2 ** 16):
                near += 1
                continue
            assert xq[m, k] == max(-127, min(127, round(v)))
    assert near < 32   # of ~2300 sampled codes: almost all are checked exactly
    assert np.abs(xq).max() == 127


def test_w4a8_group_dots_exact_and_bounded():
    N, K, M = 48, 512, 3
    _, q, s, z = _quantized(N, K, 61)
    x = randn_bits((M, K), 62)
    xq, sx = oracle.act_quant(x, K)
    D = oracle.w4a8_group_dots(xq, q, z)
    qq = q.reshape(N, K // 32, 32).astype(np.int64) - z[:, :, None]
    ref = np.einsum("ngi,mgi->mng", qq, xq.reshape(M, K // 32, 32).astype(np.int64))
    np.testing.assert_array_equal(D, ref)
    assert np.abs(D).max() <= 32 * 15 * 127


def test_w4a8_reduces_to_w4a16_on_integer_activations():
    # x integer-valued with max |x| = 127 -> sx = 1 and xq = x exactly, so the
    # W4A8 result equals the W4A16 result of the same x.
    N, K, M = 64, 768, 2
    _, q, s, z = _quantized(N, K, 71)
    rng = np.random.default_rng(72)
    xi = rng.integers(-127, 128, (M, K))
    xi[:, 5::32] = 127      # every group reaches 127, so every group scale is 1
    x = np.array([[float_to_bits(float(v)) for v in row] for row in xi], np.uint16)
    xq, sx = oracle.act_quant(x, K)
    assert np.all(sx == 1.0) and np.array_equal(xq, xi)
    np.testing.assert_allclose(oracle.w4a8(xq, sx, q, s, z), oracle.w4a16(x, q, s, z),
                               rtol=1e-13, atol=1e-9)


def test_w4a8_precision_class_against_w4a16_gaussian():
    # "test_int4_quantized_gemm.py", Int4QuantizedGemmPrecisionTest:
    # mean |a8 - a16| / mean |a16| <= 0.02 on gaussian activations.
    N, K = 512, 6656
    _, q, s, z = _quantized(N, K, 81)
    for M in (1, 4):
        x = randn_bits((M, K), 82 + M)
        xq, sx = oracle.act_quant(x, K)
        a8 = oracle.w4a8(xq, sx, q, s, z)
        a16 = oracle.w4a16(x, q, s, z)
        assert np.abs(a8 - a16).mean() / np.abs(a16).mean() < 0.02


def test_w4a8_combination_is_the_sum_of_scaled_exact_group_dots():
    # out[m, n] = sum_g sx[m, g] * s[n, g] * D[m, n, g], D from an int64 einsum
    N, K, M = 40, 256, 3
    _, q, s, z = _quantized(N, K, 83)
    x = randn_bits((M, K), 84)
    xq, sx = oracle.act_quant(x, K)
    qq = q.reshape(N, K // 32, 32).astype(np.int64) - z[:, :, None]
    D = np.einsum("ngi,mgi->mng", qq, xq.reshape(M, K // 32, 32).astype(np.int64))
    sf = np.vectorize(bits_to_float)(s).astype(np.float64)    # [N, G], decoded here
    ref = np.einsum("mg,ng,mng->mn", sx.astype(np.float64), sf, D.astype(np.float64))
    np.testing.assert_allclose(oracle.w4a8(xq, sx, q, s, z), ref, rtol=1e-12, atol=1e-12)


def test_w4a8_outlier_precision_criteria():
    # "test_int4_quantized_gemm.py", Int4QuantizedGemmPrecisionTest,
    # _check_precision_case with the outlier activations of _activation
    # (channels 0, K/3, 2K/3, K-1 scaled by 50, 35, 25, 20): against the dense
    # product, mean error within 1.10x of W4A16's, mean |a8 - a16| / mean |a16|
    # <= 0.02, and max error within max(2, 0.02 max|dense|) of W4A16's.
    N, K = 256, 6656
    W = workloads.w4_weight(N, K, seed=85)
    q, s, z = oracle.quantize_w4(W, N, K)
    for M in (1, 4):
        x = workloads.outlier_activation(M, K, seed=86 + M)
        dense = (x.double() @ W.double().T).numpy()
        xq, sx = oracle.act_quant(x, K)
        a8 = oracle.w4a8(xq, sx, q, s, z)
        a16 = oracle.w4a16(x, q, s, z)
        e8, e16 = np.abs(a8 - dense), np.abs(a16 - dense)
        assert e8.mean() / e16.mean() <= 1.10
        assert np.abs(a8 - a16).mean() / np.abs(a16).mean() <= 0.02
        assert e8.max() <= e16.max() + max(2.0, 0.02 * np.abs(dense).max())


# --------------------------------------------------------------------------
# W4A8 with one activation scale per whole row (scale = absmax / 127)
# --------------------------------------------------------------------------


def test_act_quant_row_hand_derived():
    # one scale for the whole row: the row maximum 127 (in group 1) gives
    # sx = 1 exactly, so group 0's values round on their own
    # (0.5 -> 0, 1.5 -> 2, 2.5 -> 2: half to even) and a group of small
    # values is flattened to zero; max 254 gives sx = 2 (x / 2 = .5 ties);
    # an all-zero row gives sx = 0 and codes 0.
    K = 96
    r0 = ([0.5, 1.5, 2.5, -0.5, -1.5, 3.0, 0.0, -3.5] + [0.0] * 24
          + [127.0, -127.0] + [0.0] * 30
          + [0.25, -0.25, 0.375, 0.5] + [0.0] * 28)
    r1 = [254.0, 1.0, 3.0, -1.0, 5.0, 0.0, -254.0, 2.0] + [0.0] * 88
    r2 = [0.0] * K
    x = np.array([[float_to_bits(v) for v in r] for r in (r0, r1, r2)], np.uint16)
    xq, sx = oracle.act_quant_row(x, K)
    assert sx.shape == (3,) and sx.tolist() == [1.0, 2.0, 0.0]
    assert list(xq[0, :8]) == [0, 2, 2, 0, -2, 3, 0, -4]
    assert list(xq[0, 32:34]) == [127, -127]
    assert list(xq[0, 64:68]) == [0, 0, 0, 0]           # |v| <= 0.5 at sx = 1
    assert list(xq[1, :8]) == [127, 0, 2, 0, 2, 0, -127, 1]
    assert not xq[2].any()


def test_act_quant_row_matches_exact_rounding_away_from_ties():
    M, K = 3, 4096
    x = randn_bits((M, K), 151)
    xq, sx = oracle.act_quant_row(x, K)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(sx, (amax / np.float32(127)).astype(np.float32))
    near = 0
    for m in range(M):
        for k in range(0, K, 5):
            v = Fraction(float(xf[m, k])) / Fraction(float(sx[m]))
            if abs(abs(v - int(v)) - Fraction(1, 2)) < Fraction(1, 2 ** 16):
                near += 1
                continue
            assert xq[m, k] == max(-127, min(127, round(v)))
    assert near < 16
    assert (np.abs(xq).max(axis=1) == 127).all()        # every row reaches its maximum code


def test_act_quant_row_one_large_value_rescales_the_whole_row():
    # the opposite of the per-group rule: a large value anywhere changes the
    # scale, and so the codes, of every group of its row
    K = 96
    base = randn_bits((1, K), 152)[0]
    big = base.copy()
    big[40] = float_to_bits(500.0)
    xq, sx = oracle.act_quant_row(np.stack([base, big]), K)
    assert sx[1] > 50 * sx[0]
    assert not np.array_equal(xq[0, :32], xq[1, :32])
    assert not np.array_equal(xq[0, 64:], xq[1, 64:])


def test_act_quant_row_equals_per_group_when_every_group_has_the_row_max():
    # where every group of 32 holds the row's max |x|, the per-group scales all
    # equal the row scale, so both rules give the same scale and codes
    M, K = 2, 512
    x = randn_bits((M, K), 153)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    top = float(np.abs(xf).max()) * 2
    for m in range(M):
        for g in range(K // 32):
            x[m, 32 * g + (g * 7 + m) % 32] = float_to_bits(top if g % 2 else -top)
    xq_r, sx_r = oracle.act_quant_row(x, K)
    xq_g, sx_g = oracle.act_quant(x, K)
    assert np.array_equal(np.repeat(sx_r[:, None], K // 32, axis=1), sx_g)
    assert np.array_equal(xq_r, xq_g)


def test_w4a8_row_reduces_to_w4a16_on_integer_activations():
    # integer rows that reach 127: sx = 1 and xq = x, so per-row W4A8 is W4A16
    N, K, M = 64, 768, 3
    _, q, s, z = _quantized(N, K, 154)
    rng = np.random.default_rng(155)
    xi = rng.integers(-126, 127, (M, K))
    xi[:, 17] = 127
    x = np.array([[float_to_bits(float(v)) for v in row] for row in xi], np.uint16)
    xq, sx = oracle.act_quant_row(x, K)
    assert np.all(sx == 1.0) and np.array_equal(xq, xi)
    np.testing.assert_allclose(oracle.w4a8_row(xq, sx, q, s, z), oracle.w4a16(x, q, s, z),
                               rtol=1e-13, atol=1e-9)


def test_w4a8_row_combination_is_the_row_scale_times_the_scaled_group_dots():
    # out[m, n] = sx[m] * sum_g s[n, g] * D[m, n, g], D from an int64 einsum
    N, K, M = 40, 512, 4
    _, q, s, z = _quantized(N, K, 156)
    x = randn_bits((M, K), 157)
    xq, sx = oracle.act_quant_row(x, K)
    qq = q.reshape(N, K // 32, 32).astype(np.int64) - z[:, :, None]
    D = np.einsum("ngi,mgi->mng", qq, xq.reshape(M, K // 32, 32).astype(np.int64))
    sf = np.vectorize(bits_to_float)(s).astype(np.float64)
    ref = sx.astype(np.float64)[:, None] * np.einsum("ng,mng->mn", sf, D.astype(np.float64))
    np.testing.assert_allclose(oracle.w4a8_row(xq, sx, q, s, z), ref, rtol=1e-12, atol=1e-12)
    # and the per-group combination with the row scale broadcast to every group
    sxg = np.repeat(sx[:, None], K // 32, axis=1)
    np.testing.assert_allclose(oracle.w4a8(xq, sxg, q, s, z), ref, rtol=1e-12, atol=1e-12)


def test_w4a8_row_precision_class_against_w4a16_gaussian():
    # "test_int4_quantized_gemm.py", Int4QuantizedGemmPrecisionTest: on
    # gaussian activations mean |a8 - a16| / mean |a16| <= 0.02 (one scale
    # per row suffices there; the outlier case needs the per-group rule).
    N, K = 512, 6656
    _, q, s, z = _quantized(N, K, 158)
    for M in (1, 4):
        x = randn_bits((M, K), 159 + M)
        xq, sx = oracle.act_quant_row(x, K)
        a8 = oracle.w4a8_row(xq, sx, q, s, z)
        a16 = oracle.w4a16(x, q, s, z)
        assert np.abs(a8 - a16).mean() / np.abs(a16).mean() < 0.02


# --------------------------------------------------------------------------
# W8
# --------------------------------------------------------------------------


def test_w8_all_ones_gives_integer_row_sums_times_scale():
    W, scales, _ = workloads.w8_inputs(N=64, K=512, M=1, seed=91)
    Wn = W.numpy()
    x = np.full((1, 512), 0x3F80, np.uint16)
    out = oracle.w8(x, Wn, scales)
    sums = Wn.astype(np.int64).sum(axis=1).astype(np.float64)
    sc = oracle.bf16_bits_to_f64(scales.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(out[0], sums * sc)


def test_w8_matches_library_matmul():
    W, scales, x = workloads.w8_inputs(N=128, K=1024, M=3, seed=92)
    ref = (x.double() @ W.double().T * scales.double()).numpy()
    np.testing.assert_allclose(oracle.w8(x, W.numpy(), scales), ref, rtol=1e-12, atol=1e-9)


# --------------------------------------------------------------------------
# Compact metadata: uint8 scale / zero codes on per-row fp16 steps
# ("test_int4_quantized_gemm.py", CudaCoalescedInt4Tensor: scale and
# zero_point uint8 [N, K/32], scale_step and zero_point_step float16 [N, 1];
# read as code x step for both)
# --------------------------------------------------------------------------

_FP16 = None


def positive_fp16():
    """Every finite positive fp16 as (value, bits), sorted (by enumeration)."""
    global _FP16
    if _FP16 is None:
        bits = np.arange(1, 0x7C00, dtype=np.uint16)
        vals = bits.view(np.float16).astype(np.float64)
        _FP16 = (vals, bits)
    return _FP16


def ru_fp16_search(v):
    """Smallest fp16 >= v > 0, by search over every fp16 number."""
    vals, bits = positive_fp16()
    i = int(np.searchsorted(vals, v, side="left"))
    return float(vals[i]), int(bits[i])


def brute_quant_row_c(wbits):
    """A restatement of the compact quantizer on one row, from its definition:
    IEEE fp64 steps (Python floats), fp16 rounding up by search, round half
    to even."""
    vals = [bits_to_float(b) for b in wbits]
    G = len(vals) // GROUP
    groups = [vals[GROUP * g:GROUP * (g + 1)] for g in range(G)]

    def sstar(gv):
        mx, mn = max(gv), min(gv)
        if mx == mn:
            return 1.0 if mx == 0 else abs(mx) / 15.0
        return (mx - mn) / 15.0
    ds, dsb = ru_fp16_search(max(sstar(gv) for gv in groups) / 255.0)
    sc = [min(255, max(1, int(np.ceil(sstar(gv) / ds)))) for gv in groups]
    zs = [min(15.0, max(0.0, -min(gv) / (c * ds))) for gv, c in zip(groups, sc)]
    if max(zs) > 0:
        dz, dzb = ru_fp16_search(max(zs) / 255.0)
    else:
        dz, dzb = 1.0, 0x3C00
    zc = [min(255, round(z / dz)) for z in zs]
    q = []
    for gv, c, zz in zip(groups, sc, zc):
        s, z = c * ds, zz * dz
        q += [min(15, max(0, round(v / s + z))) for v in gv]
    return q, sc, zc, (dsb, dzb)


@pytest.mark.parametrize("name", ["randn", "scaled", "constant", "zeros", "same_sign", "tiny", "big"])
def test_compact_quantizer_matches_restatement(name):
    K = 256
    rng = np.random.default_rng(170 + len(name))
    v = rng.standard_normal((4, K))
    if name == "scaled":
        v *= 2.0 ** rng.integers(-6, 7, (4, K // GROUP)).repeat(GROUP, axis=1)
    elif name == "constant":
        v[:, :GROUP] = 3.0
        v[:, GROUP:2 * GROUP] = -0.5
    elif name == "zeros":
        v[:, :3 * GROUP] = 0.0
    elif name == "same_sign":
        v[:, :GROUP] = np.abs(v[:, :GROUP]) + 1.0
        v[:, GROUP:2 * GROUP] = -np.abs(v[:, GROUP:2 * GROUP]) - 2.0
    elif name == "tiny":
        v *= 1e-3
    elif name == "big":
        v *= 300.0
    W = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16)
    wb = W.view(torch.int16).numpy().view(np.uint16)
    q, sc, zc, st = oracle.quantize_w4c(W, 4, K)
    for n in range(4):
        bq, bsc, bzc, bst = brute_quant_row_c(wb[n])
        assert list(q[n]) == bq, (name, n)
        assert list(sc[n]) == bsc and list(zc[n]) == bzc, (name, n)
        assert tuple(int(x) for x in st[n]) == bst, (name, n)


def test_compact_quantizer_hand_derived_row():
    # one row, two groups: group 0 spans [-1, 2] (s* = 0.2), group 1 spans
    # [-0.5, 1] (s* = 0.1); ds = RU_fp16(0.2 / 255): 0.2/255 = 7.84e-4 lies
    # in [2^-11, 2^-10), fp16 spacing 2^-21 there, so ds = 1645 * 2^-21;
    # sc = ceil(s* / ds) = 255 and 128
    K = 64
    g0 = [-1.0, 2.0] + [0.5] * 30
    g1 = [-0.5, 1.0] + [0.25] * 30
    x = np.array([[float_to_bits(v) for v in g0 + g1]], np.uint16)
    q, sc, zc, st = oracle.quantize_w4c(x, 1, K)
    ds = float(np.array([st[0, 0]], np.uint16).view(np.float16)[0])
    assert ds == 1645 * 2.0 ** -21
    assert list(sc[0]) == [255, 128]
    s0, s1 = 255 * ds, 128 * ds
    assert s0 >= 0.2 and s1 >= 0.1
    # the codes of the ends of each group land on 0 and 15 or next to them
    assert q[0, 0] == 0 and q[0, 32] == 0
    assert q[0, 1] == 15 and q[0, 33] == 15


def test_compact_quantizer_invariants_on_randn():
    N, K = 256, 1024
    W = workloads.w4_weight(N, K, seed=171)
    q, sc, zc, st = oracle.quantize_w4c(W, N, K)
    assert q.max() <= 15 and sc.min() >= 1
    wh = oracle.dequant_w4c(q, sc, zc, st)
    w = W.double().numpy()
    ds = st[:, 0].view(np.float16).astype(np.float64)
    s = sc.astype(np.float64) * ds[:, None]                       # [N, G]
    g = w.reshape(N, K // GROUP, GROUP)
    sstar = (g.max(axis=2) - g.min(axis=2)) / 15.0
    assert (s >= sstar).all()                                     # the scale code rounds up
    vals, _ = positive_fp16()
    smax = sstar.max(axis=1) / 255.0
    assert (ds >= smax).all()
    below = vals[np.searchsorted(vals, ds) - 1]                   # the next smaller fp16
    assert (below < smax).all()                                   # ds is the least such
    straddle = (g.min(axis=2) <= 0) & (g.max(axis=2) >= 0)
    err = np.abs(w - wh).reshape(N, K // GROUP, GROUP).max(axis=2)
    assert (err[straddle] <= s[straddle] / 2 * (1 + 1e-12)).all()


def test_compact_zero_group_dequantizes_to_zero():
    K = 64
    x = np.zeros((1, K), np.uint16)
    x[0, 32:] = [float_to_bits(v / 16.0) for v in range(-16, 16)]
    q, sc, zc, st = oracle.quantize_w4c(x, 1, K)
    assert (oracle.dequant_w4c(q, sc, zc, st)[0, :32] == 0).all()


def decode_layout_c(packed, N, K):
    """Independent decoder of the compact layout (nibbles as the standard
    layout, 2304-byte tiles, code pairs, steps after the tiles)."""
    KB, G = K // 256, K // GROUP
    Np = (N + 127) // 128 * 128
    tiles = packed[: (Np // 128) * 8 * KB * 2304].reshape(Np // 128, KB, 8, 2304)
    q = np.zeros((Np, K), np.uint8)
    sc = np.zeros((Np, G), np.uint8)
    zc = np.zeros((Np, G), np.uint8)
    for gp in range(Np // 128):
        for b in range(KB):
            for t in range(8):
                tile = tiles[gp, b, t]
                rows = gp * 128 + t * 16
                codes = tile[:2048].reshape(4, 32, 4, 4)      # [sub-block][lane][word][byte]
                words = codes.copy().view(np.uint32).reshape(4, 32, 4)
                for l in range(32):
                    r, c = l // 4, 2 * (l % 4)
                    for sbk in range(4):
                        for j in range(4):
                            w = int(words[sbk, l, j])
                            for a in range(2):
                                for e in range(2):
                                    for h in range(2):
                                        q[rows + r + 8 * a, 256 * b + 64 * sbk + 16 * j + c + 8 * e + h] = \
                                            (w >> (8 * a + 4 * e + 16 * h)) & 0xF
                for r in range(8):
                    for gg in range(8):
                        for half in range(2):
                            sc[rows + r + 8 * half, 8 * b + gg] = tile[2048 + 16 * r + 2 * gg + half]
                            zc[rows + r + 8 * half, 8 * b + gg] = tile[2176 + 16 * r + 2 * gg + half]
    steps = packed[(Np // 128) * 8 * KB * 2304:].view(np.uint16).reshape(Np, 2)
    return q[:N], sc[:N], zc[:N], steps[:N]


@pytest.mark.parametrize("N,K", [(16, 256), (130, 512)])
def test_compact_pack_matches_independent_decoder(N, K):
    W = workloads.w4_weight(N, K, seed=172)
    q, sc, zc, st = oracle.quantize_w4c(W, N, K)
    packed = oracle.pack_w4c(q, sc, zc, st)
    assert packed.size == oracle.packed_bytes_c(N, K) == \
        (N + 127) // 128 * (8 * (K // 256) * 2304 + 128 * 4)
    dq, dsc, dzc, dst = decode_layout_c(packed, N, K)
    assert np.array_equal(dq, q) and np.array_equal(dsc, sc) and np.array_equal(dzc, zc)
    assert np.array_equal(dst, st)
    uq, usc, uzc, ust = oracle.unpack_w4c(packed, N, K)
    assert np.array_equal(uq, q) and np.array_equal(usc, sc) and np.array_equal(ust, st)


def test_compact_pack_hand_derived_positions():
    # row 9 = tile 0 row r = 1 of its upper half, group 3 of super-block 0:
    # scale code at 2048 + 16 * 1 + 2 * 3 + 1 = 2071, zero code at 2199;
    # row 130 (tile group 1, tile 0, row 2), K = 512: its steps at
    # 2 * 8 * 2 * 2304 + 4 * 130
    N, K = 140, 512
    q = np.zeros((N, K), np.uint8)
    sc = np.ones((N, K // GROUP), np.uint8)
    zc = np.zeros((N, K // GROUP), np.uint8)
    st = np.zeros((N, 2), np.uint16)
    sc[9, 3], zc[9, 3] = 77, 99
    st[130] = (0x1234, 0x5678)
    p = oracle.pack_w4c(q, sc, zc, st)
    assert p[2071] == 77 and p[2199] == 99
    off = 2 * 8 * 2 * 2304 + 4 * 130
    assert p[off:off + 4].tobytes() == bytes([0x34, 0x12, 0x78, 0x56])


def test_compact_w4a16_matches_library_matmul_and_one_hot():
    N, K, M = 96, 512, 3
    W = workloads.w4_weight(N, K, seed=173)
    q, sc, zc, st = oracle.quantize_w4c(W, N, K)
    wh = oracle.dequant_w4c(q, sc, zc, st)
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(174)).to(torch.bfloat16)
    ref = x.double().numpy() @ wh.T
    np.testing.assert_allclose(oracle.w4a16c(x, q, sc, zc, st), ref, rtol=1e-12, atol=1e-12)
    e = torch.zeros(1, K, dtype=torch.bfloat16)
    e[0, 77] = 1.0
    np.testing.assert_array_equal(oracle.w4a16c(e, q, sc, zc, st)[0], wh[:, 77])
