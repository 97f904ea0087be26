"""Pins of the oracle's weight-only quantisation and GEMV (the pages' second
technique: "La compressione dei pesi GLM modifica il compromesso tra le fasi",
remio.ai -- INT4 weights for decode, FP8 as the comparison).

* closed forms: weights that are exactly q * s with s a power of two and one
  |q| = 7 in the group come back as exactly (q, s); an all-zero group has
  s = 0 and q = 0; non-finite weights code to 0;
* the rounding bound |w - q s| <= s/2 inside the clamp range, and codes that
  are nearest integers (ties to even) of w / s;
* the e4m3 weights equal the cache quantiser's codes for the row's scale;
* GEMV against numpy's matmul (a library routine) on the dequantised weights;
* the slice layouts against an inverse written from the header's text.
"""
import numpy as np
import pytest

import oracle
from workloads import bf16_bits, bf16_to_f32


def _rand_w(seed, N, K, spread=True):
    g = np.random.default_rng(seed)
    w = g.standard_normal((N, K)).astype(np.float32)
    if spread:
        w *= (10.0 ** g.uniform(-3, 3, size=(N, 1))).astype(np.float32)
    return bf16_bits(w)


def test_w4_exact_weights_round_trip():
    g = np.random.default_rng(1)
    N, K = 32, 256
    q = g.integers(-7, 8, size=(N, K)).astype(np.int8)
    q[:, ::128] = 7 * np.where(g.random((N, K // 128)) < 0.5, 1, -1)   # a |q| = 7 in every group
    e = g.integers(-20, 20, size=(N, K // 128))
    s = (2.0 ** e).astype(np.float32)
    w = (q.astype(np.float32).reshape(N, K // 128, 128) * s[:, :, None]).reshape(N, K)
    q2, sc = oracle.w4_quantize(bf16_bits(w))
    assert np.array_equal(q2, q)
    assert np.array_equal(bf16_to_f32(sc), s)


def test_w4_zero_group_and_non_finite():
    w = np.zeros((16, 256), np.float32)
    w[3, 130:140] = [1, -2, 3, np.inf, -np.inf, np.nan, 0.5, 7, 0, 0]
    q, sc = oracle.w4_quantize(bf16_bits(w))
    assert not q[:, :128].any() and not bf16_to_f32(sc[:, 0]).any()      # all-zero groups: s = 0, q = 0
    s = bf16_to_f32(sc[3, 1])
    assert s == np.float32(bf16_to_f32(bf16_bits(np.array([7 / 7], np.float32)))[0])
    assert q[3, 133] == 0 and q[3, 134] == 0 and q[3, 135] == 0          # +inf, -inf, NaN -> 0
    assert q[3, 137] == 7 and q[3, 130] == 1 and q[3, 131] == -2


@pytest.mark.parametrize("seed", range(4))
def test_w4_rounding_bound_and_nearest(seed):
    wb = _rand_w(seed, 48, 384)
    q, sc = oracle.w4_quantize(wb)
    w = bf16_to_f32(wb).astype(np.float64).reshape(48, 3, 128)
    s = bf16_to_f32(sc).astype(np.float64)[:, :, None]
    qq = q.astype(np.float64).reshape(48, 3, 128)
    r = w / s
    assert np.all(np.abs(r) <= 7.0 * 1.01)             # amax / s ~ 7 (s is amax/7 rounded to bf16)
    assert np.all(np.abs(w - qq * s) <= s / 2 * (1 + 1e-6))
    # the nearest integer, ties to even (numpy's rint), of the fp32 quotient
    r32 = (bf16_to_f32(wb).reshape(48, 3, 128) / bf16_to_f32(sc)[:, :, None]).astype(np.float32)
    assert np.array_equal(qq, np.clip(np.rint(r32), -8, 7))


def test_w8_matches_cache_quantiser():
    wb = _rand_w(7, 16, 512)
    c, r = oracle.w8_quantize(wb)
    w = bf16_to_f32(wb)
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(r, (amax / np.float32(448)).astype(np.float32))
    for n in range(16):
        assert np.array_equal(c[n], oracle.quantize_bf16(wb[n], r[n]))
    dec = oracle.e4m3_decode(c) * r[:, None]
    assert np.all(np.abs(dec - w) <= np.abs(w) * 2.0 ** -4 + r[:, None] * 2.0 ** -10)


@pytest.mark.parametrize("B", [1, 5, 16])
def test_gemv_equals_numpy_matmul(B):
    g = np.random.default_rng(B)
    N, K = 48, 384
    wb = _rand_w(10 + B, N, K)
    xb = bf16_bits(g.standard_normal((B, K)).astype(np.float32))
    x = bf16_to_f32(xb).astype(np.float64)
    q, sc = oracle.w4_quantize(wb)
    wd = q.astype(np.float64) * np.repeat(bf16_to_f32(sc).astype(np.float64), 128, axis=1)
    ref = x @ wd.T
    y = oracle.w4_gemv(xb, q, sc)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    c, r = oracle.w8_quantize(wb)
    wd8 = oracle.e4m3_decode(c) * r.astype(np.float64)[:, None]
    y8 = oracle.w8_gemv(xb, c, r)
    ref8 = x @ wd8.T
    assert np.allclose(y8, ref8, rtol=1e-12, atol=1e-12 * np.abs(ref8).max())


def _w4_unpack(packed, N, K):
    """The INT4 slice layout read back from the header's description."""
    G = K // 128
    out = np.zeros((N, K), np.int8)
    b = packed.reshape(N // 16, G, 2, 32, 4, 4)            # slice, group, h, lane, word, byte
    for p in range(8):
        nib = (b[..., p // 2] >> (4 * (p & 1))) & 0xF       # [s, g, h, l, u]
        for u in range(4):
            v = 2 * u + ((p >> 1) & 1)
            i = 2 * (p & 1) + (p >> 2)
            for l in range(32):
                rows = 16 * np.arange(N // 16)[:, None, None] + 8 * np.arange(2)[None, None, :] + l // 4
                ks = 128 * np.arange(G)[None, :, None] + 16 * v + 4 * (l % 4) + i
                out[np.broadcast_to(rows, (N // 16, G, 2)), np.broadcast_to(ks, (N // 16, G, 2))] = \
                    nib[:, :, :, l, u].astype(np.int8) - 8
    return out


def _w8_unpack(packed, N, K):
    G = K // 128
    out = np.zeros((N, K), np.uint8)
    b = packed.reshape(N // 16, G, 2, 2, 32, 16)           # slice, group, h, c, lane, byte
    for c in range(2):
        for l in range(32):
            for bb in range(16):
                rows = 16 * np.arange(N // 16)[:, None, None] + 8 * np.arange(2)[None, None, :] + l // 4
                ks = 128 * np.arange(G)[None, :, None] + 16 * (4 * c + bb // 4) + 4 * (l % 4) + bb % 4
                out[np.broadcast_to(rows, (N // 16, G, 2)), np.broadcast_to(ks, (N // 16, G, 2))] = \
                    b[:, :, :, c, l, bb]
    return out


def test_slice_layouts_are_the_documented_permutations():
    g = np.random.default_rng(3)
    N, K = 32, 256
    q = g.integers(-8, 8, size=(N, K)).astype(np.int8)
    assert np.array_equal(_w4_unpack(oracle.w4_pack(q), N, K), q)
    c = g.integers(0, 256, size=(N, K)).astype(np.uint8)
    assert np.array_equal(_w8_unpack(oracle.w8_pack(c), N, K), c)
    # a permutation: distinct inputs stay distinct, byte counts are as documented
    assert oracle.w4_pack(q).size == N * K // 2 and oracle.w8_pack(c).size == N * K
