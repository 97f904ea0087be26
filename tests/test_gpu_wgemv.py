"""GPU parity of the weight-only quantised decode GEMV (INT4 groups of 128;
e4m3 with a row scale as the comparison).

Quantiser output (codes in the slice layout and scales) bit-exact against the
oracle; y within a bound derived from the arithmetic.  Up to 4 tokens the
weights enter the tensor cores as exact f16 (an INT4 code, 16 times one, or an
e4m3 value) and the activations as f16 copies of the bf16 values times a power
of two (per token and K chunk, largest |x| taken into [2^14, 2^15); for INT4
every other pair divided by 16), exact except for values that fall below 2^-14
after scaling, which round to f16 subnormals with an error under 2^-25 of the
scaled unit, i.e. 2^-35 max|x| before scaling; from 5 tokens on, both enter as
exact bf16.  Every other product is exact in fp32.  The
tensor cores sum 16 per step in fp32, a group's steps are summed in fp32 (two
chains, then added), scaled once, and the K/128 group sums (and the split-K
chunks) are added in fp32: at most (8 + 2 + K/128 + 2) roundings of relative
size 2^-24 (2^-23 if the tensor core truncates) on a sum bounded by
sum_k |w x|:
|y - y_ref| <= 4 (16 + K/128) 2^-24 sum_k |w_k x_k|  (plus a 2^-30 max|x|
sum_k |w_k| allowance for the subnormal activations and for results near the
bottom of the fp32 range).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300 import (FpkError, fpk_w4_gemv, fpk_w4_quantize, fpk_w8_gemv,
                                fpk_w8_quantize)
from fp8_paged_kv_gb300.pool import to_device
from workloads import bf16_bits, bf16_to_f32

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _weights(seed, N, K, specials=False):
    g = np.random.default_rng(seed)
    w = (g.standard_normal((N, K)) * 0.02).astype(np.float32)
    w *= (10.0 ** g.uniform(-2, 2, size=(N, 1))).astype(np.float32)
    w[:, g.integers(0, K, size=max(1, K // 500))] *= 30          # outlier columns
    if specials:
        w[0, :128] = 0.0                                           # an all-zero group
        w[1, 5], w[2, 7], w[3, 9] = np.inf, -np.inf, np.nan        # non-finite weights (INT4: code 0)
    return bf16_bits(w)


def _gpu_w4(wb):
    N, K = wb.shape
    codes = torch.empty(N * K // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(N, K // 128, dtype=torch.bfloat16, device=DEV)
    fpk_w4_quantize(to_device(wb, DEV), codes, scales)
    return codes, scales


def _gpu_w8(wb):
    N, K = wb.shape
    codes = torch.empty(N * K, dtype=torch.uint8, device=DEV)
    rs = torch.empty(N, dtype=torch.float32, device=DEV)
    fpk_w8_quantize(to_device(wb, DEV), codes, rs)
    return codes, rs


@pytest.mark.parametrize("N,K", [(16, 128), (96, 384), (256, 2176)])
def test_w4_quantiser_bit_exact(N, K):
    wb = _weights(N + K, N, K, specials=True)
    codes, scales = _gpu_w4(wb)
    q, sc = oracle.w4_quantize(wb)
    assert np.array_equal(codes.cpu().numpy(), oracle.w4_pack(q))
    assert np.array_equal(scales.view(torch.int16).cpu().numpy().view(np.uint16), sc)


@pytest.mark.parametrize("N,K", [(16, 128), (96, 384), (256, 2176)])
def test_w8_quantiser_bit_exact(N, K):
    wb = _weights(N + K + 1, N, K)
    codes, rs = _gpu_w8(wb)
    c, r = oracle.w8_quantize(wb)
    assert np.array_equal(rs.cpu().numpy(), r)
    assert np.array_equal(codes.cpu().numpy(), oracle.w8_pack(c))


def _tol(wd, x, K):
    xmax = np.abs(x).max(axis=1, keepdims=True)
    return (4 * (16 + K / 128) * 2.0 ** -24 * (np.abs(x) @ np.abs(wd).T)
            + 2.0 ** -30 * xmax * np.abs(wd).sum(axis=1)[None, :] + 1e-30)


@pytest.mark.parametrize("B", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("N,K", [(16, 128), (144, 2048), (64, 2176), (32, 4352), (48, 8192)])
def test_w4_gemv_within_bound(B, N, K):
    wb = _weights(7 * B + K, N, K, specials=True)
    g = np.random.default_rng(B + N)
    xb = bf16_bits(g.standard_normal((B, K)).astype(np.float32))
    codes, scales = _gpu_w4(wb)
    y = torch.full((B, N), float("nan"), device=DEV)
    fpk_w4_gemv(to_device(xb, DEV), codes, scales, y)
    q, sc = oracle.w4_quantize(wb)
    ref = oracle.w4_gemv(xb, q, sc)
    wd = q.astype(np.float64) * np.repeat(bf16_to_f32(sc).astype(np.float64), 128, axis=1)
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= _tol(wd, bf16_to_f32(xb).astype(np.float64), K))


@pytest.mark.parametrize("B", [1, 8, 16])
@pytest.mark.parametrize("N,K", [(16, 128), (144, 2048), (32, 4352)])
def test_w8_gemv_within_bound(B, N, K):
    wb = _weights(11 * B + K, N, K)
    g = np.random.default_rng(B + N + 1)
    xb = bf16_bits(g.standard_normal((B, K)).astype(np.float32))
    codes, rs = _gpu_w8(wb)
    y = torch.full((B, N), float("nan"), device=DEV)
    fpk_w8_gemv(to_device(xb, DEV), codes, rs, y)
    c, r = oracle.w8_quantize(wb)
    ref = oracle.w8_gemv(xb, c, r)
    wd = oracle.e4m3_decode(c) * r.astype(np.float64)[:, None]
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= _tol(wd, bf16_to_f32(xb).astype(np.float64), K))


@pytest.mark.parametrize("w4", [True, False])
def test_gemv_activation_range(w4):
    # rows of very different magnitude (far beyond the f16 range) and a zero row
    N, K, B = 64, 2176, 4
    wb = _weights(3, N, K)
    g = np.random.default_rng(9)
    x = g.standard_normal((B, K)).astype(np.float32)
    x[0] *= 1e20
    x[1] *= 1e-20
    x[2] = 0
    x[3, :100] *= 1e5
    xb = bf16_bits(x)
    y = torch.full((B, N), float("nan"), device=DEV)
    if w4:
        codes, scales = _gpu_w4(wb)
        fpk_w4_gemv(to_device(xb, DEV), codes, scales, y)
        q, sc = oracle.w4_quantize(wb)
        ref = oracle.w4_gemv(xb, q, sc)
        wd = q.astype(np.float64) * np.repeat(bf16_to_f32(sc).astype(np.float64), 128, axis=1)
    else:
        codes, rs = _gpu_w8(wb)
        fpk_w8_gemv(to_device(xb, DEV), codes, rs, y)
        c, r = oracle.w8_quantize(wb)
        ref = oracle.w8_gemv(xb, c, r)
        wd = oracle.e4m3_decode(c) * r.astype(np.float64)[:, None]
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)) and not got[2].any()
    assert np.all(np.abs(got - ref) <= _tol(wd, bf16_to_f32(xb).astype(np.float64), K))


def test_gemv_rejects_unsupported_shapes():
    wb = _weights(1, 16, 128)
    codes, scales = _gpu_w4(wb)
    x = to_device(bf16_bits(np.ones((17, 128), np.float32)), DEV)
    y = torch.empty(17, 16, device=DEV)
    with pytest.raises(FpkError):
        fpk_w4_gemv(x, codes, scales, y)                    # more than 16 decode tokens
    w_bad = to_device(bf16_bits(np.ones((24, 128), np.float32)), DEV)
    with pytest.raises(FpkError):
        fpk_w4_quantize(w_bad, torch.empty(24 * 64, dtype=torch.uint8, device=DEV),
                        torch.empty(24, 1, dtype=torch.bfloat16, device=DEV))   # N not a multiple of 16
