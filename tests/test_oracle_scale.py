"""Pins of the oracle's per-tensor e4m3 scale (amax / 448 over finite values).

The Cloudflare write-up names the cache format, FP8 e4m3, and nothing finer
("Cosa ha cambiato Cloudflare per Kimi e GLM", remio.ai); the scale reading is
one fp32 scale per tensor mapping the tensor's largest finite magnitude to the
largest finite e4m3 value, 448.  The pins:

* numpy's own max of |x| over the finite values, divided in float32;
* closed forms: amax = 448 * 2^k gives exactly 2^k; an all-zero or empty
  tensor gives 1;
* invariances: permutation, sign flips, and added infinities / NaNs leave the
  scale unchanged;
* the defining property: the largest element quantises to the largest code
  (0x7E, or 0xFE when negative) and no element saturates past it.
"""
import numpy as np
import pytest

import oracle
from workloads import bf16_bits, bf16_to_f32

INF_BITS, NINF_BITS, NAN_BITS = np.uint16(0x7F80), np.uint16(0xFF80), np.uint16(0x7FC0)


def _numpy_scale(bits: np.ndarray) -> np.float32:
    x = bf16_to_f32(bits)
    x = x[np.isfinite(x)]
    amax = np.max(np.abs(x)) if x.size else np.float32(0)
    return np.float32(1) if amax == 0 else np.float32(amax) / np.float32(448)


@pytest.mark.parametrize("seed", range(6))
def test_matches_numpy_max(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 5000))
    x = g.standard_normal(n).astype(np.float32) * np.float32(10.0 ** g.uniform(-30, 30))
    bits = bf16_bits(x)
    assert oracle.amax_scale_bf16(bits) == _numpy_scale(bits)


@pytest.mark.parametrize("k", [-40, -7, -1, 0, 1, 5, 20])
def test_power_of_two_closed_form(k):
    g = np.random.default_rng(k + 100)
    amax = np.float32(448.0) * np.float32(2.0) ** k
    x = (g.uniform(-1, 1, 300) * amax * 0.9).astype(np.float32)
    x[17] = -amax  # the largest magnitude, negative
    s = oracle.amax_scale_bf16(bf16_bits(x))
    assert s == np.float32(2.0) ** k


def test_zero_and_empty_give_one():
    assert oracle.amax_scale_bf16(np.zeros(10, np.uint16)) == 1.0
    assert oracle.amax_scale_bf16(np.array([0x8000] * 4, np.uint16)) == 1.0  # -0
    assert oracle.amax_scale_bf16(np.zeros(0, np.uint16)) == 1.0
    # only non-finite values: nothing to scale
    assert oracle.amax_scale_bf16(np.array([INF_BITS, NAN_BITS, NINF_BITS], np.uint16)) == 1.0


def test_invariances():
    g = np.random.default_rng(7)
    bits = bf16_bits(g.standard_normal(4096).astype(np.float32) * 3)
    s = oracle.amax_scale_bf16(bits)
    assert oracle.amax_scale_bf16(g.permutation(bits)) == s
    assert oracle.amax_scale_bf16(bits ^ np.uint16(0x8000)) == s
    noisy = np.concatenate([bits, np.array([INF_BITS, NINF_BITS, NAN_BITS, 0xFFC1], np.uint16)])
    assert oracle.amax_scale_bf16(g.permutation(noisy)) == s


@pytest.mark.parametrize("seed", range(4))
def test_largest_element_maps_to_largest_code(seed):
    g = np.random.default_rng(seed + 20)
    bits = bf16_bits((g.standard_normal(2000) * 10.0 ** g.uniform(-5, 5)).astype(np.float32))
    s = oracle.amax_scale_bf16(bits)
    codes = oracle.quantize_bf16(bits, s)
    i = int(np.argmax(np.abs(bf16_to_f32(bits))))
    assert codes[i] & 0x7F == 0x7E
    # every other code decodes to at most 448 in magnitude
    vals = np.abs(oracle.e4m3_decode(codes))
    assert vals.max() == 448.0
