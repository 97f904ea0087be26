"""Pins of the oracle's e4m3 codec against things other than itself.

* closed-form anchors from the OCP E4M3 definition (tests/golden/e4m3_anchors.txt);
* PyTorch's float8_e4m3fn type as an independent library decode (all 256
  codes) and, inside the finite range, an independent library encode;
* a brute-force nearest-value search with ties to the even code;
* round trip of every code, midpoint rounding, monotonicity;
* the fp32 division that defines the quantiser input, done by numpy.

The cache format is named "FP8 e4m3" in the Cloudflare write-up pages
(section "Cosa ha cambiato Cloudflare per Kimi e GLM" of the Italian edition).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, bf16_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_anchors.txt")


def _parse_value(tok: str) -> np.float32:
    t = tok.lower()
    if t in ("inf", "+inf"):
        return np.float32(np.inf)
    if t == "-inf":
        return np.float32(-np.inf)
    if t == "nan":
        return np.float32(np.nan)
    if "0x" in t:
        return np.float32(float.fromhex(t))
    return np.float32(float(t))


def _anchors():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v, c = line.split()[:2]
            rows.append((_parse_value(v), int(c, 16), line))
    return rows


def test_anchor_values_encode():
    rows = _anchors()
    assert len(rows) >= 25
    x = np.array([r[0] for r in rows], np.float32)
    got = oracle.e4m3_encode(x)
    for (v, code, line), g in zip(rows, got):
        assert g == code, f"{line}: got 0x{g:02x}"


def test_anchor_values_decode_exact():
    for v, code, line in _anchors():
        if math.isfinite(v) and abs(v) <= 448 and oracle.e4m3_encode(np.array([v]))[0] == code:
            d = oracle.e4m3_decode(np.array([code], np.uint8))[0]
            # exact representable anchors decode to themselves
            if float(v) in (1.0, 1.125, -1.0, 448.0, -448.0, 2**-6, 2**-9, 256.0, 384.0, 7 * 2**-9):
                assert d == float(v), line


def test_decode_matches_torch_float8_e4m3fn_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_o, nan_l = np.isnan(ours), np.isnan(lib)
    assert (nan_o == nan_l).all()
    assert sorted(np.flatnonzero(nan_o)) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan_o], lib[~nan_l])
    # signed zeros
    assert math.copysign(1.0, ours[0x80]) == -1.0 and ours[0x00] == 0.0


def test_roundtrip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(vals.astype(np.float32))
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert back[c] == 0x7F
        else:
            assert back[c] == c, hex(c)


def test_monotone_and_distinct():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(pos) > 0).all()
    assert pos[-1] == 448.0 and pos[1] == 2.0**-9


def test_midpoints_round_to_even_code():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2          # exact in fp32
        want = c if c % 2 == 0 else c + 1
        for sgn in (1, -1):
            got = oracle.e4m3_encode(np.array([sgn * mid], np.float32))[0]
            assert got == (want | (0x80 if sgn < 0 else 0)), (c, lo, hi)
        above = np.nextafter(mid, np.float32(np.inf))
        below = np.nextafter(mid, np.float32(0))
        assert oracle.e4m3_encode(np.array([above], np.float32))[0] == c + 1
        assert oracle.e4m3_encode(np.array([below], np.float32))[0] == c


def _brute_force_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search; ties to the even code."""
    table = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    out = np.empty(x.shape, np.uint8)
    for i, v in enumerate(x.astype(np.float64)):
        if np.isnan(v):
            out[i] = 0x7F
            continue
        a = min(abs(v), 448.0)      # saturation
        dist = np.abs(table - a)
        best = np.flatnonzero(dist == dist.min())
        code = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        out[i] = code | (0x80 if np.signbit(v) else 0)
    return out


def test_brute_force_nearest_on_all_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bf16_to_f32(bits)
    got = oracle.e4m3_encode(x)
    want = _brute_force_encode(x)
    assert np.array_equal(got, want)


def test_brute_force_nearest_on_random_fp32():
    g = np.random.default_rng(7)
    e = g.uniform(-14, 10, size=20000)
    x = (np.exp2(e) * g.choice([-1, 1], size=e.size)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _brute_force_encode(x))


def test_library_encode_inside_finite_range():
    g = np.random.default_rng(8)
    x = (g.standard_normal(200000) * g.choice([1e-3, 0.1, 1, 30, 200], size=200000)).astype(np.float32)
    x = x[np.abs(x) <= 448]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), lib)


@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.5, 1 / 448, 7.0e-5])
def test_quantiser_is_fp32_division_then_encode(scale):
    g = np.random.default_rng(9)
    xb = bf16_bits(g.standard_normal(5000).astype(np.float32) * np.float32(4))
    s = np.float32(scale)
    q = (bf16_to_f32(xb) / s).astype(np.float32)      # numpy: IEEE fp32 division
    assert np.array_equal(oracle.quantize_bf16(xb, s), oracle.e4m3_encode(q))


def test_quantiser_error_bound():
    """|decode(code)*s - x| <= half the e4m3 spacing at x/s (times s), in range."""
    g = np.random.default_rng(10)
    xb = bf16_bits(g.standard_normal(20000).astype(np.float32))
    x = bf16_to_f32(xb).astype(np.float64)
    s = np.float32(np.abs(x).max() / 448.0)
    codes = oracle.quantize_bf16(xb, s)
    y = oracle.e4m3_decode(codes) * float(s)
    a = np.abs(x / float(s))
    e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
    spacing = np.exp2(e - 3)                      # 3 mantissa bits; subnormal spacing 2^-9
    assert (np.abs(y - x) <= 0.5 * spacing * float(s) * (1 + 1e-6) + 1e-30).all()
