"""GPU parity of the bulk prompt write and of the per-tensor scale reduction.

Bit-exact against the oracle on the same seeded inputs: whole-pool bytes and
abort masks after prompt writes (tile-wise kernel, and the per-token kernel
that serves batches of more than 8192 requests), including guarded tiles that
must not be written, and the amax / 448 scale computed on the device.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300 import (FpkError, fpk_amax_scale_bf16, fpk_kv_prefill_bf16,
                                fpk_kv_prefill_fp8)
from fp8_paged_kv_gb300.pool import NAN_BF16, NAN_E4M3, to_device
from workloads import bf16_bits, bf16_to_f32, custom

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu_scale(bits: np.ndarray, offset: int = 0) -> np.float32:
    x = to_device(np.concatenate([np.zeros(offset, np.uint16), bits]), DEV)[offset:]
    s = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    scratch = torch.full((2,), 12345, dtype=torch.int32, device=DEV)
    fpk_amax_scale_bf16(x, s, scratch)
    return np.float32(s.item())


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000, 4099, (1 << 20) + 3, 1 << 24])
def test_amax_scale_bit_exact(n):
    g = np.random.default_rng(n % 997 + 3)
    x = (g.standard_normal(n) * 10.0 ** g.uniform(-20, 20)).astype(np.float32)
    bits = bf16_bits(x)
    if n >= 8:
        # non-finite values are skipped; the largest finite one sits in the ragged tail
        idx = g.choice(n - 1, size=3, replace=False)
        bits[idx] = np.array([0x7F80, 0xFF80, 0x7FC1], np.uint16)
        bits[n - 1] = bf16_bits(np.array([-np.abs(x).max() * 3], np.float32))[0]
    want = oracle.amax_scale_bf16(bits)
    got = _gpu_scale(bits)
    assert got == want, (got, want)


def test_amax_scale_special_cases():
    assert _gpu_scale(np.zeros(100, np.uint16)) == 1.0
    assert _gpu_scale(np.array([0x7F80, 0x7FC0, 0xFF80] * 11, np.uint16)) == 1.0
    assert _gpu_scale(bf16_bits(np.array([448.0 * 2 ** -20] * 33, np.float32))) == np.float32(2 ** -20)
    with pytest.raises(FpkError):
        _gpu_scale(np.ones(64, np.uint16), offset=1)  # not 16-byte aligned


def _run_prefill(wl, fp8, pt, ex, scales=None):
    n = 2 * wl.num_pages * wl.Hkv * wl.page_size * wl.D
    if fp8:
        pool = torch.full((n,), NAN_E4M3, dtype=torch.uint8, device=DEV)
    else:
        pool = torch.full((n,), NAN_BF16, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    k, v = to_device(wl.k_prompt, DEV), to_device(wl.v_prompt, DEV)
    cu = to_device(wl.cu_prompt.astype(np.int32), DEV)
    mask = torch.zeros(wl.B, dtype=torch.uint8, device=DEV)
    kw = dict(Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size, num_pages=wl.num_pages)
    pt_d, live_d, ex_d = to_device(pt, DEV), to_device(wl.live_tags, DEV), to_device(ex, DEV)
    if fp8:
        if scales is None:
            ks = torch.tensor([float(wl.k_scale)], device=DEV)
            vs = torch.tensor([float(wl.v_scale)], device=DEV)
        else:
            ks, vs = scales
        fpk_kv_prefill_fp8(k, v, cu, pool, ks, vs, pt_d, live_d, ex_d, mask, **kw)
        got = pool.cpu().numpy()
    else:
        fpk_kv_prefill_bf16(k, v, cu, pool, pt_d, live_d, ex_d, mask, **kw)
        got = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    return got, mask.cpu().numpy()


def _oracle_prefill(wl, fp8, pt, ex, k_scale=None, v_scale=None):
    n = 2 * wl.num_pages * wl.Hkv * wl.page_size * wl.D
    ref = np.full(n, NAN_E4M3 if fp8 else NAN_BF16, np.uint8 if fp8 else np.uint16)
    mask = np.zeros(wl.B, np.uint8)
    oracle.kv_prefill(wl.k_prompt, wl.v_prompt, wl.cu_prompt, ref,
                      wl.k_scale if k_scale is None else k_scale,
                      wl.v_scale if v_scale is None else v_scale, pt, wl.live_tags, ex, mask,
                      fp8=fp8, Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size, num_pages=wl.num_pages)
    return ref, mask


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("what", ["none", "stale", "page_oob", "neg_page", "beyond_table"])
def test_guarded_prefill_bit_exact(fp8, what):
    wl = custom(91, B=4, Hq=8, Hkv=2, ps=16, prompt_lens=[40, 70, 16, 33], steps=0,
                sigma=2.0, outlier_frac=0.05)
    pt, ex = wl.page_table.copy(), wl.expected_tags.copy()
    r = 1
    if what == "stale":
        ex[r, 2] += np.uint32(1)
    elif what == "page_oob":
        pt[r, 1] = wl.num_pages
    elif what == "neg_page":
        pt[r, 4] = -1          # the request's last, partly filled page
    elif what == "beyond_table":
        pt, ex = np.ascontiguousarray(pt[:, :4]), np.ascontiguousarray(ex[:, :4])
    got, mask = _run_prefill(wl, fp8, pt, ex)
    ref, want = _oracle_prefill(wl, fp8, pt, ex)
    assert np.array_equal(got, ref)
    assert np.array_equal(mask, want)
    assert want[r] == (0 if what == "none" else 1) and want.sum() == want[r]


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("ps", [16, 64, 256])
def test_prefill_many_ragged_requests(fp8, ps):
    g = np.random.default_rng(ps)
    lens = g.choice([0, 1, 2, 15, 16, 17, 31, 33, 100, 257, 600], size=300)
    wl = custom(92 + ps, B=300, Hq=4, Hkv=2, ps=ps, prompt_lens=lens, steps=0, sigma=1.5)
    got, mask = _run_prefill(wl, fp8, wl.page_table, wl.expected_tags)
    ref, want = _oracle_prefill(wl, fp8, wl.page_table, wl.expected_tags)
    assert np.array_equal(got, ref)
    assert not mask.any() and not want.any()


def test_prefill_more_requests_than_the_tile_scan_holds():
    # 8193 requests: served by the per-token kernel, same bytes
    g = np.random.default_rng(93)
    lens = g.integers(0, 4, size=8193)
    wl = custom(93, B=8193, Hq=2, Hkv=1, ps=16, prompt_lens=lens, steps=0)
    got, mask = _run_prefill(wl, True, wl.page_table, wl.expected_tags)
    ref, want = _oracle_prefill(wl, True, wl.page_table, wl.expected_tags)
    assert np.array_equal(got, ref)
    assert np.array_equal(mask, want)


def test_prefill_with_device_scales():
    """amax / 448 computed on the device, read by the prompt write on the device."""
    wl = custom(94, B=6, Hq=16, Hkv=4, ps=32, prompt_lens=[500, 1, 0, 77, 1024, 33], steps=0,
                sigma=0.5, outlier_frac=0.02)
    k, v = to_device(wl.k_prompt, DEV), to_device(wl.v_prompt, DEV)
    ks = torch.empty(1, dtype=torch.float32, device=DEV)
    vs = torch.empty(1, dtype=torch.float32, device=DEV)
    scratch = torch.empty(2, dtype=torch.int32, device=DEV)
    fpk_amax_scale_bf16(k, ks, scratch)
    fpk_amax_scale_bf16(v, vs, scratch)
    k_ref = oracle.amax_scale_bf16(wl.k_prompt.reshape(-1))
    v_ref = oracle.amax_scale_bf16(wl.v_prompt.reshape(-1))
    assert np.float32(ks.item()) == k_ref and np.float32(vs.item()) == v_ref
    got, _ = _run_prefill(wl, True, wl.page_table, wl.expected_tags, scales=(ks, vs))
    ref, _ = _oracle_prefill(wl, True, wl.page_table, wl.expected_tags, k_ref, v_ref)
    assert np.array_equal(got, ref)


def _scales_under_test():
    g = np.random.default_rng(2024)
    s = [1.0, 3.0, 7.0, 0.1, 448.0, 1 / 448, 2.0 ** -30, 2.0 ** 30, 1e-30, 1e30, 2.0 ** -126,
         2.0 ** -127, 2.0 ** -149, 3.0e38, np.finfo(np.float32).max]
    s += [float(np.float32((2 - 2.0 ** -23) * 2.0 ** e)) for e in range(-24, 25, 3)]   # all-ones significands
    s += [float(np.float32((1 + 2.0 ** -23) * 2.0 ** e)) for e in range(-24, 25, 3)]
    s += list((2.0 ** g.uniform(-40, 40, 520)).astype(np.float32))
    return [np.float32(v) for v in s]


def test_quantiser_every_bf16_pattern_many_scales():
    """The bf16-input quantiser of the cache writes (one reciprocal per tensor,
    one corrected product per element) against the oracle's IEEE division:
    every finite bf16 pattern, as K and as V, at ~570 scales including the
    ones whose reciprocal is not a normal number."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    pats = pats[~np.isnan(bf16_to_f32(pats))]        # NaN inputs: compared elsewhere by NaN-ness
    D, ps = 128, 16
    T = -(-pats.size // D)
    k = np.zeros(T * D, np.uint16)
    k[:pats.size] = pats
    k = k.reshape(T, 1, D)
    v = np.ascontiguousarray(k[::-1])
    P = -(-T // ps)
    pt = np.arange(P, dtype=np.int32)[None, :]
    cu = np.array([0, T], np.int32)
    n = 2 * P * ps * D
    k_d, v_d = to_device(k, DEV), to_device(v, DEV)
    cu_d, pt_d = to_device(cu, DEV), to_device(pt, DEV)
    pool = torch.zeros(n, dtype=torch.uint8, device=DEV)
    sc_d = torch.empty(1, dtype=torch.float32, device=DEV)
    for sc in _scales_under_test():
        sc_d.fill_(float(sc))
        fpk_kv_prefill_fp8(k_d, v_d, cu_d, pool, sc_d, sc_d, pt_d, None, None, None, Hkv=1, D=D,
                           page_size=ps, num_pages=P)
        ref = np.zeros(n, np.uint8)
        oracle.kv_prefill(k, v, cu, ref, sc, sc, pt, None, None, None, fp8=True, Hkv=1, D=D,
                          page_size=ps, num_pages=P)
        got = pool.cpu().numpy()
        assert np.array_equal(got, ref), f"scale {float(sc)!r}: {int((got != ref).sum())} codes differ"
