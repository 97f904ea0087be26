"""Pins of the oracle's cache writes (quantise-on-append and bulk prompt writes).

The pages (Cloudflare write-up, Italian edition, "Cosa ha cambiato Cloudflare
per Kimi e GLM") store Kimi's K/V as e4m3 codes in place of bf16; the iitog.ru
summary (third technique) says requests both read and write pages of the one
shared physical cache.  The tests check the written bytes against the codec
(itself pinned in test_oracle_e4m3.py), that nothing outside the target slot
changes, that a stale destination tag blocks the write and aborts, and that a
bulk prompt write equals token-by-token appends.
"""
import numpy as np
import pytest

import oracle
from workloads import bf16_bits, bf16_to_f32, custom


def _slot_indices(page, h, off, Hkv, ps, D):
    """Flat element indices of one token's K row and V column in the KV pool
    [page][kv head][tile of 16 tokens][K block [16][D], V block [D][16]]."""
    base = (((page * Hkv + h) * (ps // 16) + off // 16) * 2) * 16 * D
    k = base + (off % 16) * D + np.arange(D)
    v = base + 16 * D + np.arange(D) * 16 + off % 16
    return k, v


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("ps", [16, 64])
def test_append_writes_exactly_the_slot(fp8, ps):
    wl = custom(21, B=3, Hq=8, Hkv=2, ps=ps, prompt_lens=[5, ps, 2 * ps - 1])
    dt = np.uint8 if fp8 else np.uint16
    n = 2 * wl.num_pages * wl.Hkv * ps * wl.D
    g = np.random.default_rng(1)
    pool0 = g.integers(0, 256 if fp8 else 65536, size=n).astype(dt)
    pool = pool0.copy()
    kn, vn = wl.step_tokens(0)
    lens = wl.seq_lens_after(0)
    mask = np.zeros(wl.B, np.uint8)
    oracle.kv_append(kn, vn, pool, wl.k_scale, wl.v_scale, wl.page_table, lens,
                     wl.live_tags, wl.expected_tags, mask, fp8=fp8, Hkv=wl.Hkv, D=wl.D,
                     page_size=ps, num_pages=wl.num_pages)
    assert not mask.any()
    touched_k, touched_v = [], []
    for r in range(wl.B):
        pos = int(lens[r]) - 1
        page = int(wl.page_table[r, pos // ps])
        for h in range(wl.Hkv):
            ki, vi = _slot_indices(page, h, pos % ps, wl.Hkv, ps, wl.D)
            touched_k.append(ki)
            touched_v.append(vi)
            if fp8:
                wantk = oracle.e4m3_encode(bf16_to_f32(kn[r, h]) / wl.k_scale)
                wantv = oracle.e4m3_encode(bf16_to_f32(vn[r, h]) / wl.v_scale)
            else:
                wantk, wantv = kn[r, h], vn[r, h]
            assert np.array_equal(pool[ki], wantk)
            assert np.array_equal(pool[vi], wantv)
    touched = np.concatenate(touched_k + touched_v)
    assert np.unique(touched).size == touched.size      # K and V slots never overlap
    rest = np.ones(n, bool)
    rest[touched] = False
    assert np.array_equal(pool[rest], pool0[rest])


@pytest.mark.parametrize("what", ["stale", "page_oob", "neg_page", "beyond_table"])
def test_guarded_append_skips_and_aborts(what):
    ps = 16
    wl = custom(22, B=2, Hq=4, Hkv=1, ps=ps, prompt_lens=[20, 40])
    n = 2 * wl.num_pages * wl.Hkv * ps * wl.D
    kp = np.zeros(n, np.uint8)
    kn, vn = wl.step_tokens(0)
    lens = wl.seq_lens_after(0).copy()
    pt, exp = wl.page_table.copy(), wl.expected_tags.copy()
    r = 1
    pi = (int(lens[r]) - 1) // ps
    if what == "stale":
        exp[r, pi] += np.uint32(1)
    elif what == "page_oob":
        pt[r, pi] = wl.num_pages
    elif what == "neg_page":
        pt[r, pi] = -3
    else:
        lens[r] = pt.shape[1] * ps + 1
    mask = np.zeros(2, np.uint8)
    oracle.kv_append(kn, vn, kp, wl.k_scale, wl.v_scale, pt, lens, wl.live_tags, exp, mask,
                     fp8=True, Hkv=1, D=wl.D, page_size=ps, num_pages=wl.num_pages)
    assert list(mask) == [0, 1]
    # request 0 wrote its slot, request 1 wrote nothing
    page0 = int(pt[0, (int(lens[0]) - 1) // ps])
    ki, vi = _slot_indices(page0, 0, (int(lens[0]) - 1) % ps, 1, ps, wl.D)
    written = np.zeros(n, bool)
    written[ki] = True
    written[vi] = True
    assert not kp[~written].any()


def test_no_tracker_means_no_tag_check():
    ps = 16
    wl = custom(23, B=1, Hq=4, Hkv=1, ps=ps, prompt_lens=[3])
    n = 2 * wl.num_pages * ps * wl.D
    kp = np.zeros(n, np.uint8)
    kn, vn = wl.step_tokens(0)
    exp = wl.expected_tags + np.uint32(1)       # all stale, but no tags given below
    oracle.kv_append(kn, vn, kp, wl.k_scale, wl.v_scale, wl.page_table, wl.seq_lens_after(0),
                     None, None, None, fp8=True, Hkv=1, D=wl.D, page_size=ps, num_pages=wl.num_pages)
    assert kp.any()
    del exp


@pytest.mark.parametrize("fp8", [True, False])
def test_prefill_equals_token_by_token_append(fp8):
    ps = 16
    wl = custom(24, B=3, Hq=8, Hkv=2, ps=ps, prompt_lens=[1, 33, 16])
    dt = np.uint8 if fp8 else np.uint16
    n = 2 * wl.num_pages * wl.Hkv * ps * wl.D
    kp1 = np.zeros(n, dt)
    kp2 = np.zeros(n, dt)
    oracle.kv_prefill(wl.k_prompt, wl.v_prompt, wl.cu_prompt, kp1, wl.k_scale, wl.v_scale,
                      wl.page_table, wl.live_tags, wl.expected_tags, None, fp8=fp8, Hkv=wl.Hkv,
                      D=wl.D, page_size=ps, num_pages=wl.num_pages)
    maxlen = int(wl.prompt_lens.max())
    for t in range(maxlen):
        kn = np.zeros((wl.B, wl.Hkv, wl.D), np.uint16)
        vn = np.zeros_like(kn)
        lens = np.zeros(wl.B, np.int32)
        for r in range(wl.B):
            if t < wl.prompt_lens[r]:
                kn[r] = wl.k_prompt[wl.cu_prompt[r] + t]
                vn[r] = wl.v_prompt[wl.cu_prompt[r] + t]
                lens[r] = t + 1
        oracle.kv_append(kn, vn, kp2, wl.k_scale, wl.v_scale, wl.page_table, lens,
                         wl.live_tags, wl.expected_tags, None, fp8=fp8, Hkv=wl.Hkv, D=wl.D,
                         page_size=ps, num_pages=wl.num_pages)
    assert np.array_equal(kp1, kp2)


def test_fp8_pool_is_half_the_bf16_bytes():
    """Capacity claim of the pages: e4m3 holds twice the tokens of bf16 in the same bytes."""
    wl = custom(25, B=2, Hq=8, Hkv=2, ps=16, prompt_lens=[10, 20])
    assert wl.kv_bytes(fp8=False) == 2 * wl.kv_bytes(fp8=True)
    assert np.dtype(np.uint16).itemsize == 2 * np.dtype(np.uint8).itemsize


def test_bf16_rounding_helper_ties_to_even():
    x = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5], np.float32)
    assert list(bf16_to_f32(bf16_bits(x))) == [1.0, 1.0 + 4 * 2**-8, -2.5]
