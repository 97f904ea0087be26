"""GPU parity of the e4m3 quantiser, the cache writes and the page-tag kernels.

Bit-exact against the oracle on the same seeded inputs: e4m3 codes (the
quantiser over every bf16 pattern, random and exhaustive fp32), whole-pool
bytes after prompt writes and decode appends (including guarded writes that
must not happen), tag bumps and abort sets / counts of the batched check.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300 import (fpk_page_tags_bump, fpk_page_tags_validate, fpk_quantize_e4m3)
from fp8_paged_kv_gb300.pool import DecodePool, to_device
from tests.gpu_helpers import oracle_pools
from workloads import bf16_to_f32, custom, rng_for, tiny

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu_quantize(x_f32: np.ndarray, scale: float) -> np.ndarray:
    x = torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(DEV)
    s = torch.tensor([scale], dtype=torch.float32, device=DEV)
    out = torch.empty(x.numel(), dtype=torch.uint8, device=DEV)
    fpk_quantize_e4m3(x, s, out)
    return out.cpu().numpy()


@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.5, 1 / 448, 7.0e-5, 1e-30])
def test_quantize_every_bf16_pattern(scale):
    x = bf16_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    s = np.float32(scale)
    want = oracle.e4m3_encode((x / s).astype(np.float32))
    got = _gpu_quantize(x, float(s))
    nan_in = np.isnan(x / s)
    # NaN inputs: the oracle's reading is 0x7F; compare the NaN-ness of the code
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert np.all((got[nan_in] & 0x7F) == 0x7F)


def test_quantize_random_fp32_bit_patterns():
    g = np.random.default_rng(5)
    bits = g.integers(0, 2**32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    got = _gpu_quantize(x, 1.0)
    want = oracle.e4m3_encode(x)
    finite = ~np.isnan(x)
    assert np.array_equal(got[finite], want[finite])


def test_quantize_exhaustive_fp32_sweep():
    """All 2^32 fp32 bit patterns through the GPU quantiser (scale 1) vs the oracle."""
    chunk = 1 << 26
    for base in range(0, 1 << 32, chunk):
        bits = np.arange(base, base + chunk, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        got = _gpu_quantize(x, 1.0)
        want = oracle.e4m3_encode(x)
        finite = ~np.isnan(x)
        assert np.array_equal(got[finite], want[finite]), hex(base)
        assert np.all((got[~finite] & 0x7F) == 0x7F)


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("ps", [16, 32, 64, 256])
def test_prefill_and_append_bytes_bit_exact(fp8, ps):
    wl = custom(51, B=5, Hq=8, Hkv=2, ps=ps, prompt_lens=[0, 1, ps - 1, ps, 3 * ps + 5], steps=1,
                sigma=3.0, outlier_frac=0.05)
    pool = DecodePool(wl, fp8=fp8, device=DEV)
    pool.prefill()
    ref = oracle_pools(wl, fp8)
    assert np.array_equal(pool.pool_bytes(), ref)
    pool.set_step(0)
    pool.append()
    kn, vn = wl.step_tokens(0)
    lens = wl.seq_lens_after(0)
    mask = np.zeros(wl.B, np.uint8)
    oracle.kv_append(kn, vn, ref, wl.k_scale, wl.v_scale, wl.page_table, lens, wl.live_tags,
                     wl.expected_tags, mask, fp8=fp8, Hkv=wl.Hkv, D=wl.D, page_size=ps,
                     num_pages=wl.num_pages)
    assert np.array_equal(pool.pool_bytes(), ref)
    assert np.array_equal(pool.abort_mask.cpu().numpy(), mask)


@pytest.mark.parametrize("what", ["stale", "page_oob", "neg_page", "beyond_table", "none"])
def test_guarded_append_bit_exact(what):
    ps = 16
    wl = custom(52, B=4, Hq=8, Hkv=2, ps=ps, prompt_lens=[20, 40, 15, 31], steps=1)
    pt, ex = wl.page_table.copy(), wl.expected_tags.copy()
    lens = wl.seq_lens_after(0).copy()
    r = 1
    pi = (int(lens[r]) - 1) // ps
    if what == "stale":
        ex[r, pi] += np.uint32(7)
    elif what == "page_oob":
        pt[r, pi] = wl.num_pages
    elif what == "neg_page":
        pt[r, pi] = -1
    elif what == "beyond_table":
        lens[r] = pt.shape[1] * ps + 3
    wl.page_table, wl.expected_tags = pt, ex
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.set_step(0)
    pool.seq_lens = to_device(lens, DEV)
    pool.append()
    ref = oracle_pools(wl, True, fill=False)
    kn, vn = wl.step_tokens(0)
    mask = np.zeros(wl.B, np.uint8)
    oracle.kv_append(kn, vn, ref, wl.k_scale, wl.v_scale, pt, lens, wl.live_tags, ex, mask,
                     fp8=True, Hkv=wl.Hkv, D=wl.D, page_size=ps, num_pages=wl.num_pages)
    assert np.array_equal(pool.pool_bytes(), ref)
    assert np.array_equal(pool.abort_mask.cpu().numpy(), mask)
    assert mask[r] == (0 if what == "none" else 1)


def test_bump_bit_exact():
    g = np.random.default_rng(6)
    num_pages = 5000
    live = g.integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    live[:4] = 0xFFFFFFFF
    pages = np.concatenate([g.integers(-10, num_pages + 10, size=20000), [0, 1, 1, 2, 2, 2, 3]])
    pages = pages.astype(np.int32)
    d_live = to_device(live, DEV)
    fpk_page_tags_bump(d_live, to_device(pages, DEV), num_pages=num_pages)
    oracle.page_tags_bump(live, pages, num_pages)
    assert np.array_equal(d_live.cpu().numpy().view(np.uint32), live)
    # n == 0 is a no-op
    fpk_page_tags_bump(d_live, to_device(pages[:0], DEV), num_pages=num_pages)
    assert np.array_equal(d_live.cpu().numpy().view(np.uint32), live)


@pytest.mark.parametrize("B,max_pages,ps", [(3, 4, 16), (64, 1040, 16), (256, 600, 16), (7, 33, 64),
                                            (4, 2048, 64), (5, 300, 16), (9, 700, 16), (2, 20000, 16)])
def test_validate_abort_sets_bit_exact(B, max_pages, ps):
    g = rng_for(53, "validate", B)
    num_pages = B * max_pages + 17
    lens = g.integers(0, max_pages * ps + 1, size=B).astype(np.int32)
    lens[: min(3, B)] = [0, 1, max_pages * ps][: min(3, B)]
    perm = g.permutation(num_pages).astype(np.int32)
    pt = np.full((B, max_pages), -1, np.int32)
    o = 0
    for r in range(B):
        P = -(-int(lens[r]) // ps)
        pt[r, :P] = perm[o:o + P]
        o += P
    live = g.integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    ex = np.zeros((B, max_pages), np.uint32)
    m = pt >= 0
    ex[m] = live[pt[m]]
    # entries past a request's pages are padding and must be ignored
    pad = pt < 0
    pt[pad] = g.integers(-3, 2 * num_pages, size=int(pad.sum())).astype(np.int32)
    ex[pad] = g.integers(0, 2**32, size=int(pad.sum()), dtype=np.uint64).astype(np.uint32)
    # corruptions inside the checked entries: stale tags and bad page ids
    for r in g.choice(B, size=max(1, B // 4), replace=False):
        P = -(-int(lens[r]) // ps)
        if P == 0:
            continue
        i = int(g.integers(0, P))
        kind = int(g.integers(0, 3))
        if kind == 0:
            ex[r, i] -= np.uint32(1)
        elif kind == 1:
            pt[r, i] = num_pages + int(g.integers(0, 5))
        else:
            pt[r, i] = -int(g.integers(1, 5))
    if B > 4:
        lens[4] = max_pages * ps + 1
    want, n = oracle.page_tags_validate(pt, ex, lens, live, num_pages, ps)
    d_mask = torch.full((B,), 7, dtype=torch.uint8, device=DEV)
    d_cnt = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    fpk_page_tags_validate(to_device(pt, DEV), to_device(ex, DEV), to_device(lens, DEV),
                           to_device(live, DEV), d_mask, d_cnt, num_pages=num_pages, page_size=ps)
    assert np.array_equal(d_mask.cpu().numpy(), want)
    assert int(d_cnt.item()) == n


@pytest.mark.parametrize("max_pages", [2048, 5000, 9000, 20000])
def test_validate_long_tables_every_part(max_pages):
    # tables above 4096 entries are shared by a cluster of 2, 4 or 8 CTAs
    # (thread t of part k takes entries k*256 + t + j*parts*256); request r
    # carries one corruption in entries r*256 .. r*256+255, which fall to part
    # r mod parts (request 8: none; request 9: its last entry), so every
    # part's finding must reach the request's abort flag, and only its own
    ps = 16
    B = 10
    g = rng_for(54, "parts", max_pages)
    num_pages = B * max_pages
    pt = g.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    live = g.integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    ex = live[pt]
    lens = np.full(B, max_pages * ps, np.int32)
    for r in range(8):
        i = r * 256 + int(g.integers(0, 256))
        if i < max_pages:
            ex[r, i] ^= np.uint32(1 << (r % 32))
    ex[9, max_pages - 1] -= np.uint32(1)
    want, n = oracle.page_tags_validate(pt, ex, lens, live, num_pages, ps)
    d_mask = torch.full((B,), 7, dtype=torch.uint8, device=DEV)
    d_cnt = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    fpk_page_tags_validate(to_device(pt, DEV), to_device(ex, DEV), to_device(lens, DEV),
                           to_device(live, DEV), d_mask, d_cnt, num_pages=num_pages, page_size=ps)
    got = d_mask.cpu().numpy()
    assert np.array_equal(got, want) and int(d_cnt.item()) == n
    assert got[8] == 0 and got[9] == 1


def test_tiny_workload_abort_set():
    wl = tiny()
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    pool.set_step(0)
    pool.append()
    pool.validate()
    mask, n = oracle.page_tags_validate(wl.page_table, wl.expected_tags, wl.seq_lens_after(0),
                                        wl.live_tags, wl.num_pages, wl.page_size)
    assert list(mask) == [0, 1] and n == 1
    assert np.array_equal(pool.abort_mask.cpu().numpy(), mask)
    assert int(pool.abort_count.item()) == 1


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("what", ["none", "stale_last", "stale_inner", "page_oob", "beyond_table"])
@pytest.mark.parametrize("table", ["short", "long"])
def test_append_check_one_launch_equals_write_then_check(fp8, what, table):
    """fpk_decode_append_check_*: bytes and abort mask equal to the oracle's append followed
    by its batched check, for clean tables and every kind of bad entry; long tables are
    checked by a cluster of CTAs per request."""
    ps = 16
    # long: 6251 table entries, checked by a cluster of two CTAs per request
    lens0 = [20, 40, 15, 31, 0, 300] if table == "short" else [20, 8000, 15, 31, 0, 100000]
    wl = custom(54, B=6, Hq=8, Hkv=2, ps=ps, prompt_lens=lens0, steps=1)
    pt, ex = wl.page_table.copy(), wl.expected_tags.copy()
    lens = wl.seq_lens_after(0).copy()
    r = 1
    last = (int(lens[r]) - 1) // ps
    if what == "stale_last":
        ex[r, last] += np.uint32(3)
    elif what == "stale_inner":
        ex[r, 0] -= np.uint32(1)
    elif what == "page_oob":
        pt[r, last] = wl.num_pages + 2
    elif what == "beyond_table":
        lens[r] = pt.shape[1] * ps + 5
    wl.page_table, wl.expected_tags = pt, ex
    pool = DecodePool(wl, fp8=fp8, device=DEV)
    pool.prefill()
    pool.set_step(0)
    pool.seq_lens = to_device(lens, DEV)
    pool.abort_mask.fill_(9)
    pool.append_check()
    torch.cuda.synchronize()
    ref = oracle_pools(wl, fp8)
    kn, vn = wl.step_tokens(0)
    oracle.kv_append(kn, vn, ref, wl.k_scale, wl.v_scale, pt, lens, wl.live_tags, ex, None,
                     fp8=fp8, Hkv=wl.Hkv, D=wl.D, page_size=ps, num_pages=wl.num_pages)
    mask, n = oracle.page_tags_validate(pt, ex, lens, wl.live_tags, wl.num_pages, ps)
    assert np.array_equal(pool.pool_bytes(), ref)
    assert np.array_equal(pool.abort_mask.cpu().numpy(), mask)
    assert mask[r] == (0 if what == "none" else 1)
