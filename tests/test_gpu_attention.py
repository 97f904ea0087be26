"""GPU parity of split-KV paged decode attention (FP8 and BF16 caches).

Every case runs the CUDA path through the C ABI and the fp64 oracle on the
same seeded inputs; outputs must satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref|,
lse |gpu - ref| <= 1e-3 + 2^-16 |ref|, and dead requests (aborted, empty,
over-long, bad page id) must give exactly 0 and lse = -inf.  Small cases span
several tiles, ragged last tiles, every supported group size, several page
sizes and split counts; the full-size workloads run in the benchmark's launch
configuration and every request is checked (the oracle runs one request per
host thread).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300 import FpkError, fpk_decode_workspace_bytes
from fp8_paged_kv_gb300.pool import DecodePool, to_device
from tests.gpu_helpers import (assert_attention_close, oracle_attention, oracle_attention_all,
                               oracle_pool_all, oracle_pools)
from workloads import b32_8k, b64_var, custom, long128k, rng_for, tiny

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
_cache = {}


def _wl(fn, **kw):
    key = (fn.__name__, tuple(sorted(kw.items())))
    if key not in _cache:
        _cache.clear()          # keep at most one full-size workload in host memory
        _cache[key] = fn(**kw)
    return _cache[key]


def _run_case(wl, fp8, num_splits, abort=None, use_mask=True, pt_override=None):
    pool = DecodePool(wl, fp8=fp8, device=DEV, num_splits=num_splits)
    pool.prefill()
    lens = wl.prompt_lens.astype(np.int32)
    if pt_override is not None:
        pool.page_table = to_device(pt_override, DEV)
    if abort is not None:
        pool.abort_mask = to_device(abort.astype(np.uint8), DEV)
    pool.attend(use_mask=use_mask)
    torch.cuda.synchronize()
    assert pool.workspace[:4].view(torch.int32).item() == 0, "bounded wait gave up"
    ref = oracle_pools(wl, fp8)
    ref_out, ref_lse = oracle_attention(wl, ref, fp8, wl.q, lens,
                                        abort=abort if use_mask else None, page_table=pt_override)
    return pool.out.cpu().numpy(), pool.lse.cpu().numpy(), ref_out, ref_lse


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("ps", [16, 32, 64, 128, 256])
def test_small_ragged(fp8, G, ps):
    Hkv = 2
    lens = [0, 1, 15, 16, 17, 100, 3 * ps + 7, 257]
    wl = custom(61 + G + ps, B=len(lens), Hq=G * Hkv, Hkv=Hkv, ps=ps, prompt_lens=lens, steps=0,
                sigma=1.5, outlier_frac=0.02)
    out, lse, ro, rl = _run_case(wl, fp8, num_splits=0)
    assert_attention_close(out, lse, ro, rl, f"fp8={fp8} G={G} ps={ps}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("Hkv,G", [(1, 8), (1, 1), (16, 4), (32, 2)])
def test_kv_head_counts(fp8, Hkv, G):
    # one kv head (multi-query) up to 32 of them
    lens = [0, 5, 16, 130, 700, 33]
    wl = custom(90 + Hkv + G, B=len(lens), Hq=G * Hkv, Hkv=Hkv, ps=16, prompt_lens=lens, steps=0,
                sigma=1.2, outlier_frac=0.02)
    out, lse, ro, rl = _run_case(wl, fp8, num_splits=0)
    assert_attention_close(out, lse, ro, rl, f"fp8={fp8} Hkv={Hkv} G={G}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("num_splits", [1, 2, 5, 37, 61, 200, 300, 4096])
def test_split_counts(fp8, num_splits):
    lens = [700, 33, 0, 1025, 64, 5]
    wl = custom(70 + num_splits, B=len(lens), Hq=16, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    out, lse, ro, rl = _run_case(wl, fp8, num_splits=num_splits)
    assert_attention_close(out, lse, ro, rl, f"splits={num_splits}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("abort_one", [False, True])
def test_uniform_batch_one_segment_per_cta(fp8, abort_one):
    # 30 requests x 8 kv heads of equal length: with the automatic split count
    # (a wave of 304 CTAs on GB300) every CTA takes one whole segment
    lens = [200] * 30
    wl = custom(83, B=30, Hq=16, Hkv=8, ps=16, prompt_lens=lens, steps=0)
    abort = None
    if abort_one:
        abort = np.zeros(wl.B, np.uint8)
        abort[7] = 1
    out, lse, ro, rl = _run_case(wl, fp8, 0, abort=abort, use_mask=abort_one)
    assert_attention_close(out, lse, ro, rl, f"uniform fp8={fp8} abort={abort_one}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("lens", [[700] * 4, [0, 333, 333, 0, 333], [160] * 20, [1] * 3])
def test_uniform_small_batch_segment_aligned_splits(fp8, lens):
    # equal context lengths (empty requests aside) and fewer segments than 3/4
    # of the CTAs: the automatic count gives every segment the same number of
    # splits, all split boundaries on segment boundaries (one whole segment
    # per CTA once the segments fill half the CTAs)
    wl = custom(89 + len(lens), B=len(lens), Hq=64, Hkv=8, ps=16, prompt_lens=lens, steps=0,
                sigma=1.0, outlier_frac=0.01)
    out, lse, ro, rl = _run_case(wl, fp8, 0)
    assert_attention_close(out, lse, ro, rl, f"uniform small fp8={fp8} lens={lens[:3]}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("lens,abort_at", [([3000, 80], None), ([1, 2500, 17, 1111, 0], 3),
                                           ([900, 16, 17, 31, 33, 1500, 700, 2, 1200], None),
                                           ([4097, 4096, 4095, 4094, 4093, 4092, 4091, 4090, 4089, 4088, 4087, 4086], 0)])
def test_mixed_small_batch_segment_aligned_splits(fp8, lens, abort_at):
    # unequal context lengths and at most a third as many segments as CTAs:
    # the automatic count cuts every segment into splits of one common tile
    # count (the last one of a segment shorter), one split per CTA, so no
    # split straddles two segments and each CTA merges into one segment only
    wl = custom(97 + len(lens), B=len(lens), Hq=64, Hkv=8, ps=16, prompt_lens=lens, steps=0,
                sigma=1.0, outlier_frac=0.01)
    abort = None
    if abort_at is not None:
        abort = np.zeros(wl.B, np.uint8)
        abort[abort_at] = 1
    out, lse, ro, rl = _run_case(wl, fp8, 0, abort=abort, use_mask=abort is not None)
    assert_attention_close(out, lse, ro, rl, f"mixed small fp8={fp8} lens={lens[:3]}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("B", [18, 30])
def test_mixed_batch_past_a_third_of_the_ctas(fp8, B):
    # 18 and 30 requests of unequal lengths (144 and 240 segments, more than a
    # third of a wave): the automatic count keeps splits of equal tile count
    # over the whole batch, straddling segments; one request aborted
    lens = [int(x) for x in rng_for(150 + B, "lens").integers(100, 3000, size=B)]
    wl = custom(150 + B, B=B, Hq=64, Hkv=8, ps=16, prompt_lens=lens, steps=0, sigma=1.0,
                outlier_frac=0.01)
    abort = np.zeros(wl.B, np.uint8)
    abort[B // 2] = 1
    out, lse, ro, rl = _run_case(wl, fp8, 0, abort=abort, use_mask=True)
    assert_attention_close(out, lse, ro, rl, f"mixed B={B} fp8={fp8}")


@pytest.mark.parametrize("fp8", [True, False])
def test_uneven_batch_of_whole_segment_size(fp8):
    # 30 x 8 segments, as above, but of uneven lengths: the host launches the
    # deep-ring FP8 variant for a batch that may run one whole segment per CTA;
    # the kernel finds the lengths uneven, splits over a full wave and then
    # runs only the shallow part of its ring, with the two-slot merge
    lens = list(rng_for(84, "lens").integers(1, 400, size=30))
    wl = custom(84, B=30, Hq=16, Hkv=8, ps=16, prompt_lens=lens, steps=0)
    out, lse, ro, rl = _run_case(wl, fp8, 0)
    assert_attention_close(out, lse, ro, rl, f"uneven fp8={fp8}")


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("num_splits", [305, 1000, 2200])
def test_more_splits_than_a_wave(fp8, num_splits):
    # more splits than a wave of CTAs (304 on GB300), a tile in every split:
    # each CTA runs an equal number of consecutive splits (k = ceil(W / wave),
    # ceil(W / k) CTAs); splits straddle requests and kv heads, one request
    # is aborted
    lens = [7000, 33, 0, 10250, 640, 5, 1500]
    wl = custom(77 + num_splits, B=len(lens), Hq=16, Hkv=2, ps=16, prompt_lens=lens, steps=0,
                sigma=1.2, outlier_frac=0.02)
    tiles = sum(-(-n // 16) for n in lens) * 2
    assert num_splits <= tiles
    abort = np.zeros(wl.B, np.uint8)
    abort[4] = 1
    out, lse, ro, rl = _run_case(wl, fp8, num_splits, abort=abort, use_mask=True)
    assert_attention_close(out, lse, ro, rl, f"splits={num_splits} fp8={fp8}")


@pytest.mark.parametrize("case", ["uniform", "uneven", "splits200", "splits4096", "wave2000"])
def test_repeated_launches_bit_identical(case):
    # the partition, each CTA's merge order and each segment's combine order
    # are fixed, whichever CTA arrives last: repeated launches must agree to
    # the bit (a race between the copy ring and its readers would not)
    if case == "uniform":
        lens, ns = [700] * 30, 0
    elif case == "uneven":
        lens, ns = list(rng_for(85, "lens").integers(1, 1400, size=30)), 0
    elif case == "wave2000":
        # more splits than a wave, a tile in every split: 7 consecutive splits per CTA
        lens, ns = list(rng_for(86, "lens").integers(2000, 6000, size=12)), 2000
    else:
        lens, ns = list(rng_for(86, "lens").integers(1, 3000, size=12)), int(case[6:])
    wl = custom(87, B=len(lens), Hq=16, Hkv=8, ps=16, prompt_lens=lens, steps=0)
    pool = DecodePool(wl, fp8=True, device=DEV, num_splits=ns)
    pool.prefill()
    pool.attend()
    first = pool.out.clone(), pool.lse.clone()
    for _ in range(20):
        pool.out.fill_(float("nan"))
        pool.attend()
        assert torch.equal(pool.out.view(torch.int32), first[0].view(torch.int32))
        assert torch.equal(pool.lse.view(torch.int32), first[1].view(torch.int32))
    assert pool.workspace[:4].view(torch.int32).item() == 0


def test_rejects_misaligned_output():
    wl = custom(88, B=2, Hq=8, Hkv=2, ps=16, prompt_lens=[40, 9], steps=0)
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    buf = torch.empty(pool.out.numel() + 1, dtype=torch.float32, device=DEV)
    pool.out = buf[1:].view(pool.out.shape)              # 4 bytes past a 16-byte boundary
    with pytest.raises(FpkError):
        pool.attend()


@pytest.mark.parametrize("fp8", [True, False])
def test_thousands_of_short_requests(fp8):
    # 3000 requests of 0..70 tokens: ~20 segments per CTA, most of them whole,
    # the rest cut between CTAs (partials, batched arrivals, combines)
    lens = list(rng_for(91, "lens").integers(0, 71, size=3000))
    wl = custom(91, B=3000, Hq=8, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    out, lse, ro, rl = _run_case(wl, fp8, 0)
    assert_attention_close(out, lse, ro, rl, f"3000 short fp8={fp8}")


def test_split_invariance():
    lens = [3000, 1, 900]
    wl = custom(80, B=3, Hq=32, Hkv=4, ps=32, prompt_lens=lens, steps=0)
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    # one workspace large enough for every split count used below
    need = max(fpk_decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, ns) for ns in (0, 1000))
    pool.workspace = torch.zeros(need, dtype=torch.uint8, device=DEV)
    outs = []
    for ns in (0, 1, 7, 64, 1000):
        pool.attend(num_splits=ns)
        outs.append(pool.out.cpu().numpy().copy())
    # P is rounded to f16 (relative 2^-11) against a running max that depends on
    # where splits start, so results agree to about 2^-10 * max|V| across splits
    bound = 2.0 ** -10 * 448.0 * float(wl.v_scale)     # 448 * v_scale = max |V-hat|
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < bound


@pytest.mark.parametrize("fp8", [True, False])
def test_abort_mask_and_noop_tracker(fp8):
    lens = [40, 90, 17, 300]
    wl = custom(81, B=4, Hq=16, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    abort = np.array([0, 1, 0, 1], np.uint8)
    out, lse, ro, rl = _run_case(wl, fp8, 0, abort=abort, use_mask=True)
    assert_attention_close(out, lse, ro, rl, "masked")
    assert np.isneginf(lse[[1, 3]]).all() and not out[[1, 3]].any()
    # the no-op tracker (no mask) ignores tags and attends everything
    out, lse, ro, rl = _run_case(wl, fp8, 0, abort=abort, use_mask=False)
    assert_attention_close(out, lse, ro, rl, "no-op tracker")
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("num_splits", [0, 3, 64])
def test_bad_page_id_fails_closed_without_tracker(num_splits):
    lens = [200, 200, 200]
    wl = custom(82, B=3, Hq=8, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    pt = wl.page_table.copy()
    pt[1, 5] = wl.num_pages + 1000        # would read past the pool
    pt[2, 0] = -2
    out, lse, ro, rl = _run_case(wl, True, num_splits, use_mask=False, pt_override=pt)
    assert_attention_close(out, lse, ro, rl, "bad page")
    assert np.isneginf(lse[1:]).all() and not out[1:].any()


def test_overlong_context_is_dead():
    wl = custom(83, B=2, Hq=8, Hkv=2, ps=16, prompt_lens=[40, 40], steps=0)
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    lens = np.array([40, wl.max_pages * 16 + 1], np.int32)
    pool.seq_lens = to_device(lens, DEV)
    pool.attend(use_mask=False)
    out, lse = pool.out.cpu().numpy(), pool.lse.cpu().numpy()
    assert np.isneginf(lse[1]).all() and not out[1].any() and np.isfinite(lse[0]).all()


def test_tiny_full_step():
    """The tiny workload end to end: prefill, append, validate, attend."""
    wl = tiny()
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    pool.set_step(0)
    pool.step(validate=True)
    torch.cuda.synchronize()
    ref = oracle_pools(wl, True)
    kn, vn = wl.step_tokens(0)
    lens = wl.seq_lens_after(0)
    mask0 = np.zeros(2, np.uint8)
    oracle.kv_append(kn, vn, ref, wl.k_scale, wl.v_scale, wl.page_table, lens, wl.live_tags,
                     wl.expected_tags, mask0, fp8=True, Hkv=wl.Hkv, D=wl.D, page_size=16,
                     num_pages=wl.num_pages)
    assert np.array_equal(pool.pool_bytes(), ref)
    mask, n = oracle.page_tags_validate(wl.page_table, wl.expected_tags, lens, wl.live_tags,
                                        wl.num_pages, 16)
    assert list(mask) == [0, 1] and np.array_equal(pool.abort_mask.cpu().numpy(), mask)
    ro, rl = oracle_attention(wl, ref, True, wl.q, lens, abort=mask)
    assert_attention_close(pool.out.cpu().numpy(), pool.lse.cpu().numpy(), ro, rl, "tiny")


def _full_size(wl, fp8, steps=1, num_splits=None):
    """Run `steps` decode steps (append, validate, attend) at full size in the
    benchmark's launch configuration and check every request against the
    oracle: the abort set of every step, the whole pool's bytes after the last
    step (pages no token was written to hold the fill code on both sides) and
    the attention of every request at the last step."""
    pool = DecodePool(wl, fp8=fp8, device=DEV, num_splits=num_splits)
    pool.prefill()
    for s in range(steps):
        pool.set_step(s)
        pool.step(validate=True)
        torch.cuda.synchronize()
        lens = wl.seq_lens_after(s)
        mask, n = oracle.page_tags_validate(wl.page_table, wl.expected_tags, lens, wl.live_tags,
                                            wl.num_pages, wl.page_size)
        assert np.array_equal(pool.abort_mask.cpu().numpy(), mask), f"abort set, step {s}"
        assert int(pool.abort_count.item()) == n
    assert pool.workspace[:4].view(torch.int32).item() == 0
    out = pool.out.cpu().numpy()
    lse = pool.lse.cpu().numpy()
    got = pool.pool_bytes()
    del pool
    torch.cuda.empty_cache()
    ref = oracle_pool_all(wl, fp8, steps)
    assert np.array_equal(got, ref), "pool bytes differ from the oracle's"
    del got
    lens = wl.seq_lens_after(steps - 1)
    q = wl.step_query(steps - 1)
    ro, rl = oracle_attention_all(wl, ref, fp8, q, lens, abort=mask)
    return assert_attention_close(out, lse, ro, rl, f"{wl.name} fp8={fp8}")


@pytest.mark.parametrize("fp8", [True, False])
def test_b32_8k_full_size_every_request(fp8):
    _full_size(_wl(b32_8k), fp8, steps=1)


def test_b64_var_full_size_every_request_after_256_steps():
    # all 256 decode steps the benchmark replays: every step's abort set, then
    # the pool and all 64 requests' attention after the last one
    _full_size(_wl(b64_var), True, steps=256)


def test_long128k_full_size_every_request_64_splits():
    _full_size(_wl(long128k), True, steps=1, num_splits=64 * 4 * 8)
