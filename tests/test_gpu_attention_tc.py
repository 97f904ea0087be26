"""GPU parity of the tensor-core FP8 attention (fpk_paged_decode_attn_fp8_tc:
tcgen05.mma of kind f8f6f4 with TMEM accumulators).

The same contract as the warp-level kernel: every case runs the CUDA path
through the C ABI and the fp64 oracle on the same seeded inputs; outputs must
satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref| and lse the derived lse bound, and
dead requests (aborted, empty, over-long, bad page id) must give exactly 0 and
lse = -inf.  The query and the softmax weights enter the MMAs as four e4m3
parts each, so the precision argument differs from the f16 kernel's; the
cases include the outlier-heavy ragged inputs that found the f16 limits.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300.pool import DecodePool, to_device
from tests.gpu_helpers import (assert_attention_close, oracle_attention, oracle_attention_all,
                               oracle_pool_all, oracle_pools)
from workloads import b32_8k, custom, long128k, rng_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _tc_case(wl, num_splits, abort=None, use_mask=True, pt_override=None):
    pool = DecodePool(wl, fp8=True, device=DEV, num_splits=num_splits, tensor_cores=True)
    pool.prefill()
    lens = wl.prompt_lens.astype(np.int32)
    if pt_override is not None:
        pool.page_table = to_device(pt_override, DEV)
    if abort is not None:
        pool.abort_mask = to_device(abort.astype(np.uint8), DEV)
    pool.out.fill_(float("nan"))
    pool.attend(use_mask=use_mask)
    torch.cuda.synchronize()
    assert pool.workspace[:4].view(torch.int32).item() == 0, "bounded wait gave up"
    ref = oracle_pools(wl, True)
    ref_out, ref_lse = oracle_attention(wl, ref, True, wl.q, lens,
                                        abort=abort if use_mask else None, page_table=pt_override)
    return pool.out.cpu().numpy(), pool.lse.cpu().numpy(), ref_out, ref_lse


@pytest.mark.parametrize("G", [1, 3, 4, 8])
@pytest.mark.parametrize("ps", [16, 32, 64, 256])
def test_small_ragged(G, ps):
    Hkv = 2
    lens = [0, 1, 15, 16, 17, 100, 127, 128, 129, 3 * ps + 7, 257]
    wl = custom(61 + G + ps, B=len(lens), Hq=G * Hkv, Hkv=Hkv, ps=ps, prompt_lens=lens, steps=0,
                sigma=1.5, outlier_frac=0.02)
    out, lse, ro, rl = _tc_case(wl, num_splits=0)
    assert_attention_close(out, lse, ro, rl, f"tc G={G} ps={ps}")


@pytest.mark.parametrize("Hkv,G", [(1, 8), (1, 1), (16, 4), (32, 2)])
def test_kv_head_counts(Hkv, G):
    lens = [0, 5, 16, 130, 700, 33]
    wl = custom(90 + Hkv + G, B=len(lens), Hq=G * Hkv, Hkv=Hkv, ps=16, prompt_lens=lens, steps=0,
                sigma=1.2, outlier_frac=0.02)
    out, lse, ro, rl = _tc_case(wl, num_splits=0)
    assert_attention_close(out, lse, ro, rl, f"tc Hkv={Hkv} G={G}")


@pytest.mark.parametrize("num_splits", [1, 2, 5, 37, 61, 200, 300, 4096])
def test_split_counts(num_splits):
    # 4096 exceeds the batch's tiles: the count is lowered to one tile per split
    lens = [700, 33, 0, 1025, 64, 5]
    wl = custom(70 + num_splits, B=len(lens), Hq=16, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    out, lse, ro, rl = _tc_case(wl, num_splits=num_splits)
    assert_attention_close(out, lse, ro, rl, f"tc splits={num_splits}")


@pytest.mark.parametrize("abort_one", [False, True])
def test_uniform_batch_one_segment_per_cta(abort_one):
    lens = [200] * 30
    wl = custom(83, B=30, Hq=16, Hkv=8, ps=16, prompt_lens=lens, steps=0)
    abort = None
    if abort_one:
        abort = np.zeros(wl.B, np.uint8)
        abort[7] = 1
    out, lse, ro, rl = _tc_case(wl, 0, abort=abort, use_mask=abort_one)
    assert_attention_close(out, lse, ro, rl, f"tc uniform abort={abort_one}")


@pytest.mark.parametrize("lens", [[700] * 4, [0, 333, 333, 0, 333], [1] * 3, [3000, 80],
                                  [900, 16, 17, 31, 33, 1500, 700, 2, 1200]])
def test_small_batches(lens):
    wl = custom(89 + len(lens), B=len(lens), Hq=64, Hkv=8, ps=16, prompt_lens=lens, steps=0,
                sigma=1.0, outlier_frac=0.01)
    out, lse, ro, rl = _tc_case(wl, 0)
    assert_attention_close(out, lse, ro, rl, f"tc small lens={lens[:3]}")


@pytest.mark.parametrize("num_splits", [305, 1000, 2200])
def test_more_splits_than_a_wave(num_splits):
    lens = [7000, 33, 0, 10250, 640, 5, 1500]
    wl = custom(77 + num_splits, B=len(lens), Hq=16, Hkv=2, ps=16, prompt_lens=lens, steps=0,
                sigma=1.2, outlier_frac=0.02)
    abort = np.zeros(wl.B, np.uint8)
    abort[4] = 1
    out, lse, ro, rl = _tc_case(wl, num_splits, abort=abort, use_mask=True)
    assert_attention_close(out, lse, ro, rl, f"tc splits={num_splits}")


def test_thousands_of_short_requests():
    lens = list(rng_for(91, "lens").integers(0, 71, size=3000))
    wl = custom(91, B=3000, Hq=8, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    out, lse, ro, rl = _tc_case(wl, 0)
    assert_attention_close(out, lse, ro, rl, "tc 3000 short")


@pytest.mark.parametrize("num_splits", [0, 3, 64])
def test_bad_page_id_fails_closed_without_tracker(num_splits):
    lens = [200, 200, 200]
    wl = custom(82, B=3, Hq=8, Hkv=2, ps=16, prompt_lens=lens, steps=0)
    pt = wl.page_table.copy()
    pt[1, 5] = wl.num_pages + 1000        # would read past the pool
    pt[2, 0] = -2
    out, lse, ro, rl = _tc_case(wl, num_splits, use_mask=False, pt_override=pt)
    assert_attention_close(out, lse, ro, rl, "tc bad page")
    assert np.isneginf(lse[1:]).all() and not out[1:].any()


@pytest.mark.parametrize("case", ["uniform", "uneven", "splits200", "wave2000"])
def test_repeated_launches_bit_identical(case):
    if case == "uniform":
        lens, ns = [700] * 30, 0
    elif case == "uneven":
        lens, ns = list(rng_for(85, "lens").integers(1, 1400, size=30)), 0
    elif case == "wave2000":
        lens, ns = list(rng_for(86, "lens").integers(2000, 6000, size=12)), 2000
    else:
        lens, ns = list(rng_for(86, "lens").integers(1, 3000, size=12)), 200
    wl = custom(87, B=len(lens), Hq=16, Hkv=8, ps=16, prompt_lens=lens, steps=0)
    pool = DecodePool(wl, fp8=True, device=DEV, num_splits=ns, tensor_cores=True)
    pool.prefill()
    pool.attend()
    first = pool.out.clone(), pool.lse.clone()
    for _ in range(10):
        pool.out.fill_(float("nan"))
        pool.attend()
        assert torch.equal(pool.out.view(torch.int32), first[0].view(torch.int32))
        assert torch.equal(pool.lse.view(torch.int32), first[1].view(torch.int32))
    assert pool.workspace[:4].view(torch.int32).item() == 0


def _full_size_tc(wl, num_splits=None):
    """One decode step at full size (append + tag check through the step entry
    point), then attention through the tensor-core entry point; every request
    is checked against the oracle."""
    pool = DecodePool(wl, fp8=True, device=DEV, num_splits=num_splits, tensor_cores=True)
    pool.prefill()
    pool.set_step(0)
    pool.step(validate=True)
    pool.out.fill_(float("nan"))
    pool.attend()
    torch.cuda.synchronize()
    assert pool.workspace[:4].view(torch.int32).item() == 0
    lens = wl.seq_lens_after(0)
    mask, _ = oracle.page_tags_validate(wl.page_table, wl.expected_tags, lens, wl.live_tags,
                                        wl.num_pages, wl.page_size)
    got = pool.pool_bytes()
    out, lse = pool.out.cpu().numpy(), pool.lse.cpu().numpy()
    del pool
    torch.cuda.empty_cache()
    ref = oracle_pool_all(wl, True, 1)
    assert np.array_equal(got, ref), "pool bytes differ from the oracle's"
    del got
    ro, rl = oracle_attention_all(wl, ref, True, wl.step_query(0), lens, abort=mask)
    return assert_attention_close(out, lse, ro, rl, f"tc {wl.name}")


def test_b32_8k_full_size_every_request():
    _full_size_tc(b32_8k())


def test_long128k_full_size_every_request_64_splits():
    _full_size_tc(long128k(), num_splits=64 * 4 * 8)
