"""The allocation-free FP8 attention entry point matches the workspace one.

fpk_paged_decode_attn_fp8_noalloc serves callers that cannot allocate device
memory (operator hosts that hand an operator only its inputs and outputs,
fixed device-memory budgets, loops that cannot take cudaMalloc's implicit
synchronisation): its scratch is a fixed array inside the library.  This test
calls it through the C ABI twice in a row -- on two different batches, so the
second call runs on scratch the first one left behind -- and compares each
result with fpk_paged_decode_attn_fp8 on the same inputs, within the
tolerance every attention test uses.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from fp8_paged_kv_gb300 import fpk_paged_decode_attn_fp8_noalloc
from fp8_paged_kv_gb300.pool import DecodePool, to_device
from workloads import custom

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ATOL, RTOL = 2e-3, 1e-2


def _compare(pool, use_mask):
    wl = pool.wl
    pool.attend(use_mask=use_mask)
    ref_out = pool.out.clone()
    ref_lse = pool.lse.clone()
    out = torch.full_like(pool.out, float("nan"))
    lse = torch.full_like(pool.lse, float("nan"))
    fpk_paged_decode_attn_fp8_noalloc(pool.q, pool.kv_pool, pool.k_scale, pool.v_scale,
                                      pool.page_table, pool.seq_lens,
                                      pool.abort_mask if use_mask else None, out, lse, Hkv=wl.Hkv,
                                      page_size=wl.page_size, num_pages=wl.num_pages,
                                      sm_scale=wl.sm_scale, num_splits=pool.num_splits)
    torch.cuda.synchronize()
    o, r = out.cpu().numpy().astype(np.float64), ref_out.cpu().numpy().astype(np.float64)
    lo, lr = lse.cpu().numpy().astype(np.float64), ref_lse.cpu().numpy().astype(np.float64)
    dead = np.isneginf(lr)
    assert np.array_equal(np.isneginf(lo), dead)
    assert np.all(o[dead] == 0.0) and np.all(np.isfinite(o))
    assert np.all(np.abs(o - r) <= ATOL + RTOL * np.abs(r))
    live = ~dead
    assert np.all(np.abs(lo[live] - lr[live]) <= ATOL + RTOL * np.abs(lr[live]))


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    # first call: ragged contexts, one aborted request, automatic split count
    wl1 = custom(91, B=6, Hq=32, Hkv=4, ps=16, prompt_lens=[0, 1, 300, 77, 1500, 64], steps=0)
    p1 = DecodePool(wl1, fp8=True, device=DEV)
    p1.prefill()
    p1.abort_mask = to_device(np.array([0, 0, 0, 1, 0, 0], np.uint8), DEV)
    _compare(p1, use_mask=True)
    # second call: another batch and a fixed split count, so partials and
    # arrival counters from the first call are reused
    wl2 = custom(92, B=3, Hq=64, Hkv=8, ps=64, prompt_lens=[4000, 129, 2049], steps=0)
    p2 = DecodePool(wl2, fp8=True, device=DEV, num_splits=200)
    p2.prefill()
    _compare(p2, use_mask=False)


def test_noalloc_rejects_a_batch_larger_than_its_scratch():
    from fp8_paged_kv_gb300 import FpkError
    wl = custom(93, B=2, Hq=8, Hkv=1, ps=16, prompt_lens=[40, 40], steps=0)
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    with pytest.raises(FpkError, match="status 3"):
        # 20 000 splits need ~80 MB of partials, beyond the fixed 16 MiB
        fpk_paged_decode_attn_fp8_noalloc(pool.q, pool.kv_pool, pool.k_scale,
                                          pool.v_scale, pool.page_table, pool.seq_lens, None,
                                          pool.out, pool.lse, Hkv=wl.Hkv, page_size=16,
                                          num_pages=wl.num_pages, sm_scale=wl.sm_scale,
                                          num_splits=20000)
