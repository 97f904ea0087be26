"""The allocation-free FP8 attention entry point gives the workspace one's results.

fpk_paged_decode_attn_fp8_noalloc serves callers that cannot allocate device
memory (operator hosts that hand an operator only its inputs and outputs,
fixed device-memory budgets, loops that cannot take cudaMalloc's implicit
synchronisation): its scratch is a fixed array inside the library.  Both entry
points run the same kernel with the same partition of the work, so their
results must agree to the bit; a partial or counter left in the shared
scratch by an earlier call would show up as a difference.  This test calls
the allocation-free entry point through the C ABI three times in a row -- a
small batch, a larger one with many more splits, then a small one again, so
the later calls run on scratch the earlier ones left behind -- and checks each
result bit for bit against fpk_paged_decode_attn_fp8 on the same inputs and
split count, and against the fp64 oracle within the tolerance every attention
test uses.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from fp8_paged_kv_gb300 import fpk_decode_status, fpk_paged_decode_attn_fp8_noalloc
from fp8_paged_kv_gb300.pool import DecodePool, to_device
from tests.gpu_helpers import assert_attention_close, oracle_attention, oracle_pools
from workloads import custom

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check(pool, abort=None):
    wl = pool.wl
    if abort is not None:
        pool.abort_mask = to_device(abort.astype(np.uint8), DEV)
    use_mask = abort is not None
    pool.out.fill_(float("nan"))
    pool.lse.fill_(float("nan"))
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
    assert fpk_decode_status(None) == 0, "a bounded wait gave up in the allocation-free call"
    assert fpk_decode_status(pool.workspace) == 0
    # same kernel, same partition: identical bits (NaN sentinels included)
    assert torch.equal(out.view(torch.int32), ref_out.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    ref = oracle_pools(wl, True)
    lens = wl.prompt_lens.astype(np.int32)
    ro, rl = oracle_attention(wl, ref, True, wl.q, lens, abort=abort)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, wl.name)


def test_noalloc_matches_workspace_entry_point_three_calls_in_a_row():
    # first call: ragged contexts, one aborted request, automatic split count
    wl1 = custom(91, B=6, Hq=32, Hkv=4, ps=16, prompt_lens=[0, 1, 300, 77, 1500, 64], steps=0)
    p1 = DecodePool(wl1, fp8=True, device=DEV)
    p1.prefill()
    _check(p1, abort=np.array([0, 0, 0, 1, 0, 0], np.uint8))
    # second call: a larger batch with 2000 splits (two-level combine), so
    # partials and arrival counters cover much more of the scratch
    wl2 = custom(92, B=5, Hq=64, Hkv=8, ps=64, prompt_lens=[4000, 129, 2049, 3333, 700], steps=0)
    p2 = DecodePool(wl2, fp8=True, device=DEV, num_splits=2000)
    p2.prefill()
    _check(p2)
    # third call: a small batch again, on the scratch the larger one left
    wl3 = custom(94, B=3, Hq=16, Hkv=2, ps=32, prompt_lens=[900, 33, 1200], steps=0)
    p3 = DecodePool(wl3, fp8=True, device=DEV, num_splits=7)
    p3.prefill()
    _check(p3)


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
