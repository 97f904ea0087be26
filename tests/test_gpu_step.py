"""The whole decode step as one call (fpk_decode_step_*): the write + tag check
kernel, then attention launched as its programmatic dependent.

It must give exactly what the two launches give one after the other (same
kernels, same split: bit-identical), match the oracle (cache bytes and abort
mask bit-exact, attention within tolerance), behave the same inside a CUDA
graph, and launch nothing when an argument is rejected.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300 import FpkError, fpk_decode_step_fp8
from fp8_paged_kv_gb300.pool import DecodePool, to_device
from tests.gpu_helpers import assert_attention_close, oracle_attention, oracle_pools
from workloads import custom, tiny

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _workload(what):
    ps = 16
    wl = custom(57, B=7, Hq=16, Hkv=2, ps=ps, prompt_lens=[20, 700, 15, 31, 0, 300, 64], steps=1,
                sigma=1.5, outlier_frac=0.02)
    pt, ex = wl.page_table.copy(), wl.expected_tags.copy()
    if what == "stale_inner":
        ex[1, 3] -= np.uint32(1)
    elif what == "page_oob":
        pt[5, 2] = wl.num_pages + 1
    wl.page_table, wl.expected_tags = pt, ex
    return wl


def _fresh(wl, fp8, num_splits):
    pool = DecodePool(wl, fp8=fp8, device=DEV, num_splits=num_splits)
    pool.prefill()
    pool.set_step(0)
    pool.count_aborts = False
    return pool


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("what", ["none", "stale_inner", "page_oob"])
@pytest.mark.parametrize("num_splits", [0, 37])
def test_step_equals_separate_launches_and_oracle(fp8, what, num_splits):
    wl = _workload(what)
    a = _fresh(wl, fp8, num_splits)
    a.step(validate=True)                     # one call, dependent launch
    b = _fresh(wl, fp8, num_splits)
    b.append_check()                          # the same two kernels, plain launches
    b.attend(use_mask=True)
    torch.cuda.synchronize()
    assert np.array_equal(a.pool_bytes(), b.pool_bytes())
    assert torch.equal(a.abort_mask, b.abort_mask)
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)
    assert a.workspace[:4].view(torch.int32).item() == 0

    # against the oracle: append, check, attention over the passing requests
    ref = oracle_pools(wl, fp8)
    kn, vn = wl.step_tokens(0)
    lens = wl.seq_lens_after(0)
    oracle.kv_append(kn, vn, ref, wl.k_scale, wl.v_scale, wl.page_table, lens, wl.live_tags,
                     wl.expected_tags, None, fp8=fp8, Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size,
                     num_pages=wl.num_pages)
    mask, _ = oracle.page_tags_validate(wl.page_table, wl.expected_tags, lens, wl.live_tags,
                                        wl.num_pages, wl.page_size)
    assert np.array_equal(a.pool_bytes(), ref)
    assert np.array_equal(a.abort_mask.cpu().numpy(), mask)
    assert bool(mask.any()) == (what != "none")
    ro, rl = oracle_attention(wl, ref, fp8, wl.step_query(0), lens, abort=mask)
    assert_attention_close(a.out.cpu().numpy(), a.lse.cpu().numpy(), ro, rl, f"step {what}")


@pytest.mark.parametrize("fp8", [True, False])
def test_noop_tracker_step_equals_separate_launches(fp8):
    # a tag goes stale after the prompts were written; the no-op tracker does
    # not check it: nothing aborts and request 1 is attended like the others
    wl = _workload("none")
    pools = []
    for _ in range(2):
        p = _fresh(wl, fp8, 0)
        p.expected_tags[1, 3] += 1
        p.abort_mask.fill_(5)
        pools.append(p)
    a, b = pools
    a.step(validate=False)
    b.append(guard=False)
    b.attend(use_mask=False)
    torch.cuda.synchronize()
    assert np.array_equal(a.pool_bytes(), b.pool_bytes())
    assert torch.equal(a.out.view(torch.int32), b.out.view(torch.int32))
    assert torch.equal(a.lse.view(torch.int32), b.lse.view(torch.int32))
    assert bool((a.abort_mask == 5).all())                    # untouched
    live = torch.tensor([True, True, True, True, True, True, True], device=DEV)
    assert bool(torch.isfinite(a.lse[live]).all())            # all attended, request 1 too


def test_step_in_a_cuda_graph():
    wl = _workload("stale_inner")
    a = _fresh(wl, True, 0)
    a.step(validate=True)
    torch.cuda.synchronize()
    want_out, want_mask = a.out.clone(), a.abort_mask.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        a.step(validate=True)                 # warm-up on the capture stream
        with torch.cuda.graph(g, stream=s):
            a.step(validate=True)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        a.out.fill_(float("nan"))
        a.abort_mask.fill_(7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(a.out, want_out) and torch.equal(a.abort_mask, want_mask)


def test_rejected_step_launches_nothing():
    wl = _workload("none")
    a = _fresh(wl, True, 0)
    before = a.pool_bytes().copy()
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)   # far too small a workspace
    with pytest.raises(FpkError):
        fpk_decode_step_fp8(a.k_new, a.v_new, a.kv_pool, a.k_scale, a.v_scale, a.page_table,
                            a.seq_lens, a.live_tags, a.expected_tags, a.abort_mask, a.q, a.out,
                            a.lse, small, Hkv=wl.Hkv, page_size=wl.page_size,
                            num_pages=wl.num_pages, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert np.array_equal(a.pool_bytes(), before)   # the write did not run either


def test_bounded_wait_gives_up_and_reports():
    """A wait that nothing completes ends after its limit with the timeout bit
    set, and the context stays usable (a full decode step runs after it)."""
    from fp8_paged_kv_gb300 import fpk_selftest_bounded_wait
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    fpk_selftest_bounded_wait(status, elapsed)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert 1.9e9 <= int(elapsed.item()) <= 4e9
    wl = tiny()
    pool = DecodePool(wl, fp8=True, device=DEV)
    pool.prefill()
    pool.set_step(0)
    pool.count_aborts = False
    pool.step(validate=True)
    torch.cuda.synchronize()
    assert pool.workspace[:4].view(torch.int32).item() == 0
    assert list(pool.abort_mask.cpu().numpy()) == [0, 1]
