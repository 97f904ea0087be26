"""Churn + integrity on the GPU: continuous batching with page reallocation and
injected stale lookups, abort sets bit-exact against the oracle at every step.

The scenario is the integrity evaluation's shape in the Cloudflare write-up
("La sicurezza della cache KV condivisa diventa una questione di
produzione", remio.ai: 8192-token inputs, 1000 output tokens): 256 request
slots, Hq=32/Hkv=8, page size 16; every 50 steps 10 % of the requests finish
and their pages are reallocated (tags bumped); each step every request's
lookup goes stale with probability 1 %.  The host ledger decides; the device
bumps its live tags, writes the step's tokens and checks every mapping in one
launch, then attends.  The oracle bumps its own copy of the tags and runs its
own check on the same tables.  Only tags and abort sets are compared here, so
the cache values are drawn on the device.  A smaller run
(test_churn_attention_matches_oracle) draws every value on the host instead, so
that the oracle keeps its own pool through every prompt write and append:
there the attention outputs under churn are compared too.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_gb300 import (fpk_decode_append_check_fp8, fpk_decode_workspace_bytes,
                                fpk_kv_prefill_fp8, fpk_page_tags_bump, fpk_page_tags_validate,
                                fpk_paged_decode_attn_fp8)
from fp8_paged_kv_gb300.pool import to_device
from tests.gpu_helpers import _threads, assert_attention_close
from workloads import bf16_bits, rng_for
from workloads.churn import ChurnScenario

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _prefill(sc, kv_pool, k_scale, v_scale, page_table_rows, live, expected_rows, gen, n_tok):
    """Write `len(rows)` prompts of n_tok tokens each (values drawn on the device)."""
    R = page_table_rows.shape[0]
    k = torch.randn(R * n_tok, sc.Hkv, sc.D, device=DEV, generator=gen).to(torch.bfloat16)
    v = torch.randn(R * n_tok, sc.Hkv, sc.D, device=DEV, generator=gen).to(torch.bfloat16)
    cu = torch.arange(0, (R + 1) * n_tok, n_tok, dtype=torch.int32, device=DEV)
    fpk_kv_prefill_fp8(k, v, cu, kv_pool, k_scale, v_scale, page_table_rows, live, expected_rows,
                       None, Hkv=sc.Hkv, D=sc.D, page_size=sc.ps, num_pages=sc.num_pages)


@pytest.mark.parametrize("steps", [1000])
def test_churn_abort_sets_bit_exact(steps):
    sc = ChurnScenario(steps=steps)
    L = sc.ledger
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    kv_pool = torch.full((2 * sc.num_pages * sc.Hkv * sc.ps * sc.D,), 0x7F, dtype=torch.uint8,
                         device=DEV)
    k_scale = torch.tensor([4.5 / 448], device=DEV)
    v_scale = torch.tensor([4.5 / 448], device=DEV)
    live_d = to_device(sc.initial_tags, DEV)
    live_o = sc.initial_tags.copy()
    pt_d = to_device(L.page_table, DEV)
    ex_d = to_device(L.expected, DEV)
    for r0 in range(0, sc.B, 16):
        _prefill(sc, kv_pool, k_scale, v_scale, pt_d[r0:r0 + 16], live_d, ex_d[r0:r0 + 16], gen,
                 sc.prompt)
    torch.cuda.synchronize()
    mask_d = torch.zeros(sc.B, dtype=torch.uint8, device=DEV)
    out = torch.empty(sc.B, sc.Hq, sc.D, device=DEV)
    lse = torch.empty(sc.B, sc.Hq, device=DEV)
    ws = torch.zeros(fpk_decode_workspace_bytes(sc.B, sc.Hq, sc.Hkv, sc.D, 0), dtype=torch.uint8,
                     device=DEV)
    aborted = ()
    n_abort = n_admit = 0
    check_ms = attn_ms = 0.0
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for s in range(steps):
        ev = sc.next_step(s, aborted)
        # device: reallocation bumps, table upload, prompts of admitted requests
        if ev.bump.size:
            fpk_page_tags_bump(live_d, to_device(ev.bump, DEV), num_pages=sc.num_pages)
        pt_d.copy_(to_device(L.page_table, DEV))
        ex_d.copy_(to_device(L.expected, DEV))
        for r in ev.admitted:
            _prefill(sc, kv_pool, k_scale, v_scale, pt_d[r:r + 1], live_d, ex_d[r:r + 1], gen,
                     sc.prompt)
        lens_d = to_device(ev.lens, DEV)
        k_new = torch.randn(sc.B, sc.Hkv, sc.D, device=DEV, generator=gen).to(torch.bfloat16)
        v_new = torch.randn(sc.B, sc.Hkv, sc.D, device=DEV, generator=gen).to(torch.bfloat16)
        q = torch.randn(sc.B, sc.Hq, sc.D, device=DEV, generator=gen).to(torch.bfloat16)
        e[0].record()
        fpk_decode_append_check_fp8(k_new, v_new, kv_pool, k_scale, v_scale, pt_d, lens_d, live_d,
                                    ex_d, mask_d, Hkv=sc.Hkv, D=sc.D, page_size=sc.ps,
                                    num_pages=sc.num_pages)
        e[1].record()
        fpk_paged_decode_attn_fp8(q, kv_pool, k_scale, v_scale, pt_d, lens_d, mask_d, out, lse, ws,
                                  Hkv=sc.Hkv, page_size=sc.ps, num_pages=sc.num_pages,
                                  sm_scale=sc.sm_scale)
        e[2].record()
        # oracle: its own tags, its own check on the same tables
        oracle.page_tags_bump(live_o, ev.bump, sc.num_pages)
        want, n = oracle.page_tags_validate(L.page_table, L.expected, ev.lens, live_o,
                                            sc.num_pages, sc.ps)
        got = mask_d.cpu().numpy()
        assert np.array_equal(got, want), f"abort set differs at step {s}"
        assert set(np.flatnonzero(want)) == set(ev.corrupted), f"injected set differs at step {s}"
        if s % 50 == 0:
            o = out.cpu().numpy()
            ls = lse.cpu().numpy()
            dead = want.astype(bool)
            assert not o[dead].any() and np.isneginf(ls[dead]).all()
            assert np.isfinite(o[~dead]).all() and np.isfinite(ls[~dead]).all()
        check_ms += e[0].elapsed_time(e[1])
        attn_ms += e[1].elapsed_time(e[2])
        aborted = tuple(np.flatnonzero(want))
        n_abort += int(n)
        n_admit += len(ev.admitted)
    assert np.array_equal(live_d.cpu().numpy().view(np.uint32), live_o)
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert n_abort > 0 and n_admit > 0
    # the batched check alone against attention on the final tables: n launches
    # captured in one CUDA graph, so host launch cost stays out of the device time
    def per_launch_us(fn, n):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n
    chk = torch.zeros(sc.B, dtype=torch.uint8, device=DEV)
    val_us = per_launch_us(lambda: fpk_page_tags_validate(pt_d, ex_d, lens_d, live_d, chk, None,
                                                          num_pages=sc.num_pages, page_size=sc.ps), 50)
    att_us = per_launch_us(lambda: fpk_paged_decode_attn_fp8(q, kv_pool, k_scale, v_scale, pt_d, lens_d,
                                                             chk, out, lse, ws, Hkv=sc.Hkv,
                                                             page_size=sc.ps, num_pages=sc.num_pages,
                                                             sm_scale=sc.sm_scale), 10)
    print(f"churn: {steps} steps, {n_abort} aborts, {n_admit} admissions; per step (host-synchronised): "
          f"write+check {check_ms / steps * 1e3:.1f} us, attention {attn_ms / steps * 1e3:.1f} us; "
          f"in one graph: check {val_us:.1f} us vs attention {att_us:.1f} us ({100 * val_us / att_us:.2f} %)")


def _host_bf16(g, shape):
    return bf16_bits(g.standard_normal(shape, dtype=np.float32))


def test_churn_attention_matches_oracle():
    """Churn at a smaller scale (32 slots, 1024-token prompts, 200 steps, the
    same event rules) with every prompt, new token and query drawn on the
    host: the oracle bumps its own tags and writes its own pool through every
    admission and append.  Abort sets bit-exact at every step; attention of
    every request at every 50th step and at the last within the standard
    tolerance; the whole pool bit-exact at the end."""
    sc = ChurnScenario(seed=9, B=32, prompt=1024, steps=200)
    L = sc.ledger
    scale = np.float32(4.5 / 448)
    n = 2 * sc.num_pages * sc.Hkv * sc.ps * sc.D
    pool_o = np.full(n, 0x7F, np.uint8)
    kv_pool = torch.full((n,), 0x7F, dtype=torch.uint8, device=DEV)
    k_scale = torch.tensor([float(scale)], device=DEV)
    v_scale = torch.tensor([float(scale)], device=DEV)
    live_o = sc.initial_tags.copy()
    live_d = to_device(live_o, DEV)
    dims = dict(Hkv=sc.Hkv, D=sc.D, page_size=sc.ps, num_pages=sc.num_pages)

    def prefill(rows, g):
        R = len(rows)
        k = _host_bf16(g, (R * sc.prompt, sc.Hkv, sc.D))
        v = _host_bf16(g, (R * sc.prompt, sc.Hkv, sc.D))
        cu = np.arange(0, (R + 1) * sc.prompt, sc.prompt, dtype=np.int32)
        pt = np.ascontiguousarray(L.page_table[rows])
        ex = np.ascontiguousarray(L.expected[rows])
        fpk_kv_prefill_fp8(to_device(k, DEV), to_device(v, DEV), to_device(cu, DEV), kv_pool, k_scale,
                           v_scale, to_device(pt, DEV), live_d, to_device(ex, DEV), None, **dims)
        oracle.kv_prefill(k, v, cu, pool_o, scale, scale, pt, live_o, ex, None, fp8=True, **dims)

    prefill(list(range(sc.B)), rng_for(9, "churn-prompts"))
    pt_d = to_device(L.page_table, DEV)
    ex_d = to_device(L.expected, DEV)
    mask_d = torch.zeros(sc.B, dtype=torch.uint8, device=DEV)
    out = torch.empty(sc.B, sc.Hq, sc.D, device=DEV)
    lse = torch.empty(sc.B, sc.Hq, device=DEV)
    ws = torch.zeros(fpk_decode_workspace_bytes(sc.B, sc.Hq, sc.Hkv, sc.D, 0), dtype=torch.uint8,
                     device=DEV)
    aborted = ()
    n_abort = n_admit = checked = 0
    for s in range(sc.steps):
        ev = sc.next_step(s, aborted)
        if ev.bump.size:
            fpk_page_tags_bump(live_d, to_device(ev.bump, DEV), num_pages=sc.num_pages)
            oracle.page_tags_bump(live_o, ev.bump, sc.num_pages)
        pt_d.copy_(to_device(L.page_table, DEV))
        ex_d.copy_(to_device(L.expected, DEV))
        g = rng_for(9, "churn-step", s)
        if ev.admitted:
            prefill(list(ev.admitted), g)
        k_new = _host_bf16(g, (sc.B, sc.Hkv, sc.D))
        v_new = _host_bf16(g, (sc.B, sc.Hkv, sc.D))
        q = _host_bf16(g, (sc.B, sc.Hq, sc.D))
        lens = ev.lens
        lens_d = to_device(lens, DEV)
        fpk_decode_append_check_fp8(to_device(k_new, DEV), to_device(v_new, DEV), kv_pool, k_scale,
                                    v_scale, pt_d, lens_d, live_d, ex_d, mask_d, **dims)
        fpk_paged_decode_attn_fp8(to_device(q, DEV), kv_pool, k_scale, v_scale, pt_d, lens_d, mask_d,
                                  out, lse, ws, Hkv=sc.Hkv, page_size=sc.ps,
                                  num_pages=sc.num_pages, sm_scale=sc.sm_scale)
        oracle.kv_append(k_new, v_new, pool_o, scale, scale, L.page_table, lens, live_o, L.expected,
                         None, fp8=True, **dims)
        want, nab = oracle.page_tags_validate(L.page_table, L.expected, lens, live_o, sc.num_pages,
                                              sc.ps)
        assert np.array_equal(mask_d.cpu().numpy(), want), f"abort set differs at step {s}"
        if s % 50 == 0 or s == sc.steps - 1:
            ref_o = np.empty((sc.B, sc.Hq, sc.D))
            ref_l = np.empty((sc.B, sc.Hq))

            def one(r):
                o, l_ = oracle.paged_attention(
                    np.ascontiguousarray(q[r:r + 1]), pool_o, np.ascontiguousarray(L.page_table[r:r + 1]),
                    np.ascontiguousarray(lens[r:r + 1]), fp8=True, k_scale=scale, v_scale=scale,
                    abort_mask=np.ascontiguousarray(want[r:r + 1]), sm_scale=sc.sm_scale, Hkv=sc.Hkv,
                    page_size=sc.ps, num_pages=sc.num_pages)
                ref_o[r], ref_l[r] = o[0], l_[0]

            with _threads() as ex_:
                list(ex_.map(one, range(sc.B)))
            assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, f"churn step {s}")
            checked += 1
        aborted = tuple(np.flatnonzero(want))
        n_abort += int(nab)
        n_admit += len(ev.admitted)
    assert checked == 5 and n_abort > 0 and n_admit > 0
    assert np.array_equal(live_d.cpu().numpy().view(np.uint32), live_o)
    assert np.array_equal(kv_pool.cpu().numpy(), pool_o), "pool bytes differ from the oracle's"
    assert int(ws[:4].view(torch.int32).item()) == 0
