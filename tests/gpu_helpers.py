"""Shared helpers of the GPU parity tests: oracle reference runs on the same
seeded inputs and the comparison rules (bit-exact bytes and abort sets;
attention within |d| <= 2e-3 + 1e-2 |ref| in fp32 output)."""
import numpy as np

import oracle

ATOL = 2e-3
RTOL = 1e-2


def oracle_pools(wl, fp8, fill=True):
    """The oracle's KV pool after the prompts are written (unwritten slots hold NaN codes)."""
    dt = np.uint8 if fp8 else np.uint16
    n = 2 * wl.num_pages * wl.Hkv * wl.page_size * wl.D
    pool = np.full(n, 0x7F if fp8 else 0x7FC0, dt)
    if fill:
        oracle.kv_prefill(wl.k_prompt, wl.v_prompt, wl.cu_prompt, pool, wl.k_scale, wl.v_scale,
                          wl.page_table, wl.live_tags, wl.expected_tags, None, fp8=fp8, Hkv=wl.Hkv,
                          D=wl.D, page_size=wl.page_size, num_pages=wl.num_pages)
    return pool


def oracle_attention(wl, pool, fp8, q, lens, abort=None, rows=None, page_table=None):
    """fp64 oracle attention, optionally on a subset of requests (`rows`)."""
    pt = wl.page_table if page_table is None else page_table
    if rows is None:
        return oracle.paged_attention(q, pool, pt, lens, fp8=fp8, k_scale=wl.k_scale,
                                      v_scale=wl.v_scale, abort_mask=abort, sm_scale=wl.sm_scale,
                                      Hkv=wl.Hkv, page_size=wl.page_size, num_pages=wl.num_pages)
    rows = list(rows)
    sub_abort = None if abort is None else np.ascontiguousarray(abort[rows])
    return oracle.paged_attention(np.ascontiguousarray(q[rows]), pool, np.ascontiguousarray(pt[rows]),
                                  np.ascontiguousarray(lens[rows]), fp8=fp8, k_scale=wl.k_scale,
                                  v_scale=wl.v_scale, abort_mask=sub_abort, sm_scale=wl.sm_scale,
                                  Hkv=wl.Hkv, page_size=wl.page_size, num_pages=wl.num_pages)


def assert_attention_close(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    dead = np.isneginf(ref_lse)
    # dead (aborted / empty / bad-page) rows: exactly zero output, lse = -inf
    assert np.all(out[dead] == 0.0), f"{what}: nonzero output for a dead request"
    assert np.all(np.isneginf(lse[dead])), f"{what}: finite lse for a dead request"
    live = ~dead
    assert np.all(np.isfinite(out[live])), f"{what}: non-finite output"
    err = np.abs(out[live] - ref_out[live])
    bound = ATOL + RTOL * np.abs(ref_out[live])
    bad = err > bound
    if bad.any():
        i = np.argmax(err - bound)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst |d|="
                             f"{err.flat[i]:.3e} vs bound {bound.flat[i]:.3e} (max-abs "
                             f"{err.max():.3e})")
    lerr = np.abs(lse[live] - ref_lse[live])
    lbound = ATOL + RTOL * np.abs(ref_lse[live])
    assert np.all(lerr <= lbound), f"{what}: lse max err {lerr.max():.3e}"
    return float(err.max()) if err.size else 0.0
