"""Shared helpers of the GPU parity tests: oracle reference runs on the same
seeded inputs and the comparison rules (bit-exact bytes and abort sets;
attention within |d| <= 2e-3 + 1e-2 |ref| in fp32 output)."""
import os

import numpy as np

import oracle

ATOL = 2e-3
RTOL = 1e-2
# lse (natural log of the softmax denominator): the kernel's scores are exact
# f16 products summed in fp32 (error about |s| 2^-21) and its weight sums are
# fp32 chains of at most a few thousand additions even at 131 072 tokens
# (relative error <= 4096 * 2^-24 = 2.4e-4, which is the error of ln W); the
# bound below leaves about four times that.
LSE_ATOL = 1e-3
LSE_RTOL = 2.0 ** -16


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
    lbound = LSE_ATOL + LSE_RTOL * np.abs(ref_lse[live])
    log = os.environ.get("FPK_TEST_ERRLOG")
    if log and err.size:
        with open(log, "a") as f:
            f.write(f"{what}\tout_max_abs={err.max():.3e}\tout_max_rel={(err / (np.abs(ref_out[live]) + 1e-30)).max():.3e}"
                    f"\tlse_max_abs={lerr.max():.3e}\n")
    assert np.all(lerr <= lbound), f"{what}: lse max err {lerr.max():.3e}"
    return float(err.max()) if err.size else 0.0


def _threads(n=None):
    import concurrent.futures as cf
    import os
    return cf.ThreadPoolExecutor(max_workers=n or max(1, min(32, os.cpu_count() or 1)))


def oracle_pool_all(wl, fp8, steps):
    """The oracle's KV pool after every prompt and `steps` decode-step appends,
    built one request per host thread (requests own disjoint pages; the
    oracle's C work releases the interpreter lock)."""
    dt = np.uint8 if fp8 else np.uint16
    n = 2 * wl.num_pages * wl.Hkv * wl.page_size * wl.D
    pool = np.full(n, 0x7F if fp8 else 0x7FC0, dt)
    toks = [wl.step_tokens(s) for s in range(steps)]
    lens = [wl.seq_lens_after(s) for s in range(steps)]

    def one(r):
        a, b = int(wl.cu_prompt[r]), int(wl.cu_prompt[r + 1])
        pt = np.ascontiguousarray(wl.page_table[r:r + 1])
        ex = np.ascontiguousarray(wl.expected_tags[r:r + 1])
        oracle.kv_prefill(wl.k_prompt[a:b], wl.v_prompt[a:b], np.array([0, b - a], np.int32), pool,
                          wl.k_scale, wl.v_scale, pt, wl.live_tags, ex, None, fp8=fp8, Hkv=wl.Hkv,
                          D=wl.D, page_size=wl.page_size, num_pages=wl.num_pages)
        for s in range(steps):
            kn, vn = toks[s]
            oracle.kv_append(kn[r:r + 1], vn[r:r + 1], pool, wl.k_scale, wl.v_scale, pt,
                             lens[s][r:r + 1], wl.live_tags, ex, None, fp8=fp8, Hkv=wl.Hkv, D=wl.D,
                             page_size=wl.page_size, num_pages=wl.num_pages)

    with _threads() as ex_:
        list(ex_.map(one, range(wl.B)))
    return pool


def oracle_attention_all(wl, pool, fp8, q, lens, abort=None):
    """fp64 oracle attention of every request, one request per host thread."""
    out = np.empty((wl.B, wl.Hq, wl.D), np.float64)
    lse = np.empty((wl.B, wl.Hq), np.float64)

    def one(r):
        o, l_ = oracle_attention(wl, pool, fp8, q, lens, abort=abort, rows=[r])
        out[r], lse[r] = o[0], l_[0]

    with _threads() as ex_:
        list(ex_.map(one, range(wl.B)))
    return out, lse
