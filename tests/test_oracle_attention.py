"""Pins of the oracle's paged decode attention (fp64).

The pages (Cloudflare write-up, Italian edition, "Perche le cache piu piccole
di Cloudflare battono la velocita pura") say only that the attention kernel
converts the FP8 values as it reads them, and ("La sicurezza della cache KV
condivisa...") that paged attention maps each sequence's logical blocks to
physical pages.  They print no numbers for attention, so the oracle is pinned
by closed forms and by independent routines:

* uniform keys give the exact mean of the values; one token gives its value;
* the paged walk equals a dense textbook attention on gathered rows;
* it equals torch's scaled_dot_product_attention in float64 (library routine);
* moving pages in the pool (and the table with them) changes nothing;
* a power-of-two k_scale folds into the query exactly;
* aborted, empty and bad-page requests give zeros and lse = -inf.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, bf16_to_f32, custom


def _pools(wl, fp8):
    """The KV pool after the prompts are written (the oracle's own writer)."""
    dt = np.uint8 if fp8 else np.uint16
    n = 2 * wl.num_pages * wl.Hkv * wl.page_size * wl.D
    pool = np.zeros(n, dt)
    oracle.kv_prefill(wl.k_prompt, wl.v_prompt, wl.cu_prompt, pool, wl.k_scale, wl.v_scale,
                      wl.page_table, None, None, None, fp8=fp8, Hkv=wl.Hkv, D=wl.D,
                      page_size=wl.page_size, num_pages=wl.num_pages)
    return pool, pool


def _gather(wl, kp, vp, fp8, r, h, L):
    """Dense [L][D] float64 K-hat and V-hat of (request r, kv head h) from the pool layout
    [page][kv head][tile of 16 tokens][K block [16][D], V block [D][16]]."""
    ps, D, Hkv = wl.page_size, wl.D, wl.Hkv
    K = np.empty((L, D))
    V = np.empty((L, D))
    for j in range(L):
        page = int(wl.page_table[r, j // ps])
        off = j % ps
        base = (((page * Hkv + h) * (ps // 16) + off // 16) * 2) * 16 * D
        ki = base + (off % 16) * D + np.arange(D)
        vi = base + 16 * D + np.arange(D) * 16 + off % 16
        if fp8:
            K[j] = oracle.e4m3_decode(kp[ki]) * float(wl.k_scale)
            V[j] = oracle.e4m3_decode(vp[vi]) * float(wl.v_scale)
        else:
            K[j] = bf16_to_f32(kp[ki])
            V[j] = bf16_to_f32(vp[vi])
    return K, V


def _attn(wl, kp, vp, fp8, lens, abort=None, pt=None):
    assert kp is vp                                 # one KV pool
    return oracle.paged_attention(wl.q, kp, wl.page_table if pt is None else pt, lens, fp8=fp8,
                                  k_scale=wl.k_scale, v_scale=wl.v_scale, abort_mask=abort,
                                  sm_scale=wl.sm_scale, Hkv=wl.Hkv, page_size=wl.page_size,
                                  num_pages=wl.num_pages)


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("ps", [16, 32, 64])
def test_paged_equals_dense_bruteforce(fp8, ps):
    wl = custom(31, B=2, Hq=8, Hkv=2, ps=ps, prompt_lens=[40, 23], steps=0, pool_factor=3.0)
    kp, vp = _pools(wl, fp8)
    lens = wl.prompt_lens
    out, lse = _attn(wl, kp, vp, fp8, lens)
    for r in range(wl.B):
        for h in range(wl.Hq):
            K, V = _gather(wl, kp, vp, fp8, r, h // wl.G, int(lens[r]))
            q = bf16_to_f32(wl.q[r, h]).astype(np.float64)
            o, l = oracle.dense_attention(q, K, V, wl.sm_scale)
            assert np.allclose(out[r, h], o, rtol=1e-12, atol=1e-12)
            assert abs(lse[r, h] - l) < 1e-12


@pytest.mark.parametrize("fp8", [True, False])
def test_matches_torch_sdpa_float64(fp8):
    wl = custom(32, B=3, Hq=8, Hkv=2, ps=16, prompt_lens=[1, 17, 64], steps=0, sigma=2.0)
    kp, vp = _pools(wl, fp8)
    lens = wl.prompt_lens
    out, lse = _attn(wl, kp, vp, fp8, lens)
    for r in range(wl.B):
        L = int(lens[r])
        Ks, Vs = [], []
        for h in range(wl.Hkv):
            K, V = _gather(wl, kp, vp, fp8, r, h, L)
            Ks.append(K)
            Vs.append(V)
        K = torch.tensor(np.stack(Ks)).repeat_interleave(wl.G, dim=0)     # [Hq][L][D]
        V = torch.tensor(np.stack(Vs)).repeat_interleave(wl.G, dim=0)
        q = torch.tensor(bf16_to_f32(wl.q[r]).astype(np.float64))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=wl.sm_scale)[:, 0]
        assert np.allclose(out[r], ref.numpy(), rtol=1e-10, atol=1e-12)
        s = torch.einsum("hd,hld->hl", q[:, 0], K) * wl.sm_scale
        assert np.allclose(lse[r], torch.logsumexp(s, dim=1).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fp8", [True, False])
def test_uniform_keys_give_mean_of_values(fp8):
    wl = custom(33, B=1, Hq=4, Hkv=1, ps=16, prompt_lens=[37], steps=0)
    # every key row identical -> equal scores -> out = mean(V-hat)
    wl.k_prompt[:] = wl.k_prompt[0]
    kp, vp = _pools(wl, fp8)
    out, lse = _attn(wl, kp, vp, fp8, wl.prompt_lens)
    K, V = _gather(wl, kp, vp, fp8, 0, 0, 37)
    for h in range(4):
        assert np.allclose(out[0, h], V.mean(axis=0), rtol=1e-13, atol=1e-15)
        s = float(np.dot(bf16_to_f32(wl.q[0, h]).astype(np.float64), K[0])) * wl.sm_scale
        assert abs(lse[0, h] - (s + math.log(37))) < 1e-12


@pytest.mark.parametrize("fp8", [True, False])
def test_single_token_returns_its_value(fp8):
    wl = custom(34, B=2, Hq=8, Hkv=2, ps=16, prompt_lens=[1, 1], steps=0)
    kp, vp = _pools(wl, fp8)
    out, lse = _attn(wl, kp, vp, fp8, wl.prompt_lens)
    for r in range(2):
        for h in range(8):
            K, V = _gather(wl, kp, vp, fp8, r, h // 4, 1)
            assert np.array_equal(out[r, h], V[0])
            s = float(np.dot(bf16_to_f32(wl.q[r, h]).astype(np.float64), K[0])) * wl.sm_scale
            assert abs(lse[r, h] - s) < 1e-12


def test_physical_page_permutation_invariance():
    wl = custom(35, B=2, Hq=8, Hkv=2, ps=16, prompt_lens=[50, 70], steps=0, pool_factor=2.0)
    kp, vp = _pools(wl, True)
    out0, lse0 = _attn(wl, kp, vp, True, wl.prompt_lens)
    g = np.random.default_rng(3)
    perm = g.permutation(wl.num_pages)           # physical page p moves to perm[p]
    blk = 2 * wl.Hkv * wl.page_size * wl.D         # one page: K and V of every kv head
    kp2 = np.empty_like(kp)
    for p in range(wl.num_pages):
        kp2[perm[p] * blk:(perm[p] + 1) * blk] = kp[p * blk:(p + 1) * blk]
    vp2 = kp2
    pt2 = wl.page_table.copy()
    m = pt2 >= 0
    pt2[m] = perm[pt2[m]]
    out1, lse1 = _attn(wl, kp2, vp2, True, wl.prompt_lens, pt=pt2)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_power_of_two_k_scale_folds_into_query():
    wl = custom(36, B=1, Hq=4, Hkv=1, ps=16, prompt_lens=[45], steps=0)
    kp, vp = _pools(wl, True)
    out_a, lse_a = oracle.paged_attention(wl.q, kp, wl.page_table, wl.prompt_lens, fp8=True,
                                          k_scale=4.0, v_scale=1.0, sm_scale=wl.sm_scale, Hkv=1,
                                          page_size=16, num_pages=wl.num_pages)
    q4 = bf16_bits(bf16_to_f32(wl.q) * np.float32(4))
    out_b, lse_b = oracle.paged_attention(q4, kp, wl.page_table, wl.prompt_lens, fp8=True,
                                          k_scale=1.0, v_scale=1.0, sm_scale=wl.sm_scale, Hkv=1,
                                          page_size=16, num_pages=wl.num_pages)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_dead_requests_give_zero_and_minus_inf():
    wl = custom(37, B=4, Hq=8, Hkv=2, ps=16, prompt_lens=[20, 20, 20, 20], steps=0)
    kp, vp = _pools(wl, True)
    lens = wl.prompt_lens.copy()
    lens[1] = 0                                     # empty
    abort = np.array([0, 0, 1, 0], np.uint8)        # aborted by the tag check
    pt = wl.page_table.copy()
    pt[3, 1] = wl.num_pages + 5                     # bad page id: fail closed
    out, lse = _attn(wl, kp, vp, True, lens, abort=abort, pt=pt)
    for r in (1, 2, 3):
        assert not out[r].any() and np.isneginf(lse[r]).all()
    assert np.isfinite(lse[0]).all() and out[0].any()


def test_gqa_head_mapping():
    """Query head h reads kv head h // G: zeroing kv head 1's values only changes heads 4..7."""
    wl = custom(38, B=1, Hq=8, Hkv=2, ps=16, prompt_lens=[19], steps=0)
    kp, vp = _pools(wl, False)
    out0, _ = _attn(wl, kp, vp, False, wl.prompt_lens)
    vp2 = vp.copy()
    page = int(wl.page_table[0, 0])
    # zero kv head 1's V blocks on page 0 (each 16-token tile: K block, then V block)
    D, ps = wl.D, wl.page_size
    for t in range(ps // 16):
        base = (((page * 2 + 1) * (ps // 16) + t) * 2) * 16 * D
        vp2[base + 16 * D: base + 32 * D] = 0
    out1, _ = _attn(wl, vp2, vp2, False, wl.prompt_lens)
    assert np.array_equal(out0[0, :4], out1[0, :4])
    assert not np.array_equal(out0[0, 4:], out1[0, 4:])
