"""Pins of the oracle's page-tag bump and batched validation.

The pages (Cloudflare write-up, Italian edition, sections "Cosa ha cambiato
Cloudflare per Kimi e GLM" and "La sicurezza della cache KV condivisa diventa
una questione di produzione"; the iitog.ru summary's third technique) state:
a tag per physical page changes on every reallocation, the server records the
(page, tag) pairs each request expects, the mapping is checked before the
pages are read, and a mismatch aborts that request instead of returning
another request's data.  These tests pin the oracle to that by brute force:
every single corruption of a small table must abort exactly its request.
"""
import itertools

import numpy as np
import pytest

import oracle
from workloads import rng_for


def _table(seed, B, ps, lens, num_pages, max_pages):
    g = rng_for(seed, "t")
    perm = g.permutation(num_pages).astype(np.int32)
    pt = np.full((B, max_pages), -1, np.int32)
    o = 0
    for r in range(B):
        P = -(-lens[r] // ps)
        pt[r, :P] = perm[o:o + P]
        o += P
    live = g.integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    exp = np.zeros((B, max_pages), np.uint32)
    m = pt >= 0
    exp[m] = live[pt[m]]
    return pt, exp, live


@pytest.mark.parametrize("ps", [4, 16])
def test_all_valid_is_empty(ps):
    lens = np.array([0, 1, ps, ps + 1, 3 * ps], np.int32)
    pt, exp, live = _table(1, 5, ps, lens, 64, 4)
    mask, n = oracle.page_tags_validate(pt, exp, lens, live, 64, ps)
    assert n == 0 and not mask.any()


@pytest.mark.parametrize("ps", [4, 16])
def test_every_single_corruption_aborts_exactly_its_request(ps):
    lens = np.array([5, 17, 1, 12], np.int32) if ps == 4 else np.array([40, 17, 1, 33], np.int32)
    B, num_pages, max_pages = len(lens), 40, 6
    pt, exp, live = _table(2, B, ps, lens, num_pages, max_pages)
    for r in range(B):
        P = -(-int(lens[r]) // ps)
        for i in range(max_pages):
            for kind in ("tag-1", "tag+big", "page=-1", "page=num_pages", "page=other"):
                pt2, exp2 = pt.copy(), exp.copy()
                if kind == "tag-1":
                    exp2[r, i] -= np.uint32(1)
                elif kind == "tag+big":
                    exp2[r, i] ^= np.uint32(0x80000000)
                elif kind == "page=-1":
                    pt2[r, i] = -1
                elif kind == "page=num_pages":
                    pt2[r, i] = num_pages
                else:
                    # another physical page whose live tag differs from the expected one
                    cand = [p for p in range(num_pages) if live[p] != exp[r, i]]
                    pt2[r, i] = cand[(r * 7 + i) % len(cand)]
                mask, n = oracle.page_tags_validate(pt2, exp2, lens, live, num_pages, ps)
                want = np.zeros(B, np.uint8)
                if i < P:
                    want[r] = 1
                assert np.array_equal(mask, want), (r, i, kind)
                assert n == int(want.sum())


def test_reallocation_bump_aborts_every_holder():
    ps, num_pages = 16, 32
    lens = np.array([30, 50, 16], np.int32)
    pt, exp, live = _table(3, 3, ps, lens, num_pages, 4)
    # request 1 and 2 share a page (prefix sharing): same page, same tag
    pt[2, 0] = pt[1, 0]
    exp[2, 0] = exp[1, 0]
    mask, _ = oracle.page_tags_validate(pt, exp, lens, live, num_pages, ps)
    assert not mask.any()
    live2 = live.copy()
    oracle.page_tags_bump(live2, np.array([pt[1, 0]], np.int32), num_pages)
    mask, n = oracle.page_tags_validate(pt, exp, lens, live2, num_pages, ps)
    assert list(mask) == [0, 1, 1] and n == 2


def test_bump_semantics():
    live = np.array([0, 5, 0xFFFFFFFF, 9], np.uint32)
    oracle.page_tags_bump(live, np.array([1, 2, 3, 3, -1, 4, 100], np.int32), 4)
    assert list(live) == [0, 6, 0, 11]      # wrap mod 2^32, repeats count, out of range ignored


def test_bump_wraparound_identity_after_2_32():
    """ABA limit: 2^32 bumps return a tag to its value (documented reading)."""
    live = np.array([123], np.uint32)
    x = (int(live[0]) + 2**32) % 2**32
    assert x == 123


def test_overlong_context_aborts_and_empty_does_not():
    ps, num_pages = 16, 16
    lens = np.array([0, 4 * 16 + 1, 64], np.int32)     # request 1 needs 5 pages, table holds 4
    pt, exp, live = _table(4, 3, ps, np.array([0, 64, 64]), num_pages, 4)
    mask, n = oracle.page_tags_validate(pt, exp, lens, live, num_pages, ps)
    assert list(mask) == [0, 1, 0] and n == 1


def test_padding_beyond_context_is_not_checked():
    ps, num_pages = 16, 16
    lens = np.array([17], np.int32)
    pt, exp, live = _table(5, 1, ps, np.array([17]), num_pages, 4)
    pt[0, 2:] = -7
    exp[0, 2:] = 12345
    mask, n = oracle.page_tags_validate(pt, exp, lens, live, num_pages, ps)
    assert n == 0


def test_abort_set_matches_exhaustive_pairs():
    """Random multi-corruption tables: abort set == requests with any bad checked entry."""
    g = np.random.default_rng(11)
    for trial in range(50):
        B, ps, num_pages, max_pages = 6, 8, 48, 6
        lens = g.integers(0, max_pages * ps + 1, size=B).astype(np.int32)
        need = int((-(-lens // ps)).sum())
        if need > num_pages:
            continue
        pt, exp, live = _table(100 + trial, B, ps, lens, num_pages, max_pages)
        bad = set()
        for r, i in itertools.product(range(B), range(max_pages)):
            if g.random() < 0.05:
                exp[r, i] += np.uint32(1)
                if i < -(-int(lens[r]) // ps):
                    bad.add(r)
        mask, n = oracle.page_tags_validate(pt, exp, lens, live, num_pages, ps)
        assert set(np.flatnonzero(mask)) == bad and n == len(bad)
