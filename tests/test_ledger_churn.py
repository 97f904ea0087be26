"""Host ledger and churn scenario (CPU): the server-side bookkeeping that feeds
the batched tag check, run against the oracle's bump and validation.

The pages' rule (Cloudflare write-up, "Cosa ha cambiato..." and "La sicurezza
della cache KV condivisa...", remio.ai): a page's tag changes on every
reallocation and a request whose recorded (page, tag) no longer matches must
abort.  Invariants checked: with no injected staleness nothing aborts; every
injected stale lookup aborts exactly its request; a mapping kept past its
page's reallocation aborts; the ledger's tag mirror equals the oracle's live
tags after every bump.
"""
import numpy as np

import oracle
from fp8_paged_kv_gb300.ledger import PageLedger
from workloads.churn import ChurnScenario


def test_allocation_bumps_and_records():
    live = np.arange(10, dtype=np.uint32) * 100
    led = PageLedger(10, 4, 2, 16, live)
    got = led.admit(0, 20)                      # 2 pages
    assert len(got) == 2
    for i, p in enumerate(got):
        assert led.tags[p] == live[p] + 1 and led.expected[0, i] == led.tags[p]
    assert led.grow(0) == [] and led.lens[0] == 21
    for _ in range(11):
        led.grow(0)
    assert led.lens[0] == 32 and led.pages_of_table(0) == 2
    assert len(led.grow(0)) == 1 and led.pages_of_table(0) == 3
    freed = led.release(0)
    assert len(freed) == 3 and set(freed) <= set(led.free)
    assert led.pages_of_table(0) == 0


def test_stale_mapping_after_reallocation_aborts():
    """A request whose table kept a page that was freed and reallocated aborts."""
    live = np.zeros(4, np.uint32)
    led = PageLedger(4, 4, 2, 16, live)        # a 4-page pool forces reuse
    led.admit(0, 32)
    stale_row, stale_exp = led.page_table[0].copy(), led.expected[0].copy()
    led.release(0)
    led.admit(1, 64)                            # takes (some of) the freed pages, bumped
    pt = np.stack([stale_row, led.page_table[1]])
    ex = np.stack([stale_exp, led.expected[1]])
    mask, n = oracle.page_tags_validate(pt, ex, np.array([32, 64], np.int32), led.tags, 4, 16)
    reused = set(stale_row[stale_row >= 0]) & set(led.page_table[1][led.page_table[1] >= 0])
    assert reused and list(mask) == [1, 0] and n == 1


def _run(sc: ChurnScenario, steps: int):
    live = sc.initial_tags.copy()
    aborted = ()
    n_corrupt = n_abort = 0
    for s in range(steps):
        ev = sc.next_step(s, aborted)
        oracle.page_tags_bump(live, ev.bump, sc.num_pages)
        assert np.array_equal(live, sc.ledger.tags), "tag mirror diverged"
        mask, n = oracle.page_tags_validate(sc.ledger.page_table, sc.ledger.expected, ev.lens, live,
                                            sc.num_pages, sc.ps)
        assert set(np.flatnonzero(mask)) == set(ev.corrupted), f"step {s}"
        aborted = tuple(np.flatnonzero(mask))
        n_corrupt += len(ev.corrupted)
        n_abort += n
    return n_corrupt, n_abort


def test_churn_scenario_small_abort_sets():
    sc = ChurnScenario(seed=9, B=24, prompt=64, steps=300, finish_every=20, stale_prob=0.02)
    n_corrupt, n_abort = _run(sc, 300)
    assert n_corrupt == n_abort and n_corrupt > 0 and sc.admissions > 0


def test_churn_scenario_no_injection_never_aborts():
    sc = ChurnScenario(seed=10, B=16, prompt=40, steps=200, finish_every=10, stale_prob=0.0)
    n_corrupt, n_abort = _run(sc, 200)
    assert n_corrupt == 0 and n_abort == 0


def test_churn_full_size_first_steps():
    """The full 256-request scenario's bookkeeping for its first 120 steps (two churn events)."""
    sc = ChurnScenario()
    assert sc.max_pages == 575 and sc.num_pages == int(np.ceil(1.2 * 256 * 575))
    n_corrupt, n_abort = _run(sc, 120)
    assert n_corrupt == n_abort
