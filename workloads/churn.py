"""Churn + integrity workload: continuous batching with page reallocation and
injected stale lookups (shape of the integrity evaluation in the Cloudflare
write-up: 8192-token prompts, 1000 output tokens, a fixed concurrency).

256 request slots (Hq=32, Hkv=8, page_size 16), each starting with an
8192-token prompt.  Every decode step appends one token per request (a page is
reallocated each time a request crosses a page boundary).  Every 50 steps 10 %
of the requests finish; their slots take new 8192-token requests whose pages
are reallocated from the freed ones.  Each step, every request's lookup is
made stale with probability 1 % (one entry of its table: a tag that lags one
reallocation, or a page reallocated to another request); a request that
aborted is retired at the next step like a finished one.

The event stream is seeded; all randomness is drawn here.  The host
bookkeeping is fp8_paged_kv_gb300.ledger.PageLedger; the tag bumps it orders
are applied by each side (device kernel / oracle) to its own live tags.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from fp8_paged_kv_gb300.ledger import PageLedger
from workloads import rng_for


@dataclasses.dataclass
class StepEvents:
    step: int
    bump: np.ndarray          # int32 page ids reallocated this step (in order)
    admitted: list            # slots that took a new request this step
    corrupted: dict           # slot -> (entry, kind)
    lens: np.ndarray          # context lengths after this step's append


class ChurnScenario:
    def __init__(self, seed: int = 5, B: int = 256, Hq: int = 32, Hkv: int = 8, ps: int = 16,
                 prompt: int = 8192, steps: int = 1000, finish_every: int = 50,
                 finish_frac: float = 0.10, stale_prob: float = 0.01, pool_factor: float = 1.2):
        self.seed, self.B, self.Hq, self.Hkv, self.ps = seed, B, Hq, Hkv, ps
        self.D = 128
        self.prompt, self.steps = prompt, steps
        self.finish_every, self.finish_n = finish_every, int(round(finish_frac * B))
        self.stale_prob = stale_prob
        self.max_pages = -(-(prompt + steps) // ps)
        self.num_pages = int(math.ceil(pool_factor * B * self.max_pages))
        g = rng_for(seed, "churn-init")
        live = g.integers(0, 2**32, size=self.num_pages, dtype=np.uint64).astype(np.uint32)
        self.initial_tags = live.copy()
        # the initial batch: every slot holds a prompt on pages of a seeded permutation
        perm = g.permutation(self.num_pages).astype(np.int32)
        P0 = -(-prompt // ps)
        pt = np.full((B, self.max_pages), -1, np.int32)
        pt[:, :P0] = perm[:B * P0].reshape(B, P0)
        self.initial_table = pt.copy()
        self.ledger = PageLedger(self.num_pages, self.max_pages, B, ps, live, pt,
                                 np.full(B, prompt, np.int32))
        # free-list order: the rest of the permutation
        used = set(perm[:B * P0].tolist())
        self.ledger.free.clear()
        self.ledger.free.extend(int(p) for p in perm[B * P0:] if int(p) not in used)
        self.rng = rng_for(seed, "churn-events")
        self.aborted_prev: set = set()
        self.admissions = 0

    @property
    def sm_scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.D)))

    def next_step(self, step: int, aborted_last_step=()) -> StepEvents:
        """Host decisions for decode step `step` (0-based)."""
        L = self.ledger
        bump: list[int] = []
        admitted: list[int] = []
        retire = set(int(r) for r in aborted_last_step)
        if step > 0 and step % self.finish_every == 0:
            live = [r for r in range(self.B) if r not in retire]
            k = min(self.finish_n, len(live))
            retire |= set(int(r) for r in self.rng.choice(live, size=k, replace=False))
        for r in sorted(retire):
            L.release(r)
        for r in sorted(retire):
            bump += L.admit(r, self.prompt)
            admitted.append(r)
            self.admissions += 1
        for r in range(self.B):
            bump += L.grow(r)
        corrupted = {}
        hits = np.flatnonzero(self.rng.random(self.B) < self.stale_prob)
        for r in hits:
            corrupted[int(r)] = L.corrupt(int(r), self.rng)
        return StepEvents(step=step, bump=np.asarray(bump, np.int32), admitted=admitted,
                          corrupted=corrupted, lens=L.lens.copy())
