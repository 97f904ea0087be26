"""Host-side page ledger: the server's record of pages, owners and expected tags.

The Cloudflare write-up ("Cosa ha cambiato Cloudflare per Kimi e GLM" and "La
sicurezza della cache KV condivisa diventa una questione di produzione",
remio.ai) has the serving system keep, for every request, the physical pages
it maps and the tag it expects on each; a page's tag changes whenever the
page is reallocated, so a mapping that outlived a reallocation no longer
matches.  The ledger is that bookkeeping for one layer's pool:

* a free list of physical pages and, per request, its page list;
* a mirror of the live tags (the device holds the real ones; every tag bump
  the ledger orders is applied on the device by ``fpk_page_tags_bump``);
* per request, the table row (page ids) and the expected tags.

Every allocation is a reallocation and bumps the page's tag; the pages
returned by ``allocate`` are the bump list for that step.  The ledger does no
GPU work itself and holds none of the kernels' arithmetic beyond the +1 it
must mirror to know the tag a fresh mapping should expect.
"""
from __future__ import annotations

from collections import deque

import numpy as np


class PageLedger:
    def __init__(self, num_pages: int, max_pages: int, B: int, page_size: int,
                 live_tags: np.ndarray, page_table: np.ndarray | None = None,
                 seq_lens: np.ndarray | None = None):
        self.num_pages = num_pages
        self.max_pages = max_pages
        self.B = B
        self.page_size = page_size
        self.tags = np.asarray(live_tags, np.uint32).copy()
        self.page_table = np.full((B, max_pages), -1, np.int32)
        self.expected = np.zeros((B, max_pages), np.uint32)
        self.lens = np.zeros(B, np.int32)
        self.owner = np.full(num_pages, -1, np.int64)
        if page_table is not None:
            self.page_table[:] = page_table
            m = page_table >= 0
            self.expected[m] = self.tags[page_table[m]]
            rows, _ = np.nonzero(m)
            self.owner[page_table[m]] = rows
            self.lens[:] = seq_lens
        self.free = deque(int(p) for p in np.flatnonzero(self.owner < 0))

    # ----------------------------------------------------------- allocation
    def pages_of(self, r: int) -> int:
        return -(-int(self.lens[r]) // self.page_size)

    def allocate(self, r: int, n: int) -> list[int]:
        """Give request r `n` more pages; each is reallocated (its tag bumped)."""
        have = self.pages_of_table(r)
        if have + n > self.max_pages:
            raise RuntimeError(f"request {r}: page table full")
        if n > len(self.free):
            raise RuntimeError("pool exhausted")
        got = [self.free.popleft() for _ in range(n)]
        for i, p in enumerate(got):
            self.tags[p] = self.tags[p] + np.uint32(1)
            self.owner[p] = r
            self.page_table[r, have + i] = p
            self.expected[r, have + i] = self.tags[p]
        return got

    def pages_of_table(self, r: int) -> int:
        row = self.page_table[r]
        return int(np.count_nonzero(row >= 0))

    def release(self, r: int) -> list[int]:
        """Request r finished (or was aborted): its pages return to the free list."""
        row = self.page_table[r]
        pages = [int(p) for p in row[row >= 0] if 0 <= p < self.num_pages and self.owner[p] == r]
        for p in pages:
            self.owner[p] = -1
            self.free.append(p)
        self.page_table[r] = -1
        self.expected[r] = 0
        self.lens[r] = 0
        return pages

    def admit(self, r: int, prompt_len: int) -> list[int]:
        """Slot r takes a new request with `prompt_len` tokens already computed."""
        assert self.pages_of_table(r) == 0, "slot still holds pages"
        self.lens[r] = prompt_len
        return self.allocate(r, -(-prompt_len // self.page_size))

    def grow(self, r: int) -> list[int]:
        """One decode token for request r; a page is reallocated when it crosses a boundary."""
        self.lens[r] += 1
        need = self.pages_of(r) - self.pages_of_table(r)
        return self.allocate(r, need) if need > 0 else []

    # ------------------------------------------------------ stale mappings
    def corrupt(self, r: int, rng: np.random.Generator) -> tuple[int, str]:
        """Make one of request r's checked entries stale, as a bookkeeping bug would:
        either the expected tag of its page lags one reallocation behind, or the
        entry points at a page that has been reallocated to another request and
        carries that page's previous tag.  Returns (entry, kind)."""
        P = self.pages_of(r)
        i = int(rng.integers(0, P))
        others = np.flatnonzero((self.owner >= 0) & (self.owner != r))
        if rng.random() < 0.5 or others.size == 0:
            self.expected[r, i] = self.expected[r, i] - np.uint32(1)
            return i, "lagging tag"
        p = int(others[rng.integers(0, others.size)])
        self.page_table[r, i] = p
        self.expected[r, i] = self.tags[p] - np.uint32(1)
        return i, "reallocated page"
