"""Oracle: the DiffKV GPU memory manager as a plain sequential model.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: DiffKV verdict JSON (arXiv 2412.03131), ``pith_extraction.key_machinery``
and ``core_discovery``: a GPU-resident memory manager with unified pages, a
circular free page list and a bidirectional page table, which compacts free
pages in parallel so that per-head, per-request caches of different sizes share
one pool.

Readings (the pages name the parts, not their rules):
  * a page holds P = 128 token slots of one precision tier; each tier has one
    pool shared by every (batch, KV head) unit of the layer -- "unified": any
    page can serve any head of any request;
  * the free list is a ring of page ids with two monotone counters: pops take
    ring[head mod n] and advance head, pushes write ring[tail mod n] and advance
    tail; the free pages are ring[head .. tail);
  * the forward table maps (unit, logical page i) to a physical page, the
    reverse table maps a physical page back to unit * max_pages + i (-1 when
    free); a unit's pages are always logical pages 0 .. k-1 (tokens are only
    appended);
  * a build first returns every unit's pages (units in order, pages in logical
    order), then gives unit u its demand ceil(n_u / P) as one run of the ring
    taken in unit order: the run of unit u starts at head + sum_{v<u} d_v (an
    exclusive prefix sum of the demands -- the parallel form of the same
    sequential order);
  * a release returns the pages of the released units the same way, at the
    ring tail (exclusive prefix sum of the released counts: the compaction);
  * a decode step whose token opens logical page i of unit u pops one page.

Pins (tests/test_oracle_pages.py): page conservation (free + owned = n), no page
owned twice, forward and reverse tables inverse to each other, build and release
placements equal to numpy's cumulative sums of the demands, exhaustion detected,
and a long random mix of builds, appends and releases that keeps every invariant.
"""
from __future__ import annotations

P = 128


class PagePool:
    def __init__(self, n_pages, units, max_pages):
        self.n, self.units, self.max_pages = n_pages, units, max_pages
        self.ring = list(range(n_pages))
        self.head, self.tail = 0, n_pages
        self.pt = [[-1] * max_pages for _ in range(units)]
        self.owner = [-1] * n_pages

    # -- free ring
    def free_count(self):
        return self.tail - self.head

    def _pop(self):
        if self.free_count() <= 0:
            raise MemoryError("page pool exhausted")
        pg = self.ring[self.head % self.n]
        self.head += 1
        return pg

    def _push(self, pg):
        self.ring[self.tail % self.n] = pg
        self.tail += 1

    # -- table
    def held(self, u):
        k = 0
        while k < self.max_pages and self.pt[u][k] >= 0:
            k += 1
        return k

    def _give(self, u, i, pg):
        self.pt[u][i] = pg
        self.owner[pg] = u * self.max_pages + i

    def release(self, units):
        """Every page of the given units back to the ring tail, units in order, pages in order."""
        for u in sorted(set(units)):
            for i in range(self.held(u)):
                pg = self.pt[u][i]
                self._push(pg)
                self.owner[pg] = -1
                self.pt[u][i] = -1

    def build(self, tokens):
        """tokens[u] slots of the tier for unit u: old pages back, then ceil(n/P) pages each."""
        self.release(range(self.units))
        demand = [min((n + P - 1) // P, self.max_pages) for n in tokens]
        if sum(demand) > self.free_count():
            raise MemoryError("page pool exhausted")
        for u, d in enumerate(demand):
            for i in range(d):
                self._give(u, i, self._pop())

    def append_page(self, u):
        """The next logical page of unit u (a token opened it)."""
        i = self.held(u)
        if i >= self.max_pages:
            raise IndexError("unit at its page limit")
        pg = self._pop()
        self._give(u, i, pg)
        return pg

    def slot(self, u, s):
        """(physical page, row) of slot s of unit u."""
        pg = self.pt[u][s // P]
        if pg < 0:
            raise KeyError(f"slot {s} of unit {u} has no page")
        return pg, s % P
