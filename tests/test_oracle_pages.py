"""Pins of the page-manager oracle (oracle/pages.py) against properties the description
fixes: conservation, a bidirectional table, placement by prefix sums of the demands
(numpy's cumulative sum as the independent reference), exhaustion, and invariants over a
long random mix of operations."""
import numpy as np
import pytest

from oracle import pages as OPG


def _invariants(pool):
    owned = [pg for pg in range(pool.n) if pool.owner[pg] >= 0]
    free = [pool.ring[k % pool.n] for k in range(pool.head, pool.tail)]
    # every page is either free (once) or owned (once): conservation, no double use
    assert sorted(owned + free) == list(range(pool.n))
    assert pool.free_count() + len(owned) == pool.n
    # the reverse table inverts the forward one, and pages are a prefix of each row
    for u in range(pool.units):
        k = pool.held(u)
        assert all(pool.pt[u][i] < 0 for i in range(k, pool.max_pages))
        for i in range(k):
            assert pool.owner[pool.pt[u][i]] == u * pool.max_pages + i
    for pg in owned:
        u, i = divmod(pool.owner[pg], pool.max_pages)
        assert pool.pt[u][i] == pg


def test_build_places_runs_by_prefix_sum():
    pool = OPG.PagePool(64, 5, 8)
    tokens = [300, 0, 129, 1024, 1]
    pool.build(tokens)
    d = np.array([(n + 127) // 128 for n in tokens])
    start = np.concatenate([[0], np.cumsum(d)[:-1]])
    for u in range(5):
        assert pool.pt[u][:d[u]] == list(range(start[u], start[u] + d[u]))
    assert pool.head == d.sum() and pool.tail == 64
    _invariants(pool)


def test_release_compacts_at_the_tail_in_unit_order():
    pool = OPG.PagePool(40, 4, 8)
    pool.build([256, 128, 384, 100])                  # pages 0-1 | 2 | 3-5 | 6
    before = [list(row) for row in pool.pt]
    pool.release([2, 0])
    # released counts per unit (0 for the kept ones) -> each unit's run starts at the tail
    # plus the exclusive prefix sum of those counts
    rel_held = np.array([2, 0, 3, 0])
    base = np.concatenate([[0], np.cumsum(rel_held)[:-1]])
    tail0 = 40
    for u in (0, 2):
        for i in range(rel_held[u]):
            assert pool.ring[(tail0 + base[u] + i) % 40] == before[u][i]
    assert pool.tail == tail0 + rel_held.sum()
    assert pool.pt[0][0] == -1 and pool.pt[2][0] == -1 and pool.pt[1][0] == 2
    _invariants(pool)
    # a rebuild returns the rest, then hands out pages from the head again
    pool.build([128, 128, 128, 128])
    _invariants(pool)
    assert pool.free_count() == 36


def test_exhaustion_is_detected():
    pool = OPG.PagePool(4, 2, 8)
    with pytest.raises(MemoryError):
        pool.build([300, 300])                        # 3 + 3 pages > 4
    pool = OPG.PagePool(4, 2, 8)
    pool.build([256, 256])
    with pytest.raises(MemoryError):
        pool.append_page(0)


def test_random_operations_keep_every_invariant():
    r = np.random.default_rng(7)
    pool = OPG.PagePool(96, 6, 12)
    counts = [0] * 6
    for op in range(600):
        kind = r.integers(0, 10)
        if kind == 0:
            counts = [int(x) for x in r.integers(0, 700, size=6)]
            if sum((c + 127) // 128 for c in counts) <= 96:
                pool.build(counts)
            else:
                counts = [pool.held(u) * 128 for u in range(6)]
        elif kind == 1:
            rel = [u for u in range(6) if r.random() < 0.3]
            pool.release(rel)
            for u in rel:
                counts[u] = 0
        else:
            u = int(r.integers(0, 6))
            if counts[u] % 128 == 0:
                if pool.free_count() == 0 or pool.held(u) >= 12 or pool.held(u) * 128 > counts[u]:
                    continue
                pool.append_page(u)
            counts[u] += 1
            pg, row = pool.slot(u, counts[u] - 1)
            assert pool.owner[pg] == u * 12 + (counts[u] - 1) // 128 and row == (counts[u] - 1) % 128
        _invariants(pool)
