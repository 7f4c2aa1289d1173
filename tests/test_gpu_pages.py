"""DiffKV tiers in page pools on the GPU (the DiffKV memory manager): the same cache
life cycle with and without pages gives bit-identical outputs and tier contents; the
prefill-end allocation equals the oracle pool's exactly; appends that open pages, releases
and rebuilds keep the pool's invariants; an exhausted pool is reported, not overrun."""
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import pages as OPG
from oracle import policies as OP
from tests.helpers import assert_attn_close, np_

pytestmark = pytest.mark.gpu

G, W, P = 32, 64, kvq.PAGE_TOKENS


def _logical_rows(tier, u):
    """Unit u's stored rows of a tier (paged or not) as uint32 / uint16 numpy arrays."""
    rows = tier.rows_of(u).cuda()
    flat = lambda x: x.reshape(-1, *x.shape[2:])
    pick = lambda x: flat(x).index_select(0, rows).cpu().numpy()
    return [pick(x) for x in (tier.k_codes, tier.k_scale, tier.k_zero, tier.v_codes, tier.v_scale, tier.v_zero,
                              tier.token_id)]


def _pool_invariants(tier, units):
    n, mp = tier.n_pages, tier.max_pages
    pt = tier.page_table.cpu().numpy()
    owner = tier.page_owner.cpu().numpy()
    ring = tier.free_ring.cpu().numpy()
    head, tail = (int(x) for x in tier.ring_ctr.cpu().numpy().astype(np.uint32))
    cnt = tier.count.cpu().numpy()
    owned = [pg for pg in range(n) if owner[pg] >= 0]
    free = [int(ring[k % n]) for k in range(head, tail)]
    assert sorted(owned + free) == list(range(n)), "every page free once or owned once"
    for u in range(units):
        k = int((pt[u] >= 0).sum())
        assert (pt[u, :k] >= 0).all() and (pt[u, k:] < 0).all(), "pages are a prefix of the row"
        assert k == (cnt[u] + P - 1) // P, f"unit {u}: {k} pages for {cnt[u]} tokens"
        for i in range(k):
            assert owner[pt[u, i]] == u * mp + i, "reverse table"
    return head, tail


def _setup(B, Hq, Hkv, T, D, n_high, n_low, steps, pages, seed):
    x = inputs.make_qkv(B, Hq, Hkv, T + steps, D, seed=seed)
    cs = inputs.random_scores(B, Hq, T, seed=seed) + 0.01
    caps = [int(max(n_high)) + steps + 1, int(max(n_low)) + steps + 1]

    def make(paged):
        c = kvq.make_cache(B, Hq, Hkv, D, G, torch.float16, kvq.POLICY_DIFFKV,
                           [kvq.TierSpec(8, 4, kvq.AXIS_TOKEN, caps[0]), kvq.TierSpec(4, 2, kvq.AXIS_TOKEN, caps[1])],
                           nr=W, pages=pages if paged else None)
        if paged:
            kvq.pages_init(c)
        return c
    return x, cs, make


def _build(c, x, cs, T, n_high, n_low):
    kvq.requant_demote(c, 0, k_src=x.k[:, :, :T].contiguous().cuda(), v_src=x.v[:, :, :T].contiguous().cuda(),
                       colscore=cs.cuda(), n_high=torch.tensor(n_high, dtype=torch.int32, device="cuda"),
                       n_low=torch.tensor(n_low, dtype=torch.int32, device="cuda"))


def test_paged_equals_unpaged_and_oracle_pool():
    """Budgets right below page boundaries, so that window exits open pages during decode."""
    B, Hq, Hkv, T, D, steps = 2, 10, 2, 640, 128, 24
    g = Hq // Hkv
    n_high, n_low = [127, 0, 128, 60], [254, 128, 1, 300]
    pages = [8, 12]
    x, cs, make = _setup(B, Hq, Hkv, T, D, n_high, n_low, steps, pages, seed=51)
    plain, paged = make(False), make(True)
    _build(plain, x, cs, T, n_high, n_low)
    _build(paged, x, cs, T, n_high, n_low)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    # the prefill-end allocation is the oracle pool's, page for page
    for ti, (tier, n_tok) in enumerate(zip(paged.tiers, (n_high, n_low))):
        pool = OPG.PagePool(tier.n_pages, B * Hkv, tier.max_pages)
        pool.build(n_tok)
        assert np.array_equal(tier.page_table.cpu().numpy(), np.array(pool.pt)), f"tier {ti} page table"
        assert np.array_equal(tier.page_owner.cpu().numpy(), np.array(pool.owner)), f"tier {ti} owners"
        assert list(tier.ring_ctr.cpu().numpy()) == [pool.head, pool.tail]
        _pool_invariants(tier, B * Hkv)
    units = [OP.DiffKVUnit(np_(x.k[u // Hkv, u % Hkv, :T]), np_(x.v[u // Hkv, u % Hkv, :T]),
                           np_(cs[u // Hkv, (u % Hkv) * g:(u % Hkv + 1) * g]), n_high[u], n_low[u], W, G)
             for u in range(B * Hkv)]
    scale = 1.0 / math.sqrt(D)
    opened = 0
    for t in range(steps):
        qd = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(900 + t)).half().cuda()
        kd, vd = x.k[:, :, T + t].contiguous().cuda(), x.v[:, :, T + t].contiguous().cuda()
        before = [int(tr.ring_ctr[0].item()) for tr in paged.tiers]
        o1, l1 = kvq.decode_attn_qkv(qd, kd, vd, plain, scale)
        o2, l2 = kvq.decode_attn_qkv(qd, kd, vd, paged, scale)
        kvq.requant_demote(plain, t + 1)
        kvq.requant_demote(paged, t + 1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2), f"step {t}: paged output differs"
        opened += sum(int(tr.ring_ctr[0].item()) - b for tr, b in zip(paged.tiers, before))
        for u in range(B * Hkv):
            ro, _, _ = units[u].step(T + t, np_(qd[u // Hkv, (u % Hkv) * g:(u % Hkv + 1) * g].float()),
                                     np_(kd[u // Hkv, u % Hkv]), np_(vd[u // Hkv, u % Hkv]), scale)
            assert_attn_close(o2[u // Hkv, (u % Hkv) * g:(u % Hkv + 1) * g], ro, f"step {t} unit {u}")
    assert kvq.device_status() == 0
    assert opened > 0, "no decode step opened a page"
    for ti in range(2):
        assert torch.equal(plain.tiers[ti].count, paged.tiers[ti].count)
        _pool_invariants(paged.tiers[ti], B * Hkv)
        for u in range(B * Hkv):
            for a_, b_ in zip(_logical_rows(plain.tiers[ti], u), _logical_rows(paged.tiers[ti], u)):
                assert np.array_equal(a_, b_), f"tier {ti} unit {u} contents"


def test_release_compaction_and_rebuild():
    B, Hq, Hkv, T, D, steps = 1, 8, 4, 512, 128, 4
    n_high, n_low = [200, 50, 300, 129], [100, 250, 0, 128]
    pages = [9, 8]
    x, cs, make = _setup(B, Hq, Hkv, T, D, n_high, n_low, steps, pages, seed=53)
    c = make(True)
    _build(c, x, cs, T, n_high, n_low)
    torch.cuda.synchronize()
    before = [t.page_table.cpu().numpy().copy() for t in c.tiers]
    tails = [int(t.ring_ctr[1].item()) for t in c.tiers]
    mask = torch.tensor([0, 1, 1, 0], dtype=torch.int32, device="cuda")
    kvq.pages_release(c, mask)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    for ti, t in enumerate(c.tiers):
        ring = t.free_ring.cpu().numpy()
        held = [(before[ti][u] >= 0).sum() if mask[u] else 0 for u in range(4)]
        base = np.concatenate([[0], np.cumsum(held)[:-1]])
        for u in (1, 2):
            for i in range(held[u]):
                assert ring[(tails[ti] + base[u] + i) % t.n_pages] == before[ti][u, i], f"tier {ti} unit {u}"
        assert int(t.ring_ctr[1].item()) == tails[ti] + sum(held)
        assert int(t.count[1]) == 0 and int(t.count[2]) == 0
        _pool_invariants(t, 4)
    assert int(c.res_len[1]) == 0 and int(c.seq_len[2]) == 0
    # a rebuild takes every page back first: same contents as a fresh cache
    _build(c, x, cs, T, n_high, n_low)
    fresh = make(True)
    _build(fresh, x, cs, T, n_high, n_low)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    for ti in range(2):
        _pool_invariants(c.tiers[ti], 4)
        for u in range(4):
            for a_, b_ in zip(_logical_rows(c.tiers[ti], u), _logical_rows(fresh.tiers[ti], u)):
                assert np.array_equal(a_, b_)


def test_exhausted_pool_is_reported():
    """A pool too small for the build: the status word says so, no page is handed out and
    no token is written outside the pool."""
    B, Hq, Hkv, T, D = 1, 4, 2, 512, 128
    n_high, n_low = [300, 300], [10, 10]
    x, cs, make = _setup(B, Hq, Hkv, T, D, n_high, n_low, 0, [4, 2], seed=55)
    c = make(True)
    _build(c, x, cs, T, n_high, n_low)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_EDEVICE
    t0 = c.tiers[0]
    assert int(t0.ring_ctr[0].item()) == 0 and (t0.page_table.cpu().numpy() < 0).all()
    assert int(t0.count[0]) == 0 and int(t0.count[1]) == 0
    _pool_invariants(t0, 2)
