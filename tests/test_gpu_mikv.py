"""MiKV tiers on the GPU: INT4 top share by cumulative attention, INT2 rest, no eviction,
INT4 -> INT2 re-quantisation as ranks drop; bf16 activations."""
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import attention as OA
from oracle import policies as OP
from tests.helpers import (assert_attn_close, assert_tiers_equal, gpu_tier_rows, np_,
                           oracle_tier_rows)

pytestmark = pytest.mark.gpu

G = 32


def _make(B, Hq, Hkv, T, D, steps, nr, dtype=torch.bfloat16):
    n_q = T - nr + steps
    return kvq.make_cache(B, Hq, Hkv, D, G, dtype, kvq.POLICY_MIKV,
                          [kvq.TierSpec(4, 4, kvq.AXIS_TOKEN, n_q // 5 + 2),
                           kvq.TierSpec(2, 2, kvq.AXIS_TOKEN, n_q + 1)],
                          nr=nr, score_cap=T + steps + 1, hi_den=5)


def _check_units(cache, units):
    for u, un in enumerate(units):
        assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(un.hi), f"INT4 u{u}")
        assert_tiers_equal(gpu_tier_rows(cache.tiers[1], u), oracle_tier_rows(un.lo), f"INT2 u{u}")


@pytest.mark.parametrize("T,flat", [(700, False), (700, True), (2600, True)])
def test_mikv_decisions_bit_exact(T, flat):
    """Identical float32 cumulative scores (with many ties) on both sides: the INT4/INT2
    split, every demotion and every re-quantised code are identical.  With `flat`, every
    third step gives all tokens the same score (the ranking is then by position alone); at
    2600 tokens that tie is wider than the step's band buffer, so those steps take the
    general selection."""
    B, Hq, Hkv, D, steps, nr = 2, 8, 2, 128, 10, 16
    g = Hq // Hkv
    x = inputs.make_qkv(B, Hq, Hkv, T + steps, D, dtype=torch.bfloat16, seed=11,
                        outliers=inputs.outlier_channels(Hkv, D, 1, 11), outlier_scale=12.0)
    cs = inputs.random_scores(B, Hq, T, seed=11, ties=16)
    cache = _make(B, Hq, Hkv, T, D, steps, nr)
    k, v = x.k[:, :, :T].contiguous().cuda(), x.v[:, :, :T].contiguous().cuda()
    kvq.requant_demote(cache, 0, k_src=k, v_src=v, colscore=cs.cuda())
    units = []
    for u in range(B * Hkv):
        b, h = u // Hkv, u % Hkv
        units.append(OP.MiKVUnit(np_(x.k[b, h, :T]), np_(x.v[b, h, :T]),
                                 np_(cs[b, h * g:(h + 1) * g]), nr, G))
    _check_units(cache, units)
    assert np.array_equal(cache.cum_score[:, :T].cpu().numpy(),
                          np.stack([[un.cs[j] for j in range(T)] for un in units]))
    scale = 1.0 / math.sqrt(D)
    r = np.random.default_rng(3)
    n_dem = 0
    for t in range(steps):
        qd = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(100 + t)).bfloat16()
        kd, vd = x.k[:, :, T + t].contiguous(), x.v[:, :, T + t].contiguous()
        od, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), cache, scale)
        for u in range(B * Hkv):
            b, h = u // Hkv, u % Hkv
            ro, _ = units[u].attend(T + t, np_(qd[b, h * g:(h + 1) * g]), np_(kd[b, h]),
                                    np_(vd[b, h]), scale)
            assert_attn_close(od[b, h * g:(h + 1) * g], ro, f"step {t} unit {u}")
            # replace every cumulative score by the same synthetic values on both sides,
            # coarse enough to tie often
            vals = (np.floor(r.random(T + t + 1) * 24) / 8).astype(np.float32)
            if flat and t % 3 == 2:
                vals[:] = 1.5
            for j in range(T + t + 1):
                units[u].cs[j] = vals[j]
            cache.cum_score[u, :T + t + 1] = torch.from_numpy(vals).cuda()
        kvq.requant_demote(cache, t + 1)
        for un in units:
            _, dem = un.tail()
            n_dem += len(dem)
        _check_units(cache, units)
    assert kvq.device_status() == 0
    assert n_dem > 0


def test_mikv_pipeline():
    """GQA 8/2, bf16, 1% outlier key channel x12, prompt 1024, nr = 128, 30 steps; the GPU's
    own column scores and decode attention drive its ranking."""
    B, Hq, Hkv, T, D, steps, nr = 2, 8, 2, 1024, 128, 30, 128
    g = Hq // Hkv
    outl = inputs.outlier_channels(Hkv, D, 1, 5)
    x = inputs.make_qkv(B, Hq, Hkv, T, D, dtype=torch.bfloat16, seed=5, outliers=outl,
                        outlier_scale=12.0)
    scale = 1.0 / math.sqrt(D)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    _, _, cs = kvq.prefill_attn_scores(q, k, v, scale)
    cache = _make(B, Hq, Hkv, T, D, steps, nr)
    kvq.requant_demote(cache, 0, k_src=k, v_src=v, colscore=cs)
    units, agree = [], []
    for u in range(B * Hkv):
        b, h = u // Hkv, u % Hkv
        ref_cs = np.stack([OA.prefill_head(np_(x.q[b, hq]), np_(x.k[b, h]), np_(x.v[b, h]), scale)[2]
                           for hq in range(h * g, (h + 1) * g)]).astype(np.float32)
        un = OP.MiKVUnit(np_(x.k[b, h]), np_(x.v[b, h]), ref_cs, nr, G)
        units.append(un)
        agree.append(sorted(gpu_tier_rows(cache.tiers[0], u)) == un.hi.ids())
    assert sum(agree) >= len(agree) - 1
    for t in range(steps):
        qd, kd, vd = inputs.make_decode_step(B, Hq, Hkv, D, t, dtype=torch.bfloat16, seed=5,
                                             outliers=outl, outlier_scale=12.0)
        od, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), cache, scale)
        kvq.requant_demote(cache, t + 1)
        cum = cache.cum_score.cpu().numpy()
        for u in range(B * Hkv):
            if not agree[u]:
                continue
            b, h = u // Hkv, u % Hkv
            ro, _, _, _ = units[u].step(T + t, np_(qd[b, h * g:(h + 1) * g]), np_(kd[b, h]),
                                        np_(vd[b, h]), scale)
            assert_attn_close(od[b, h * g:(h + 1) * g], ro, f"step {t} unit {u}")
            ref = np.array([units[u].cs[j] for j in range(T + t + 1)])
            err = np.abs(cum[u, :T + t + 1] - ref)
            assert np.all(err <= 1e-4 * np.abs(ref) + 1e-6), "cumulative scores"
            if sorted(gpu_tier_rows(cache.tiers[0], u)) != units[u].hi.ids():
                agree[u] = False            # a rank flip within score rounding; stop comparing
        # nothing is ever evicted
        tot = (cache.tiers[0].count + cache.tiers[1].count + cache.res_len).cpu().numpy()
        assert np.all(tot == T + t + 1)
    assert kvq.device_status() == 0
    assert sum(agree) >= len(agree) - 1
    for u in range(B * Hkv):
        if agree[u]:
            assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(units[u].hi))
            assert_tiers_equal(gpu_tier_rows(cache.tiers[1], u), oracle_tier_rows(units[u].lo))
