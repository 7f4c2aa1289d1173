"""DiffKV tiers on the GPU: prefill-end split, window exits (K8V4 / K4V2 / pruned),
decode attention with GQA over both tiers and the window."""
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

G, W = 32, 64


def _make(B, Hq, Hkv, T, D, steps, n_high, n_low):
    caps = [int(max(n_high)) + steps + 1, int(max(n_low)) + steps + 1]
    return kvq.make_cache(B, Hq, Hkv, D, G, torch.float16, kvq.POLICY_DIFFKV,
                          [kvq.TierSpec(8, 4, kvq.AXIS_TOKEN, caps[0]),
                           kvq.TierSpec(4, 2, kvq.AXIS_TOKEN, caps[1])], nr=W)


def _counts(B, Hkv, T, seed):
    f = inputs.dirichlet_fractions(B * Hkv, seed=seed)
    nc = T - W
    n_high = np.floor(f[:, 0] * nc).astype(np.int32)
    n_low = np.floor(f[:, 1] * nc).astype(np.int32)
    return n_high, n_low


def test_diffkv_decisions_bit_exact():
    """Identical float32 scores on both sides: the split, the thresholds, the codes of every
    stored token and each window-exit decision are identical."""
    B, Hq, Hkv, T, D, steps = 2, 10, 2, 640, 128, 12
    g = Hq // Hkv
    x = inputs.make_qkv(B, Hq, Hkv, T + steps, D, seed=4)
    cs = inputs.random_scores(B, Hq, T, seed=4, ties=64) + 0.01
    n_high, n_low = _counts(B, Hkv, T, 4)
    cache = _make(B, Hq, Hkv, T, D, steps, n_high, n_low)
    k, v = x.k[:, :, :T].contiguous().cuda(), x.v[:, :, :T].contiguous().cuda()
    kvq.requant_demote(cache, 0, k_src=k, v_src=v, colscore=cs.cuda(),
                       n_high=torch.from_numpy(n_high).cuda(), n_low=torch.from_numpy(n_low).cuda())
    units = []
    for u in range(B * Hkv):
        b, h = u // Hkv, u % Hkv
        un = OP.DiffKVUnit(np_(x.k[b, h, :T]), np_(x.v[b, h, :T]), np_(cs[b, h * g:(h + 1) * g]),
                           int(n_high[u]), int(n_low[u]), W, G)
        units.append(un)
        assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(un.high), "high")
        assert_tiers_equal(gpu_tier_rows(cache.tiers[1], u), oracle_tier_rows(un.low), "low")
        al = cache.alpha[u].cpu().numpy()
        assert al[0] == un.alpha_h and al[1] == un.alpha_l
    r = np.random.default_rng(0)
    scale = 1.0 / math.sqrt(D)
    seen = set()
    for t in range(steps):
        qd = (torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(t)) * 0.5).half()
        kd, vd = x.k[:, :, T + t].contiguous(), x.v[:, :, T + t].contiguous()
        od, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), cache, scale)
        N = T + t + 1
        start = cache.res_start.cpu().numpy()
        for u in range(B * Hkv):
            b, h = u // Hkv, u % Hkv
            ro, _ = units[u].attend(T + t, np_(qd[b, h * g:(h + 1) * g]), np_(kd[b, h]),
                                    np_(vd[b, h]), scale)
            assert_attn_close(od[b, h * g:(h + 1) * g], ro, f"step {t} unit {u}")
            tc = units[u].win[0][0]
            th = float(units[u].alpha_h) / N
            level = r.random() * 1.3 * th * (N - tc)     # spans prune / low / high
            vals = (level * (0.5 + 0.5 * r.random(g))).astype(np.float32)
            units[u].win[0][3][:] = vals
            cache.win_acc[b * Hq + h * g:b * Hq + (h + 1) * g, start[u]] = torch.from_numpy(vals).cuda()
        kvq.requant_demote(cache, t + 1)
        for u in range(B * Hkv):
            dec = units[u].tail(N)
            seen.add(dec[1])
            assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(units[u].high), "high")
            assert_tiers_equal(gpu_tier_rows(cache.tiers[1], u), oracle_tier_rows(units[u].low), "low")
    assert kvq.device_status() == 0
    assert seen == {"high", "low", "pruned"}


def test_diffkv_pipeline():
    """GQA 10/2, prompt 1024, Dirichlet(2,5,3) fractions per (batch, KV head), 64-token
    window, 40 decode steps; the GPU's own column scores drive its decisions."""
    B, Hq, Hkv, T, D, steps = 2, 10, 2, 1024, 128, 40
    g = Hq // Hkv
    x = inputs.make_qkv(B, Hq, Hkv, T, D, seed=7)
    scale = 1.0 / math.sqrt(D)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    _, _, cs = kvq.prefill_attn_scores(q, k, v, scale)
    n_high, n_low = _counts(B, Hkv, T, 7)
    cache = _make(B, Hq, Hkv, T, D, steps, n_high, n_low)
    kvq.requant_demote(cache, 0, k_src=k, v_src=v, colscore=cs,
                       n_high=torch.from_numpy(n_high).cuda(), n_low=torch.from_numpy(n_low).cuda())
    units, agree = [], []
    for u in range(B * Hkv):
        b, h = u // Hkv, u % Hkv
        ref_cs = np.stack([OA.prefill_head(np_(x.q[b, hq]), np_(x.k[b, h]), np_(x.v[b, h]), scale)[2]
                           for hq in range(h * g, (h + 1) * g)]).astype(np.float32)
        un = OP.DiffKVUnit(np_(x.k[b, h]), np_(x.v[b, h]), ref_cs, int(n_high[u]), int(n_low[u]), W, G)
        units.append(un)
        same = (sorted(gpu_tier_rows(cache.tiers[0], u)) == un.high.ids() and
                sorted(gpu_tier_rows(cache.tiers[1], u)) == un.low.ids())
        if not same:
            # only a boundary token may differ, by score rounding
            sig = OP.diffkv_significance(ref_cs, T)
            diff = set(gpu_tier_rows(cache.tiers[0], u)) ^ set(un.high.ids())
            diff |= set(gpu_tier_rows(cache.tiers[1], u)) ^ set(un.low.ids())
            bounds = [float(un.alpha_h) / T, float(un.alpha_l) / T]
            for j in diff:
                assert min(abs(sig[j] - bb) for bb in bounds) <= 1e-4 * max(bounds), j
        agree.append(same)
    assert sum(agree) >= len(agree) - 1
    for t in range(steps):
        qd, kd, vd = inputs.make_decode_step(B, Hq, Hkv, D, t, seed=7)
        od, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), cache, scale)
        kvq.requant_demote(cache, t + 1)
        for u in range(B * Hkv):
            if not agree[u]:
                continue
            b, h = u // Hkv, u % Hkv
            ro, _, dec = units[u].step(T + t, np_(qd[b, h * g:(h + 1) * g]), np_(kd[b, h]),
                                       np_(vd[b, h]), scale)
            assert_attn_close(od[b, h * g:(h + 1) * g], ro, f"step {t} unit {u}")
            in_hi = dec[0] in gpu_tier_rows(cache.tiers[0], u)
            in_lo = dec[0] in gpu_tier_rows(cache.tiers[1], u)
            got = "high" if in_hi else ("low" if in_lo else "pruned")
            if got != dec[1]:
                agree[u] = False            # a decision on the threshold edge; stop comparing
    assert kvq.device_status() == 0
    assert sum(agree) >= len(agree) - 1
    for u in range(B * Hkv):
        if agree[u]:
            assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(units[u].high))
            assert_tiers_equal(gpu_tier_rows(cache.tiers[1], u), oracle_tier_rows(units[u].low))


@pytest.mark.parametrize("Hq,Hkv", [(10, 2), (2, 2)])
def test_diffkv_k4v8_mirror(Hq, Hkv):
    """The K4V8 mirror of the high tier (a codec variant the DiffKV pages report as a
    negative result): build, window exits and decode against the oracle with the same
    formats, on the tensor-core path (GQA 5) and the single-head CUDA-core path."""
    B, T, D, steps = 2, 512, 128, 10
    g = Hq // Hkv
    x = inputs.make_qkv(B, Hq, Hkv, T + steps, D, seed=61)
    cs = inputs.random_scores(B, Hq, T, seed=61) + 0.01
    n_high, n_low = _counts(B, Hkv, T, 61)
    caps = [int(max(n_high)) + steps + 1, int(max(n_low)) + steps + 1]
    cache = kvq.make_cache(B, Hq, Hkv, D, G, torch.float16, kvq.POLICY_DIFFKV,
                           [kvq.TierSpec(4, 8, kvq.AXIS_TOKEN, caps[0]), kvq.TierSpec(4, 2, kvq.AXIS_TOKEN, caps[1])],
                           nr=W)
    kvq.requant_demote(cache, 0, k_src=x.k[:, :, :T].contiguous().cuda(), v_src=x.v[:, :, :T].contiguous().cuda(),
                       colscore=cs.cuda(), n_high=torch.from_numpy(n_high).cuda(), n_low=torch.from_numpy(n_low).cuda())
    units = [OP.DiffKVUnit(np_(x.k[u // Hkv, u % Hkv, :T]), np_(x.v[u // Hkv, u % Hkv, :T]),
                           np_(cs[u // Hkv, (u % Hkv) * g:(u % Hkv + 1) * g]), int(n_high[u]), int(n_low[u]), W, G,
                           high_bits=(4, 8)) for u in range(B * Hkv)]
    for u in range(B * Hkv):
        assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(units[u].high), f"K4V8 u{u}")
    scale = 1.0 / math.sqrt(D)
    for t in range(steps):
        qd = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(300 + t)).half()
        kd, vd = x.k[:, :, T + t].contiguous(), x.v[:, :, T + t].contiguous()
        od, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), cache, scale)
        kvq.requant_demote(cache, t + 1)
        for u in range(B * Hkv):
            ro, _, _ = units[u].step(T + t, np_(qd[u // Hkv, (u % Hkv) * g:(u % Hkv + 1) * g]),
                                     np_(kd[u // Hkv, u % Hkv]), np_(vd[u // Hkv, u % Hkv]), scale)
            assert_attn_close(od[u // Hkv, (u % Hkv) * g:(u % Hkv + 1) * g], ro, f"step {t} unit {u}")
    assert kvq.device_status() == 0
    for u in range(B * Hkv):
        assert_tiers_equal(gpu_tier_rows(cache.tiers[0], u), oracle_tier_rows(units[u].high), f"K4V8 u{u}")
        assert_tiers_equal(gpu_tier_rows(cache.tiers[1], u), oracle_tier_rows(units[u].low), f"K4V2 u{u}")
