"""Parity at the full sizes the benchmark times, in its launch configuration.

Workloads and cache capacities come from bench.py (pyramid layer 16, DiffKV
GQA 40/8, MiKV GQA 32/8 at 32k context).  At these sizes the oracle checks
what it can compute one piece at a time:

* prefill: sampled query rows of sampled heads (O and lse against float64),
  sampled columns of the column scores element by element (first, middle and
  last columns of one head, from the oracle's lse of every row), and two
  properties that hold at any size (each head's scores sum to the number of
  queries; the last column equals the last query's own attention weight);
* cache build and decode: the build runs from seeded float32 importance
  scores given to both sides (so every selection and tier decision is
  comparable bit for bit), then a few decode steps; sampled units are
  replayed by the oracle: outputs within the attention tolerance, tier
  contents bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import bench
from bit_mixed_precision_gb300 import inputs, kvq
from oracle import attention as OA
from oracle import policies as OP
from oracle import select as OS
from tests.helpers import (assert_attn_close, assert_scores_close, assert_tiers_equal, gpu_tier_rows,
                           np_, oracle_tier_rows, u16, u32)

pytestmark = pytest.mark.gpu

G = 32


def _hot(name, steps, **over):
    wl = dict(bench.WORKLOADS[name])
    wl["steps"] = steps
    wl.update(over)
    return wl, bench.Hot(wl, torch.device("cuda", 0), seed=0)


def _check_prefill(hot, heads, rows):
    """Sampled rows of O / lse, and the column-score properties, of the full-size prefill."""
    wl = hot.wl
    g = wl["Hq"] // wl["Hkv"]
    T = wl["T"]
    kvq.prefill_attn_scores(hot.q, hot.k, hot.v, hot.scale, out=(hot.o_pre, hot.lse, hot.cs))
    torch.cuda.synchronize()
    for b, h in heads:
        q, k, v = np_(hot.q[b, h]), np_(hot.k[b, h // g]), np_(hot.v[b, h // g])
        ro, rl = OA.prefill_rows(q, k, v, rows, hot.scale)
        assert_attn_close(hot.o_pre[b, h, rows], ro, f"prefill O head {b},{h}")
        assert np.allclose(np_(hot.lse[b, h, rows]), rl, rtol=0, atol=1e-3), "prefill lse"
        cs = np_(hot.cs[b, h]).astype(np.float64)
        assert abs(cs.sum() - T) <= 1e-4 * T, "column scores must sum to the number of queries"
        _, rl_last = OA.prefill_rows(q, k, v, np.array([T - 1]), hot.scale)
        p_last = math.exp(float(q[T - 1].astype(np.float64) @ k[T - 1].astype(np.float64)) * hot.scale
                          - rl_last[0])
        assert abs(cs[T - 1] - p_last) <= 1e-4 * p_last + 1e-7, "last column score"
    # sampled columns of the first sampled head, element by element
    b, h = heads[0]
    q, k = np_(hot.q[b, h]), np_(hot.k[b, h // g])
    cols = np.array([0, 1, 2, 31, 127, 128, T // 3, T // 2, T // 2 + 1, T - 129, T - 2, T - 1])
    lse_ref = OA.lse_all_rows(q, k, hot.scale)
    ref = OA.colscore_cols(q, k, cols, lse_ref, hot.scale)
    assert_scores_close(hot.cs[b, h, cols], ref, f"column scores head {b},{h}")


def test_fullsize_pyramid_layer16():
    """MiniKV pyramid sweep, layer 16: batch 16, 32 heads, prompt 16384, INT2, nr = 0;
    20 decode steps (the first residual flush falls on step 16)."""
    steps = 20
    wl, hot = _hot("pyramid-layer16", 256)
    B, H, D, T = wl["B"], wl["Hq"], wl["D"], wl["T"]
    _check_prefill(hot, [(3, 7), (15, 31)], np.array([0, 1, 4095, 9000, T - 1]))
    # build from seeded scores given to both sides
    cs = inputs.random_scores(B, H, T, seed=2, ties=64)
    # the benchmark's prefill-end epilogue: selection and packing in one launch
    idx = torch.empty((B, H, hot.n_sel), dtype=torch.int32, device="cuda")
    kvq.minikv_prefill_build(hot.cache, hot.k, hot.v, cs.cuda(), hot.kh, hot.w, kmax=hot.k_hh, idx_out=idx)
    sample = [3 * H + 7, 15 * H + 31]
    units = {}
    gsel = idx.cpu().numpy().reshape(B * H, -1)
    for u in sample:
        b, h = u // H, u % H
        sel = OS.select_unit(np_(cs[b, h]), hot.k_hh, hot.w)
        assert np.array_equal(np.sort(gsel[u]), sel), f"selection of unit {u}"
        units[u] = OP.MiniKVUnit(np_(hot.k[b, h]), np_(hot.v[b, h]), sel, wl["nr"], G)
    for t in range(steps):
        qd, kd, vd = hot.dec[t]
        od, ld = kvq.decode_attn_qkv(qd, kd, vd, hot.cache, hot.scale)
        for u in sample:
            b, h = u // H, u % H
            ro, rl = units[u].step(T + t, np_(qd[b, h:h + 1]), np_(kd[b, h]), np_(vd[b, h]), hot.scale)
            assert_attn_close(od[b, h], ro[0], f"decode step {t} unit {u}")
            assert abs(float(ld[b, h]) - rl[0]) < 1e-3
    assert kvq.device_status() == 0
    t0 = hot.cache.tiers[0]
    for u in sample:
        npk = len(units[u].ids)
        assert int(t0.count[u]) == npk
        assert np.array_equal(t0.token_id[u, :npk].cpu().numpy(), np.array(units[u].ids))
        assert np.array_equal(u32(t0.k_codes[u, :npk // 16]), units[u].kw.view(np.uint32))
        assert np.array_equal(u16(t0.k_scale[u, :npk // G]), units[u].ksc.view(np.uint16))
        assert np.array_equal(u32(t0.v_codes[u, :npk]), units[u].vw.view(np.uint32))


@pytest.mark.parametrize("paged", [True, False])
def test_fullsize_diffkv(paged):
    """DiffKV: GQA 40/8, batch 32, prompt 8192, K8V4 / K4V2 / prune with per-head
    Dirichlet(2,5,3) fractions, 64-token window; 24 decode steps, one window exit each;
    the tiers in page pools (the benchmark's layout) and in fixed per-unit arrays."""
    steps = 24
    wl, hot = _hot("diffkv", 512, paged=paged)
    B, Hq, Hkv, D, T, W = wl["B"], wl["Hq"], wl["Hkv"], wl["D"], wl["T"], wl["nr"]
    g = Hq // Hkv
    _check_prefill(hot, [(0, 0), (31, 39)], np.array([0, 63, 5000, T - 1]))
    cs = inputs.random_scores(B, Hq, T, seed=4, ties=128)
    kvq.requant_demote(hot.cache, 0, k_src=hot.k, v_src=hot.v, colscore=cs.cuda(), n_high=hot.n_high,
                       n_low=hot.n_low)
    sample = [0, 5 * Hkv + 3, B * Hkv - 1]
    nh, nl = hot.n_high.cpu().numpy(), hot.n_low.cpu().numpy()
    units = {}
    for u in sample:
        b, h = u // Hkv, u % Hkv
        units[u] = OP.DiffKVUnit(np_(hot.k[b, h]), np_(hot.v[b, h]), np_(cs[b, h * g:(h + 1) * g]),
                                 int(nh[u]), int(nl[u]), W, G)
    for t in range(steps):
        qd, kd, vd = hot.dec[t]
        od, ld = kvq.decode_attn_qkv(qd, kd, vd, hot.cache, hot.scale)
        kvq.requant_demote(hot.cache, t + 1)
        for u in sample:
            b, h = u // Hkv, u % Hkv
            ro, rl, _ = units[u].step(T + t, np_(qd[b, h * g:(h + 1) * g]), np_(kd[b, h]), np_(vd[b, h]),
                                      hot.scale)
            assert_attn_close(od[b, h * g:(h + 1) * g], ro, f"decode step {t} unit {u}")
    assert kvq.device_status() == 0
    for u in sample:
        assert_tiers_equal(gpu_tier_rows(hot.cache.tiers[0], u), oracle_tier_rows(units[u].high), f"K8V4 u{u}")
        assert_tiers_equal(gpu_tier_rows(hot.cache.tiers[1], u), oracle_tier_rows(units[u].low), f"K4V2 u{u}")
    if paged:
        for tier in hot.cache.tiers:
            pt = tier.page_table.cpu().numpy()
            owner = tier.page_owner.cpu().numpy()
            cnt = tier.count.cpu().numpy()
            for u in range(B * Hkv):
                k = int((pt[u] >= 0).sum())
                assert k == (cnt[u] + kvq.PAGE_TOKENS - 1) // kvq.PAGE_TOKENS
                assert np.array_equal(owner[pt[u, :k]], u * tier.max_pages + np.arange(k))


def test_fullsize_mikv():
    """MiKV: GQA 32/8, batch 64, prompt 32768, bf16, INT4 top 20% / INT2 rest, 128-token
    residual; 40 decode steps (one residual exit and re-ranking each, with INT4 -> INT2
    demotions along the way).  After each step's attention the cumulative scores are
    compared, then both sides continue from the oracle's float32 values so that every
    later ranking is comparable bit for bit."""
    steps = 40
    wl, hot = _hot("mikv", 1024)
    B, Hq, Hkv, D, T, nr = wl["B"], wl["Hq"], wl["Hkv"], wl["D"], wl["T"], wl["nr"]
    g = Hq // Hkv
    _check_prefill(hot, [(0, 0), (63, 31)], np.array([0, 127, 20000, T - 1]))
    cs = inputs.random_scores(B, Hq, T, seed=6)
    kvq.requant_demote(hot.cache, 0, k_src=hot.k, v_src=hot.v, colscore=cs.cuda())
    sample = [9, B * Hkv - 1]
    units = {}
    for u in sample:
        b, h = u // Hkv, u % Hkv
        units[u] = OP.MiKVUnit(np_(hot.k[b, h]), np_(hot.v[b, h]), np_(cs[b, h * g:(h + 1) * g]), nr, G)
        assert_tiers_equal(gpu_tier_rows(hot.cache.tiers[0], u), oracle_tier_rows(units[u].hi), f"INT4 u{u}")
    cum = hot.cache.cum_score
    n_dem = 0
    for t in range(steps):
        qd, kd, vd = hot.dec[t]
        od, _ = kvq.decode_attn_qkv(qd, kd, vd, hot.cache, hot.scale)
        for u in sample:
            b, h = u // Hkv, u % Hkv
            ro, _ = units[u].attend(T + t, np_(qd[b, h * g:(h + 1) * g]), np_(kd[b, h]), np_(vd[b, h]),
                                    hot.scale)
            assert_attn_close(od[b, h * g:(h + 1) * g], ro, f"decode step {t} unit {u}")
            ref = np.array([units[u].cs[j] for j in range(T + t + 1)], dtype=np.float32)
            got = cum[u, :T + t + 1].cpu().numpy()
            err = np.abs(got.astype(np.float64) - ref)
            assert np.all(err <= 1e-4 * np.abs(ref) + 1e-6), f"cumulative scores step {t} unit {u}"
            cum[u, :T + t + 1] = torch.from_numpy(ref).cuda()
        kvq.requant_demote(hot.cache, t + 1)
        for u in sample:
            n_dem += len(units[u].tail()[1])
            assert_tiers_equal(gpu_tier_rows(hot.cache.tiers[0], u), oracle_tier_rows(units[u].hi),
                               f"INT4 u{u} step {t}")
            assert_tiers_equal(gpu_tier_rows(hot.cache.tiers[1], u), oracle_tier_rows(units[u].lo),
                               f"INT2 u{u} step {t}")
    assert kvq.device_status() == 0
    assert n_dem > 0, "no demotion in the run"


def test_sweep_graph_pyramid():
    """The 32-layer pyramid sweep as the benchmark runs it (every layer's budget, one CUDA
    graph of the 32 layers' decode launches per step), at batch 2: selections of sampled
    layers against the oracle's on the exported column scores, then 24 graph-replayed steps
    of sampled units of layers 0, 16 and 31 against the oracle's MiniKV life cycle (the
    first flush of each layer falls inside the run)."""
    steps = 24
    wl = dict(bench.WORKLOADS["pyramid"])
    wl["B"] = 2
    dev = torch.device("cuda", 0)
    sw = bench.Sweep(wl, dev, seed=0)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        sw.prefill_build(s)
    torch.cuda.synchronize()
    B, H, D, T = wl["B"], wl["Hq"], wl["D"], wl["T"]
    cs = sw.cs.cpu().numpy()                  # every layer prefills the same prompt
    sample = [(0, 0, 5), (16, 1, 30), (31, 1, 0)]          # (layer, batch, head)
    units = {}
    for l, b, h in sample:
        ly = sw.layers[l]
        sel = OS.select_unit(cs[b, h], ly["k_hh"], ly["w"])
        assert np.array_equal(np.sort(ly["idx"][b, h].cpu().numpy()), sel), f"selection layer {l}"
        units[(l, b, h)] = OP.MiniKVUnit(np_(sw.k[b, h]), np_(sw.v[b, h]), sel, 0, G)
    sw.capture(s)
    torch.cuda.synchronize()
    # the capture's warm-up call decoded one step of every layer from the zeroed input
    # buffers (a zero query, a zero token appended): replay it on the oracle side too
    q0, k0, v0 = np_(sw.qd), np_(sw.kd), np_(sw.vd)
    assert not q0.any() and not k0.any() and not v0.any()
    for (l, b, h), un in units.items():
        un.step(T, q0[b, h:h + 1], k0[b, h], v0[b, h], sw.scale)
    for t in range(steps):
        with torch.cuda.stream(s):
            sw.decode_step(t, s)
        torch.cuda.synchronize()
        qd, kd, vd = sw.dec[t]
        for (l, b, h), un in units.items():
            ro, _ = un.step(T + 1 + t, np_(qd[b, h:h + 1]), np_(kd[b, h]), np_(vd[b, h]), sw.scale)
            assert_attn_close(sw.o_dec[l, b, h], ro[0], f"step {t} layer {l} unit {b},{h}")
    assert kvq.device_status() == 0
    for (l, b, h), un in units.items():
        t0 = sw.layers[l]["cache"].tiers[0]
        u = b * H + h
        npk = len(un.ids)
        assert int(t0.count[u]) == npk, f"packed count layer {l}"
        assert np.array_equal(u32(t0.k_codes[u, :npk // 16]), un.kw.view(np.uint32))
        assert np.array_equal(u32(t0.v_codes[u, :npk]), un.vw.view(np.uint32))
