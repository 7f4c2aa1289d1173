"""decode_attn_qkv_static: the decode entry point for callers that cannot give the
library scratch memory (an engine whose allocator already owns all free device
memory, or C code without a device allocator).  DiffKV and MiKV caches keep the
step's logits in scratch, and single-head MiniKV caches large enough for the streamed
launch keep its partials there, so those run here: two calls in a row, each checked
against the CPU oracle (outputs, cumulative scores, tier contents) and against the
caller-workspace entry point on a twin cache.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import policies as OP
from tests.helpers import (assert_attn_close, assert_tiers_equal, gpu_tier_rows, np_,
                           oracle_tier_rows)

pytestmark = pytest.mark.gpu

G = 32


def _scratch_used(cache):
    need = kvq.lib().kvq_decode_workspace_bytes(ctypes.byref(cache.desc))
    assert 0 < need <= kvq.STATIC_SCRATCH_BYTES
    return need


def _twin_outputs(a, b, what):
    x, y = np_(a).astype(np.float64), np_(b).astype(np.float64)
    assert np.all(np.abs(x - y) <= 2e-3 + 1e-2 * np.abs(y)), what


def test_static_scratch_mikv_two_calls():
    """MiKV, GQA 8/2, bf16: the static path's outputs and cumulative scores match the
    oracle call after call, and its tiers after each re-ranking."""
    B, Hq, Hkv, T, D, nr, steps = 1, 8, 2, 320, 128, 16, 2
    g = Hq // Hkv
    x = inputs.make_qkv(B, Hq, Hkv, T + steps, D, dtype=torch.bfloat16, seed=31,
                        outliers=inputs.outlier_channels(Hkv, D, 1, 31), outlier_scale=12.0)
    cs = inputs.random_scores(B, Hq, T, seed=31)
    n_q = T - nr + steps

    def make():
        c = kvq.make_cache(B, Hq, Hkv, D, G, torch.bfloat16, kvq.POLICY_MIKV,
                           [kvq.TierSpec(4, 4, kvq.AXIS_TOKEN, n_q // 5 + 2),
                            kvq.TierSpec(2, 2, kvq.AXIS_TOKEN, n_q + 1)],
                           nr=nr, score_cap=T + steps + 1, hi_den=5)
        kvq.requant_demote(c, 0, k_src=x.k[:, :, :T].contiguous().cuda(),
                           v_src=x.v[:, :, :T].contiguous().cuda(), colscore=cs.cuda())
        return c

    st, ws = make(), make()
    _scratch_used(st)
    units = [OP.MiKVUnit(np_(x.k[0, h, :T]), np_(x.v[0, h, :T]), np_(cs[0, h * g:(h + 1) * g]), nr, G)
             for h in range(Hkv)]
    scale = 1.0 / math.sqrt(D)
    for t in range(steps):                               # two calls in a row
        qd = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(500 + t)).bfloat16()
        kd, vd = x.k[:, :, T + t].contiguous(), x.v[:, :, T + t].contiguous()
        o_st, _ = kvq.decode_attn_qkv_static(qd.cuda(), kd.cuda(), vd.cuda(), st, scale)
        o_ws, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), ws, scale)
        torch.cuda.synchronize()
        _twin_outputs(o_st, o_ws, f"static vs workspace, call {t}")
        for u in range(Hkv):
            ro, _ = units[u].attend(T + t, np_(qd[0, u * g:(u + 1) * g]), np_(kd[0, u]), np_(vd[0, u]), scale)
            assert_attn_close(o_st[0, u * g:(u + 1) * g], ro, f"call {t} unit {u}")
            ref = np.array([units[u].cs[j] for j in range(T + t + 1)], dtype=np.float32)
            got = st.cum_score[u, :T + t + 1].cpu().numpy()
            assert np.all(np.abs(got.astype(np.float64) - ref) <= 1e-4 * np.abs(ref) + 1e-6), \
                f"cumulative scores, call {t} unit {u}"
            # both caches continue from the oracle's float32 scores: later rankings compare bit for bit
            st.cum_score[u, :T + t + 1] = torch.from_numpy(ref).cuda()
            ws.cum_score[u, :T + t + 1] = torch.from_numpy(ref).cuda()
        kvq.requant_demote(st, t + 1)
        kvq.requant_demote(ws, t + 1)
        for u in range(Hkv):
            units[u].tail()
            assert_tiers_equal(gpu_tier_rows(st.tiers[0], u), oracle_tier_rows(units[u].hi), f"INT4 u{u} call {t}")
            assert_tiers_equal(gpu_tier_rows(st.tiers[1], u), oracle_tier_rows(units[u].lo), f"INT2 u{u} call {t}")
    assert kvq.device_status() == 0


def test_static_scratch_diffkv_two_calls():
    """DiffKV, GQA 10/2: the static path keeps each step's logits in the built-in array
    and adds the window scores from there; outputs and the tiers after each window exit
    match the oracle, and the twin cache with a caller workspace."""
    B, Hq, Hkv, T, D, W, steps = 1, 10, 2, 384, 128, 64, 2
    g = Hq // Hkv
    x = inputs.make_qkv(B, Hq, Hkv, T + steps, D, seed=33)
    cs = inputs.random_scores(B, Hq, T, seed=33) + 0.01
    f = inputs.dirichlet_fractions(B * Hkv, seed=33)
    n_high = np.floor(f[:, 0] * (T - W)).astype(np.int32)
    n_low = np.floor(f[:, 1] * (T - W)).astype(np.int32)

    def make():
        c = kvq.make_cache(B, Hq, Hkv, D, G, torch.float16, kvq.POLICY_DIFFKV,
                           [kvq.TierSpec(8, 4, kvq.AXIS_TOKEN, int(n_high.max()) + steps + 1),
                            kvq.TierSpec(4, 2, kvq.AXIS_TOKEN, int(n_low.max()) + steps + 1)], nr=W)
        kvq.requant_demote(c, 0, k_src=x.k[:, :, :T].contiguous().cuda(),
                           v_src=x.v[:, :, :T].contiguous().cuda(), colscore=cs.cuda(),
                           n_high=torch.from_numpy(n_high).cuda(), n_low=torch.from_numpy(n_low).cuda())
        return c

    st, ws = make(), make()
    _scratch_used(st)
    units = [OP.DiffKVUnit(np_(x.k[0, h, :T]), np_(x.v[0, h, :T]), np_(cs[0, h * g:(h + 1) * g]),
                           int(n_high[h]), int(n_low[h]), W, G) for h in range(Hkv)]
    scale = 1.0 / math.sqrt(D)
    for t in range(steps):                               # two calls in a row
        qd = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(700 + t)).half()
        kd, vd = x.k[:, :, T + t].contiguous(), x.v[:, :, T + t].contiguous()
        o_st, _ = kvq.decode_attn_qkv_static(qd.cuda(), kd.cuda(), vd.cuda(), st, scale)
        o_ws, _ = kvq.decode_attn_qkv(qd.cuda(), kd.cuda(), vd.cuda(), ws, scale)
        kvq.requant_demote(st, t + 1)
        kvq.requant_demote(ws, t + 1)
        torch.cuda.synchronize()
        _twin_outputs(o_st, o_ws, f"static vs workspace, call {t}")
        assert torch.equal(st.win_acc, ws.win_acc), f"window scores, call {t}"
        for u in range(Hkv):
            ro, _, _ = units[u].step(T + t, np_(qd[0, u * g:(u + 1) * g]), np_(kd[0, u]), np_(vd[0, u]), scale)
            assert_attn_close(o_st[0, u * g:(u + 1) * g], ro, f"call {t} unit {u}")
            assert_tiers_equal(gpu_tier_rows(st.tiers[0], u), oracle_tier_rows(units[u].high), f"K8V4 u{u}")
            assert_tiers_equal(gpu_tier_rows(st.tiers[1], u), oracle_tier_rows(units[u].low), f"K4V2 u{u}")
    assert kvq.device_status() == 0


def test_static_scratch_minikv_streamed_two_calls():
    """MiniKV with one query head per KV head, large enough for the streamed launch: its
    per-(CTA, unit) partials live in the scratch.  Two calls in a row against the oracle
    (sampled units) and against the caller-workspace call on a twin cache (every unit)."""
    from oracle import select as OS
    B, H, T, D, W, k_hh, steps = 4, 32, 17000, 128, 512, 16000, 2
    x = inputs.make_qkv(B, H, H, T, D, seed=37)
    cs = inputs.random_scores(B, H, T, seed=38)
    cap = ((k_hh + W + steps) // G + 2) * G

    def make():
        c = kvq.make_cache(B, H, H, D, G, torch.float16, kvq.POLICY_MINIKV,
                           [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=0)
        kvq.minikv_prefill_build(c, x.k.cuda(), x.v.cuda(), cs.cuda(),
                                 torch.full((B * H,), k_hh, dtype=torch.int32, device="cuda"), W)
        return c

    st, ws = make(), make()
    _scratch_used(st)
    assert kvq.decode_launches(st) == 2, "the streamed launch and its merge launch"
    sample = [0, 37, B * H - 1]
    units = {u: OP.MiniKVUnit(np_(x.k[u // H, u % H]), np_(x.v[u // H, u % H]),
                              OS.select_unit(np_(cs[u // H, u % H]), k_hh, W), 0, G) for u in sample}
    scale = 1.0 / math.sqrt(D)
    for t in range(steps):
        qd, kd, vd = (z.cuda() for z in inputs.make_decode_step(B, H, H, D, t, seed=37))
        o1, l1 = kvq.decode_attn_qkv_static(qd, kd, vd, st, scale)
        o2, l2 = kvq.decode_attn_qkv(qd, kd, vd, ws, scale)
        torch.cuda.synchronize()
        _twin_outputs(o1, o2, f"step {t}: static vs caller workspace")
        for u in sample:
            b, h = u // H, u % H
            ro, rl = units[u].step(T + t, np_(qd[b, h:h + 1]), np_(kd[b, h]), np_(vd[b, h]), scale)
            assert_attn_close(o1[b, h], ro[0], f"step {t} unit {u}")
            assert abs(float(l1[b, h]) - rl[0]) < 1e-3
    assert torch.equal(st.res_len, ws.res_len) and torch.equal(st.tiers[0].count, ws.tiers[0].count)
    assert kvq.device_status() == 0


def test_static_scratch_rejects_a_cache_too_large():
    """A cache needing more scratch than is built in is refused before any launch."""
    B, Hq, Hkv, D = 1, 8, 1, 128
    slots = kvq.STATIC_SCRATCH_BYTES // (4 * Hq) + 4096      # per-token logits outgrow the array
    c = kvq.make_cache(B, Hq, Hkv, D, 32, torch.float16, kvq.POLICY_MIKV,
                       [kvq.TierSpec(4, 4, kvq.AXIS_TOKEN, 64), kvq.TierSpec(2, 2, kvq.AXIS_TOKEN, slots)],
                       nr=16, score_cap=64)
    need = kvq.lib().kvq_decode_workspace_bytes(ctypes.byref(c.desc))
    assert need > kvq.STATIC_SCRATCH_BYTES
    q = torch.zeros((B, Hq, D), dtype=torch.float16, device="cuda")
    kn = torch.zeros((B, Hkv, D), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attn_qkv_static(q, kn, kn, c, 0.1)
    assert e.value.status == kvq.KVQ_EWORKSPACE
    assert kvq.device_status() == 0
