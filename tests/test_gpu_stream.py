"""Streamed decode (one query head per KV head, MiniKV format, at least 8 items per CTA for
the largest grid the launcher forms, so the streamed launch is taken whatever the GPU): every
unit against the oracle over steps that cross residual flushes.  Each unit's items are
spread over several CTAs (partials merged by the second launch); per-unit budgets from zero
to the capacity leave whole CTA runs with no live item."""
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import policies as OP
from oracle import select as OS
from tests.helpers import assert_attn_close, np_, u16, u32

pytestmark = pytest.mark.gpu

# 128 units x at least 64 static items each (chunks of 256 tokens for G = 32, 128 for G = 16,
# then ring pieces of 32 rows) >= 8192 = 8 items for each of 1024 CTAs
B, H, D, W, STEPS = 4, 32, 128, 512, 40


def _decode_against_oracle(cache, x, T, units, G, seed, dtype=torch.float16):
    scale = 1.0 / math.sqrt(D)
    ch = 256 if G == 32 else 128
    n_items = (cache.tiers[0].spec.cap + ch - 1) // ch + (cache.res_cap + 31) // 32
    assert B * H * n_items >= 8 * 1024
    assert kvq.decode_launches(cache) == 2, "the list launch and its merge launch" 
    for t in range(STEPS):
        qd, kd, vd = (z.cuda() for z in inputs.make_decode_step(B, H, H, D, t, dtype=dtype, seed=seed))
        od, ld = kvq.decode_attn_qkv(qd, kd, vd, cache, scale)
        torch.cuda.synchronize()
        for u, ref in units.items():
            b, h = u // H, u % H
            ro, rl = ref.step(T + t, np_(qd[b, h:h + 1]), np_(kd[b, h]), np_(vd[b, h]), scale)
            assert_attn_close(od[b, h], ro[0], f"decode step {t} unit {u}")
            assert abs(float(ld[b, h]) - rl[0]) < 1e-3, f"lse step {t} unit {u}"
    assert kvq.device_status() == 0
    t0 = cache.tiers[0]
    cnt = t0.count.cpu().numpy()
    for u, ref in units.items():
        npk = len(ref.ids)
        assert cnt[u] == npk, f"unit {u} count"
        assert np.array_equal(t0.token_id[u, :npk].cpu().numpy(), np.array(ref.ids))
        assert np.array_equal(u32(t0.k_codes[u, :npk // 16]), ref.kw.view(np.uint32))
        assert np.array_equal(u16(t0.k_scale[u, :npk // G]), ref.ksc.view(np.uint16))
        assert np.array_equal(u32(t0.v_codes[u, :npk]), ref.vw.view(np.uint32))
        assert np.array_equal(u16(t0.v_scale[u, :npk]), ref.vsc.view(np.uint16))
        assert int(cache.res_len[u]) == len(ref.res), f"unit {u} residual length"


def test_stream_per_unit_budgets():
    """Budgets 0 .. 16000 per unit (G = 32, nr = 0: flushes every 32 steps), built by the
    fused prefill-end build from seeded scores."""
    T, G, nr, seed = 17000, 32, 0, 21
    rng = np.random.default_rng(seed)
    budgets = rng.integers(0, 16001, size=B * H)
    budgets[:4] = [0, 16000, 1, 127]
    x = inputs.make_qkv(B, H, H, T, D, seed=seed)
    cs = inputs.random_scores(B, H, T, seed=seed + 1)
    kmax = int(budgets.max())
    cap = ((kmax + W + STEPS) // G + 2) * G
    cache = kvq.make_cache(B, H, H, D, G, torch.float16, kvq.POLICY_MINIKV,
                           [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr)
    idx = torch.empty((B, H, kmax + W), dtype=torch.int32, device="cuda")
    kvq.minikv_prefill_build(cache, x.k.cuda(), x.v.cuda(), cs.cuda(),
                             torch.tensor(budgets, dtype=torch.int32, device="cuda"), W, kmax=kmax, idx_out=idx)
    gsel = idx.cpu().numpy().reshape(B * H, -1)
    units = {}
    for u in range(B * H):
        b, h = u // H, u % H
        sel = OS.select_unit(np_(cs[b, h]), int(budgets[u]), W)
        assert np.array_equal(np.sort(gsel[u, :len(sel)]), sel), f"selection of unit {u}"
        units[u] = OP.MiniKVUnit(np_(x.k[b, h]), np_(x.v[b, h]), sel, nr, G)
    _decode_against_oracle(cache, x, T, units, G, seed)


def test_stream_group16_bf16():
    """Groups of 16 and a bf16 prompt, ring and output, one budget for every unit (selection +
    two-launch build), nr = 64: flushes every 16 steps once the ring holds 80 tokens."""
    T, G, nr, seed, k_hh, dt = 17000, 16, 64, 23, 15000, torch.bfloat16
    x = inputs.make_qkv(B, H, H, T, D, dtype=dt, seed=seed)
    cs = inputs.random_scores(B, H, T, seed=seed + 1)
    n_sel = k_hh + W
    cap = ((n_sel + STEPS) // G + 2) * G
    cache = kvq.make_cache(B, H, H, D, G, dt, kvq.POLICY_MINIKV,
                           [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr)
    idx, _ = kvq.select_tokens(cs.cuda(), torch.full((B * H,), k_hh, dtype=torch.int32, device="cuda"), W)
    kvq.requant_demote(cache, 0, k_src=x.k.cuda(), v_src=x.v.cuda(), sel_idx=idx, n_sel=n_sel)
    gsel = idx.cpu().numpy().reshape(B * H, -1)
    units = {}
    for u in range(B * H):
        b, h = u // H, u % H
        sel = OS.select_unit(np_(cs[b, h]), k_hh, W)
        assert np.array_equal(np.sort(gsel[u]), sel), f"selection of unit {u}"
        units[u] = OP.MiniKVUnit(np_(x.k[b, h]), np_(x.v[b, h]), sel, nr, G)
    _decode_against_oracle(cache, x, T, units, G, seed, dt)
