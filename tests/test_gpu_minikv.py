"""MiniKV life cycle end to end on the GPU against the oracle: prefill ->
heavy hitters + window -> INT2 pack -> decode steps with residual flushes."""
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import attention as OA
from oracle import policies as OP
from oracle import quant as OQ
from oracle import select as OS
from tests.helpers import assert_attn_close, assert_scores_close, np_, selection_agrees, u16, u32

pytestmark = pytest.mark.gpu


def _pipeline(B, H, T, D, steps, nr, n_out, out_scale, seed, hh=25, rw=25, G=32, dtype=torch.float16):
    dev = "cuda"
    scale = 1.0 / math.sqrt(D)
    outl = inputs.outlier_channels(H, D, n_out, seed)
    x = inputs.make_qkv(B, H, H, T, D, dtype=dtype, seed=seed, outliers=outl, outlier_scale=out_scale)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o, lse, cs = kvq.prefill_attn_scores(q, k, v, scale)
    k_hh, w = OS.budget(T, hh, rw)
    n_sel = k_hh + w
    # oracle prefill scores -> oracle selection
    ref_sel, ref_cs = [], []
    for b in range(B):
        for h in range(H):
            _, _, c = OA.prefill_head(np_(x.q[b, h]), np_(x.k[b, h]), np_(x.v[b, h]), scale)
            ref_cs.append(c)
            ref_sel.append(OS.select_unit(c.astype(np.float32), k_hh, w))
    assert_scores_close(cs.reshape(B * H, T), np.stack(ref_cs), "colscore")
    idx, n = kvq.select_tokens(cs, torch.full((B * H,), k_hh, dtype=torch.int32, device=dev), w)
    gsel = idx.cpu().numpy().reshape(B * H, -1)
    same = [selection_agrees(gsel[u], ref_sel[u], ref_cs[u], k_hh, w) for u in range(B * H)]
    r0 = n_sel if n_sel <= nr else nr + (n_sel - nr) % G
    cap = ((n_sel - r0 + steps + G - 1) // G + 1) * G
    cache = kvq.make_cache(B, H, H, D, G, dtype, kvq.POLICY_MINIKV,
                           [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr)
    kvq.requant_demote(cache, 0, k_src=k, v_src=v, sel_idx=idx, n_sel=n_sel)
    units = [OP.MiniKVUnit(np_(x.k[u // H, u % H]), np_(x.v[u // H, u % H]), ref_sel[u], nr, G)
             for u in range(B * H)]
    # packed prefill cache is bit-exact where the selections agree
    t0 = cache.tiers[0]
    cnt = t0.count.cpu().numpy()
    for u in range(B * H):
        if not same[u]:
            continue
        npk = len(units[u].ids)
        assert cnt[u] == npk
        assert np.array_equal(u32(t0.k_codes[u, :npk // 16]), units[u].kw.view(np.uint32))
        assert np.array_equal(u16(t0.k_scale[u, :npk // G]), units[u].ksc.view(np.uint16))
        assert np.array_equal(u32(t0.v_codes[u, :npk]), units[u].vw.view(np.uint32))
        assert np.array_equal(u16(t0.v_zero[u, :npk]), units[u].vze.view(np.uint16))
    max_err = 0.0
    for t in range(steps):
        qd, kd, vd = inputs.make_decode_step(B, H, H, D, t, dtype=dtype, seed=seed, outliers=outl,
                                             outlier_scale=out_scale)
        od, ld = kvq.decode_attn_qkv(qd.to(dev), kd.to(dev), vd.to(dev), cache, scale)
        kvq.requant_demote(cache, t + 1)
        for u in range(B * H):
            if not same[u]:
                continue
            b, h = u // H, u % H
            ro, rl = units[u].step(T + t, np_(qd[b, h:h + 1]), np_(kd[b, h]), np_(vd[b, h]), scale)
            max_err = max(max_err, assert_attn_close(od[b, h], ro[0], f"decode step {t} unit {u}"))
            assert abs(float(ld[b, h]) - rl[0]) < 1e-3
    assert kvq.device_status() == 0
    # final cache state: packed codes and residual positions match
    cnt = t0.count.cpu().numpy()
    for u in range(B * H):
        if not same[u]:
            continue
        npk = len(units[u].ids)
        assert cnt[u] == npk
        assert np.array_equal(t0.token_id[u, :npk].cpu().numpy(), np.array(units[u].ids))
        assert np.array_equal(u32(t0.k_codes[u, :npk // 16]), units[u].kw.view(np.uint32))
        assert np.array_equal(u32(t0.v_codes[u, :npk]), units[u].vw.view(np.uint32))
    assert sum(same) >= 1
    return max_err


def test_minikv_tiny_config():
    """Batch 1, 2 heads, head dim 64, prompt 256, two outlier key channels x8, INT2 keys per
    channel and values per token in groups of 32, 25% + 25% budget, 16 steps, seed 0."""
    _pipeline(B=1, H=2, T=256, D=64, steps=16, nr=0, n_out=2, out_scale=8.0, seed=0)


def test_minikv_residual_flushes():
    """nr = 128 residual with flushes every 32 steps (prompt 1024, 70 steps)."""
    _pipeline(B=2, H=2, T=1024, D=128, steps=70, nr=128, n_out=3, out_scale=10.0, seed=1)


def test_minikv_llama_layer():
    """LLaMA2-7B-shaped layer: 32 heads, prompt 4096, 2% outlier channels x10, nr = 128,
    128 decode steps (four flushes)."""
    _pipeline(B=1, H=32, T=4096, D=128, steps=128, nr=128, n_out=3, out_scale=10.0, seed=0)


def test_minikv_bf16():
    """bf16 prompt, decode inputs, residual ring and output (prompt 1024, 40 steps, nr = 0)."""
    _pipeline(B=2, H=2, T=1024, D=128, steps=40, nr=0, n_out=2, out_scale=8.0, seed=4, dtype=torch.bfloat16)


def test_minikv_group16():
    """Groups of 16 (the MiniKV review's default): key scale rows every 16 tokens, eight value
    groups per token, flushes every 16 steps past nr = 64 (prompt 1024, 40 steps)."""
    _pipeline(B=2, H=3, T=1024, D=128, steps=40, nr=64, n_out=3, out_scale=10.0, seed=6, G=16)


def test_group16_limits_are_reported():
    """G = 16 is built for the single-head 2-bit MiniKV path only: other shapes are refused
    before any launch."""
    B, D, T, G = 1, 128, 256, 16
    x = inputs.make_qkv(B, 2, 2, T, D, seed=3)
    with pytest.raises(RuntimeError, match="G = 16"):
        kvq.make_cache(B, 4, 2, D, G, torch.float16, kvq.POLICY_MINIKV,
                       [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, 256)], nr=32)
    c1 = kvq.make_cache(B, 2, 2, D, G, torch.float16, kvq.POLICY_MINIKV,
                        [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, 256)], nr=32)
    with pytest.raises(RuntimeError, match="G = 32"):
        kvq.minikv_prefill_build(c1, x.k.contiguous().cuda(), x.v.contiguous().cuda(),
                                 torch.ones((B, 2, T), device="cuda"),
                                 torch.full((B * 2,), 32, dtype=torch.int32, device="cuda"), 32)


def _cache_arrays(c):
    t = c.tiers[0]
    return [t.k_codes, t.k_scale, t.k_zero, t.v_codes, t.v_scale, t.v_zero, t.token_id, t.count,
            c.res_k, c.res_v, c.res_token_id, c.res_start, c.res_len, c.seq_len]


@pytest.mark.parametrize("nr,dtype", [(0, torch.float16), (128, torch.float16), (16, torch.bfloat16)])
def test_fused_build_equals_two_launch_build(nr, dtype):
    """minikv_prefill_build leaves every array of the cache exactly as select_tokens
    followed by requant_demote(step 0) does (scores with many ties; ragged prompt)."""
    B, H, T, D, G, w, k_hh = 2, 3, 700, 128, 32, 64, 177
    x = inputs.make_qkv(B, H, H, T, D, dtype=dtype, seed=41, outliers=inputs.outlier_channels(H, D, 2, 41),
                        outlier_scale=8.0)
    k, v = x.k.cuda(), x.v.cuda()
    cs = inputs.random_scores(B, H, T, seed=41, ties=24).cuda()
    kh = torch.full((B * H,), k_hh, dtype=torch.int32, device="cuda")
    n = k_hh + w
    r0 = n if n <= nr else nr + (n - nr) % G
    cap = ((n - r0) // G + 2) * G

    def make():
        return kvq.make_cache(B, H, H, D, G, dtype, kvq.POLICY_MINIKV, [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)],
                              nr=nr)
    two, fused = make(), make()
    idx, _ = kvq.select_tokens(cs, kh, w, kmax=k_hh)
    kvq.requant_demote(two, 0, k_src=k, v_src=v, sel_idx=idx, n_sel=n)
    idx_f = torch.full((B, H, k_hh + w), -7, dtype=torch.int32, device="cuda")
    kvq.minikv_prefill_build(fused, k, v, cs, kh, w, kmax=k_hh, idx_out=idx_f)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    assert torch.equal(idx, idx_f)
    for a, b in zip(_cache_arrays(two), _cache_arrays(fused)):
        assert torch.equal(a, b)


def test_fused_build_per_unit_budgets_against_oracle():
    """Per-unit heavy-hitter budgets (0, a few, most of the prompt): each unit's selection
    equals the oracle's on the same float32 scores, and its packed words, scales, zeros,
    ids and residual rows equal the oracle's MiniKV build."""
    B, H, T, D, G, w, nr = 1, 4, 520, 128, 32, 40, 32
    budgets = [0, 9, 200, 480]
    x = inputs.make_qkv(B, H, H, T, D, seed=43)
    cs = inputs.random_scores(B, H, T, seed=43, ties=16)
    kh = torch.tensor(budgets, dtype=torch.int32, device="cuda")
    cap = ((max(budgets) + w) // G + 2) * G
    c = kvq.make_cache(B, H, H, D, G, torch.float16, kvq.POLICY_MINIKV, [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)],
                       nr=nr)
    kvq.minikv_prefill_build(c, x.k.cuda(), x.v.cuda(), cs.cuda(), kh, w)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    t = c.tiers[0]
    for u in range(H):
        sel = OS.select_unit(np_(cs[0, u]), min(budgets[u], T - w), w)
        ref = OP.MiniKVUnit(np_(x.k[0, u]), np_(x.v[0, u]), sel, nr, G)
        npk = len(ref.ids)
        assert int(t.count[u]) == npk, f"unit {u}"
        assert np.array_equal(t.token_id[u, :npk].cpu().numpy(), np.array(ref.ids, dtype=np.int32))
        assert np.array_equal(u32(t.k_codes[u, :npk // 16]), ref.kw.view(np.uint32))
        assert np.array_equal(u16(t.k_scale[u, :npk // G]), ref.ksc.view(np.uint16))
        assert np.array_equal(u16(t.k_zero[u, :npk // G]), ref.kze.view(np.uint16))
        assert np.array_equal(u32(t.v_codes[u, :npk]), ref.vw.view(np.uint32))
        assert np.array_equal(u16(t.v_scale[u, :npk]), ref.vsc.view(np.uint16))
        assert np.array_equal(u16(t.v_zero[u, :npk]), ref.vze.view(np.uint16))
        r0 = len(ref.res)
        assert int(c.res_len[u]) == r0 and int(c.res_start[u]) == 0 and int(c.seq_len[u]) == T
        assert np.array_equal(c.res_token_id[u, :r0].cpu().numpy(), np.array([r[0] for r in ref.res], dtype=np.int32))
        assert np.array_equal(np_(c.res_k[u, :r0]), np.stack([r[1] for r in ref.res]) if r0 else np.zeros((0, D)))
