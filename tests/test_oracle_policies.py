"""Pins of the oracle cache life cycles: hand-worked cases under uniform attention,
conservation laws and the pages' byte closed forms (no GPU)."""
import math

import numpy as np

from oracle import accounting as acc
from oracle import attention as A
from oracle import policies as P
from oracle import quant

F32 = np.float32


def _kv(T, D, seed):
    r = np.random.default_rng(seed)
    k = r.normal(size=(T, D)).astype(np.float16).astype(F32)
    v = r.normal(size=(T, D)).astype(np.float16).astype(F32)
    return k, v


# ---------------------------------------------------------------- MiniKV

def test_minikv_full_precision_reduces_to_textbook():
    """Every token selected and the residual never full: decode is plain attention."""
    T, D = 40, 32
    k, v = _kv(T + 3, D, 0)
    u = P.MiniKVUnit(k[:T], v[:T], np.arange(T), nr=64, group=32)
    r = np.random.default_rng(1)
    for t in range(3):
        q = r.normal(size=(1, D))
        o, lse = u.step(T + t, q, k[T + t], v[T + t], 0.2)
        o2, lse2, _ = A.decode_head(q[0], k[:T + t + 1], v[:T + t + 1], 0.2)
        assert np.allclose(o[0], o2, atol=1e-12) and abs(lse[0] - lse2) < 1e-12


def test_minikv_residual_and_flush_schedule():
    T, D, G, nr = 80, 32, 32, 4
    k, v = _kv(T + 40, D, 2)
    sel = np.sort(np.random.default_rng(3).choice(T, 40, replace=False))
    u = P.MiniKVUnit(k[:T], v[:T], sel, nr=nr, group=G)
    assert len(u.ids) == 32 and len(u.res) == 8                # r0 = 4 + (36 mod 32)
    assert u.ids == list(sel[:32]) and [r[0] for r in u.res] == list(sel[32:])
    q = np.zeros((1, D))
    for t in range(30):
        u.step(T + t, q, k[T + t], v[T + t], 0.1)
        if t < 27:
            assert len(u.ids) == 32 and len(u.res) == 9 + t
        else:
            assert len(u.ids) == 64 and len(u.res) == nr + (t - 27)
    # packed block 2 = the 32 oldest residual tokens, in arrival order
    assert u.ids[32:] == list(sel[32:]) + [T + t for t in range(24)]
    # token conservation
    assert sorted(u.ids + [r[0] for r in u.res]) == sorted(list(sel) + [T + t for t in range(30)])


def test_minikv_zero_query_is_mean_of_dequantised_values():
    T, D = 64, 32
    k, v = _kv(T + 1, D, 4)
    u = P.MiniKVUnit(k[:T], v[:T], np.arange(T), nr=0, group=32)
    o, lse = u.step(T, np.zeros((1, D)), k[T], v[T], 0.5)
    vh = quant.unpack_token(*quant.quant_pack_token(v[:T], 2, 32), 2, 32)
    want = np.concatenate([vh, v[T:T + 1]]).astype(np.float64).mean(axis=0)
    assert np.allclose(o[0], want, atol=1e-12) and abs(lse[0] - math.log(T + 1)) < 1e-12


# ---------------------------------------------------------------- DiffKV

def _diffkv_case():
    T, D = 8, 32
    k, v = _kv(T + 3, D, 5)
    cs = np.array([[4, 1, 2, 0.5, 1, 0.25, 0.2, 0.5],
                   [2, 2.8, 1, 0.5, 0.5, 1, 0.1, 0.6]], F32)
    return T, D, k, v, cs


def test_diffkv_prefill_split_by_hand():
    T, D, k, v, cs = _diffkv_case()
    sig = P.diffkv_significance(cs, T)
    # max_h cs/(T-j): 0.5, 0.4, 1/3, 0.1, 0.25, 1/3 for the six candidates
    assert np.allclose(sig[:6], [0.5, 0.4, 1 / 3, 0.1, 0.25, 1 / 3], rtol=1e-7)
    u = P.DiffKVUnit(k[:T], v[:T], cs, n_high=2, n_low=2, window=2, group=32)
    assert u.high.ids() == [0, 1]
    assert u.low.ids() == [2, 5]            # 2 and 5 tie at 1/3: both low, 2 ranked first
    assert u.pruned == [3, 4]
    assert abs(float(u.alpha_h) - 3.2) < 1e-6 and abs(float(u.alpha_l) - 8 / 3) < 1e-6
    assert [w[0] for w in u.win] == [6, 7]


def test_diffkv_window_exit_by_hand():
    """q = 0 gives every cached token 1/(#cached); decisions worked out by hand:
    token 6 -> pruned (0.114 < 0.296), token 7 -> low (0.295 in [0.267, 0.32)),
    token 8 -> pruned (0.137 < 0.242)."""
    T, D, k, v, cs = _diffkv_case()
    u = P.DiffKVUnit(k[:T], v[:T], cs, n_high=2, n_low=2, window=2, group=32)
    q = np.zeros((2, D))
    got = []
    for t in range(3):
        o, lse, dec = u.step(T + t, q, k[T + t], v[T + t], 0.3)
        got.append(dec)
        n_cached = len(u.high.rows) + len(u.low.rows) + len(u.win) + (dec[1] == "pruned")
        assert np.allclose(lse, math.log(n_cached), atol=1e-12)
    assert got == [(6, "pruned"), (7, "low"), (8, "pruned")]
    assert u.low.ids() == [2, 5, 7] and u.pruned == [3, 4, 6, 8]
    # partition: every position is in exactly one of window / high / low / pruned
    every = u.high.ids() + u.low.ids() + u.pruned + [w[0] for w in u.win]
    assert sorted(every) == list(range(T + 3))


def test_diffkv_alpha_l_zero_prunes_nothing():
    T, D = 96, 32
    k, v = _kv(T + 20, D, 6)
    cs = np.random.default_rng(7).random((2, T)).astype(F32)
    u = P.DiffKVUnit(k[:T], v[:T], cs, n_high=10, n_low=T - 64 - 10, window=64, group=32)
    u.alpha_l = F32(0.0)
    r = np.random.default_rng(8)
    for t in range(20):
        _, _, dec = u.step(T + t, r.normal(size=(2, D)), k[T + t], v[T + t], 0.2)
        assert dec[1] != "pruned"
    assert u.pruned == []


# ---------------------------------------------------------------- MiKV

def test_mikv_by_hand():
    """Uniform attention keeps the order of scores; token 10 enters INT4 and
    pushes token 1 out of the top floor(11/5) = 2, which is demoted."""
    T, D = 12, 32
    k, v = _kv(T + 5, D, 9)
    cs = np.array([[10, 9, 8, 7, 6, 5, 4, 3, 2, 1, 20, 0.5]], F32)
    u = P.MiKVUnit(k[:T], v[:T], cs, nr=2, group=32)
    assert u.hi.ids() == [0, 1] and u.lo.ids() == list(range(2, 10))
    int4_1 = u.hi.dequant(1)
    q = np.zeros((1, D))
    entered, demoted = [], []
    for t in range(5):
        _, lse, e, d = u.step(T + t, q, k[T + t], v[T + t], 0.3)
        assert abs(lse[0] - math.log(T + t + 1)) < 1e-12       # nothing evicted
        entered.append(e)
        demoted.append(d)
    assert entered == [(10, "int4"), (11, "int2"), (12, "int2"), (13, "int2"), (14, "int2")]
    assert demoted == [[1], [], [], [], []]
    assert u.hi.ids() == [0, 10]
    assert sorted(u.hi.ids() + u.lo.ids() + [r[0] for r in u.res]) == list(range(T + 5))
    # cumulative score of token 0: 10 + 1/13 + 1/14 + 1/15 + 1/16 + 1/17
    want = 10 + sum(1.0 / n for n in range(13, 18))
    assert abs(float(u.cs[0]) - want) < 1e-5
    # demotion re-quantises the dequantised INT4 values: error <= s2/2
    k2, v2 = u.lo.dequant(1)
    kc, ks, kz, vc, vs, vz = u.lo.rows[1]
    for x4, x2, s2 in ((int4_1[0], k2, ks), (int4_1[1], v2, vs)):
        bound = np.repeat(s2.astype(np.float64), 32) * (0.5 + 2 ** -20) + np.spacing(np.abs(x4))
        assert np.all(np.abs(x2.astype(np.float64) - x4) <= bound)


def test_mikv_conservation_random():
    T, D = 200, 32
    k, v = _kv(T + 12, D, 10)
    r = np.random.default_rng(11)
    cs = r.random((4, T)).astype(F32)
    u = P.MiKVUnit(k[:T], v[:T], cs, nr=8, group=32)
    for t in range(12):
        u.step(T + t, r.normal(size=(4, D)), k[T + t], v[T + t], 0.2)
        nq = len(u.hi.rows) + len(u.lo.rows)
        assert len(u.hi.rows) <= nq // 5 and len(u.res) == 8
    assert sorted(u.hi.ids() + u.lo.ids() + [x[0] for x in u.res]) == list(range(T + 12))


# ---------------------------------------------------------------- accounting

def test_minikv_compression_closed_form():
    """0.33 GB vs 2.4 GB, 86% (LLaMA2-7B, prompt 4096, 512 generated, INT2, G = 16)."""
    mini = acc.minikv_cache_bytes(32, 4096, 4096, 512, 0.5, 2, 16)
    full = acc.full_cache_bytes(32, 4096, 4096, 512)
    assert round(mini / 1e9, 2) == 0.34 and round(mini / 2 ** 30, 2) == 0.31
    assert abs(mini / 1e9 - 0.33) < 0.01
    assert round(full / 1e9, 1) == 2.4
    assert round(100 * (1 - mini / full)) == 86


def test_tier_byte_closed_forms():
    assert acc.bits_per_scalar(2, 32) == 3.0
    assert acc.token_bytes(128, 2, 2, 32) == 96
    assert acc.token_bytes(128, 4, 4, 32) == 160
    assert acc.token_bytes(128, 8, 4, 32) == 224
    assert acc.token_bytes(128, 4, 2, 32) == 128
    assert acc.fp16_token_bytes(128) == 512
    assert (8 + 4) / 32 == 0.375 and (4 + 2) / 32 == 0.1875     # codes only, DiffKV tiers


def test_mikv_ties_go_to_the_lower_position():
    """Equal cumulative scores: the lower position stays INT4 whatever tier it sits in."""
    T, D = 12, 32
    k, v = _kv(T + 1, D, 12)
    # tokens 3 and 7 tie for the last INT4 place once token 10 (score 9) leaves the residual
    cs = np.array([[0, 0, 0, 5, 0, 0, 0, 5, 0, 0, 9, 0]], F32)
    u = P.MiKVUnit(k[:T], v[:T], cs, nr=2, group=32)
    assert u.hi.ids() == [3, 7]             # floor(10/5) = 2, tie 3 < 7 both in
    _, _, e, d = u.step(T, np.zeros((1, D)), k[T], v[T], 0.3)
    # population 11 -> 2 places: token 10 (9 + 1/13) and the lower of the tied 3 / 7
    assert e == (10, "int4") and d == [7]
    assert u.hi.ids() == [3, 10]


def test_mikv_gqa_group_is_summed():
    """Two query heads that disagree: the INT4 set and every cumulative score follow the
    SUM over the group (MiKV rebuttal, importance policy: H2O cumulative attention over
    the heads that read the KV head).  Head 0 alone would keep {0, 2}, the max over the
    heads {0, 1}; the sum keeps {0, 3}.  A zero query attends uniformly, so each decode
    step adds 1/N per head, 2/N for the group; a mean over the heads would add 1/N."""
    T, D = 12, 32
    k, v = _kv(T + 1, D, 13)
    cs = np.zeros((2, T), F32)
    cs[0, [0, 2, 3, 10]] = [6, 2, 1, 3]
    cs[1, [1, 3, 10]] = [4, 4, 2.5]
    acc = P.mikv_cumulative(cs)
    assert list(acc[:4]) == [6, 4, 2, 5] and acc[10] == F32(5.5)
    u = P.MiKVUnit(k[:T], v[:T], cs, nr=2, group=32)
    assert u.hi.ids() == [0, 3]                      # floor(10/5) = 2 places
    q = np.zeros((2, D))
    _, lse, e, d = u.step(T, q, k[T], v[T], 0.3)
    assert np.allclose(lse, math.log(T + 1), atol=1e-12)
    # population 11: 0 -> 6 + 2/13, 10 -> 5.5 + 2/13, 3 -> 5 + 2/13: token 10 enters, 3 leaves
    assert e == (10, "int4") and d == [3]
    assert u.hi.ids() == [0, 10]
    for j, base in ((0, 6.0), (1, 4.0), (3, 5.0), (10, 5.5), (5, 0.0), (12, 0.0)):
        assert abs(float(u.cs[j]) - (base + 2.0 / 13)) < 1e-6, f"token {j}"
