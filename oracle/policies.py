"""Oracle: the three cache life cycles (MiniKV, DiffKV, MiKV), one unit at a time.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A unit is one (batch element, KV head).  Every cached token carries its
position as token id.  A decode step with new position p first appends the
new key/value at full precision (the new token attends to itself), then runs
attention over every cached token, then applies the policy tail.  Attention
probabilities p_hj enter the score arrays rounded to float32, and every
score decision below is taken in float32 (the precision of the GPU path),
so that identical float32 score inputs give identical decisions.

MiniKV (review page "Assumptions & free parameters"; verdict JSON
``key_machinery``): the selected prompt tokens are packed once; per-channel
key groups need G consecutive tokens, so the last
r0 = nr + ((n_sel - nr) mod G) selected tokens (all of them if n_sel <= nr)
stay at full precision in the residual; when the residual reaches nr + G
tokens after a step, its G oldest tokens are packed and appended
(reading of "steps before newly generated KV states are quantized").

DiffKV (verdict JSON ``pith_extraction.key_machinery``; referee major
comment 2 and the Algorithm 1 comments): significance of a token = the mean
attention it received (sum over queries / number of queries that saw it),
max over the query heads of the GQA group.  Readings: at prefill end the
candidates are positions j < T - W; the top n_high by significance go to
K8V4, the next n_low to K4V2, the rest are pruned; alpha_h = T * score of the
last high token, alpha_l = T * score of the last low token (+inf / alpha_h
when a band is empty).  Each step the oldest window token leaves and goes to
K8V4 if score >= alpha_h / N, else K4V2 if score >= alpha_l / N, else it is
pruned, with N the sequence length after the step.  Tier formats: per-token
groups of G channels for keys and values.

MiKV (rebuttal: re-quantisation paragraph, "Q1" on long contexts, the
regrouping paragraph of the kernel answer): every token is kept; the top 20%
by cumulative attention (sum over the GQA group of H2O column scores, plus
the attention each decode step adds) are INT4, the rest INT2, keys and
values both per-token.  Readings: the last nr tokens stay at full precision;
each step the oldest residual token leaves, the top floor(N_q/5) set over the
quantised tokens plus the leaving one is recomputed (ties to the lower
position); the leaving token enters INT4 if it is in the set, else INT2;
every INT4 token outside the set is dequantised and re-quantised to INT2
from its dequantised values; no token is ever promoted.

Pins (tests/test_oracle_policies.py): token conservation (MiKV) and the
partition window / high / low / pruned (DiffKV), alpha_l = 0 prunes nothing,
a 100% budget with every tier empty reduces decode to textbook attention,
demotion error <= s_2/2 against the dequantised INT4 value, the byte closed
forms (oracle.accounting).
"""
from __future__ import annotations

import numpy as np

from . import quant
from .attention import decode_head
from .select import topk_order

F32 = np.float32


def _f32(x):
    return np.asarray(x).astype(F32)


def topk_by_id(scores, ids):
    """Token ids sorted by (score descending, id ascending)."""
    ids = np.asarray(ids, dtype=np.int64)
    order = np.lexsort((ids, -np.asarray(scores).astype(np.float64)))
    return ids[order]


# ---------------------------------------------------------------------------
# Packed token store with per-token groups (DiffKV and MiKV tiers)
# ---------------------------------------------------------------------------

class TokenTier:
    """Tokens quantised with per-token groups for both keys and values."""

    def __init__(self, k_bits, v_bits, group, d):
        self.k_bits, self.v_bits, self.group, self.d = k_bits, v_bits, group, d
        self.rows = {}   # token id -> (kc, ks, kz, vc, vs, vz)
        self._deq = {}   # token id -> (the row it was computed from, k, v): a memo only

    def add_raw(self, tid, k, v):
        kc, ks, kz = quant.quant_pack_token(_f32(k)[None], self.k_bits, self.group)
        vc, vs, vz = quant.quant_pack_token(_f32(v)[None], self.v_bits, self.group)
        self.rows[int(tid)] = (kc[0], ks[0], kz[0], vc[0], vs[0], vz[0])

    def dequant(self, tid):
        row = self.rows[int(tid)]
        memo = self._deq.get(int(tid))
        if memo is not None and memo[0] is row:          # same stored row: same values
            return memo[1], memo[2]
        kc, ks, kz, vc, vs, vz = row
        k = quant.unpack_token(kc[None], ks[None], kz[None], self.k_bits, self.group)[0]
        v = quant.unpack_token(vc[None], vs[None], vz[None], self.v_bits, self.group)[0]
        self._deq[int(tid)] = (row, k, v)
        return k, v

    def ids(self):
        return sorted(self.rows)


# ---------------------------------------------------------------------------
# MiniKV
# ---------------------------------------------------------------------------

class MiniKVUnit:
    """Persistent selection, per-channel INT-b keys, per-token INT-b values, residual."""

    def __init__(self, k, v, sel, nr, group, k_bits=2, v_bits=2):
        sel = np.asarray(sel)
        n = len(sel)
        r0 = n if n <= nr else nr + (n - nr) % group
        npk = n - r0
        self.nr, self.group, self.k_bits, self.v_bits = nr, group, k_bits, v_bits
        self.d = k.shape[1]
        ks = _f32(k)[sel[:npk]]
        vs = _f32(v)[sel[:npk]]
        self.ids = [int(t) for t in sel[:npk]]
        if npk:
            self.kw, self.ksc, self.kze = quant.quant_pack_channel(ks, k_bits, group)
            self.vw, self.vsc, self.vze = quant.quant_pack_token(vs, v_bits, group)
        else:
            d = self.d
            self.kw = np.zeros((0, d), np.uint32)
            self.ksc = np.zeros((0, d), np.float16)
            self.kze = np.zeros((0, d), np.float16)
            self.vw = np.zeros((0, d * v_bits // 32), np.uint32)
            self.vsc = np.zeros((0, d // group), np.float16)
            self.vze = np.zeros((0, d // group), np.float16)
        self.res = [(int(t), _f32(k)[t], _f32(v)[t]) for t in sel[npk:]]
        self._refresh()

    def _refresh(self):
        if len(self.ids):
            self.kh = quant.unpack_channel(self.kw, self.ksc, self.kze, self.k_bits, self.group)
            self.vh = quant.unpack_token(self.vw, self.vsc, self.vze, self.v_bits, self.group)
        else:
            self.kh = np.zeros((0, self.d), F32)
            self.vh = np.zeros((0, self.d), F32)

    def keys_values(self):
        rk = np.array([r[1] for r in self.res], F32).reshape(-1, self.d)
        rv = np.array([r[2] for r in self.res], F32).reshape(-1, self.d)
        ids = list(self.ids) + [r[0] for r in self.res]
        return ids, np.concatenate([self.kh, rk]), np.concatenate([self.vh, rv])

    def step(self, pos, qs, k_new, v_new, sm_scale):
        """qs [g, D]; returns (o [g, D], lse [g])."""
        self.res.append((int(pos), _f32(k_new), _f32(v_new)))
        _, kk, vv = self.keys_values()
        outs = [decode_head(q, kk, vv, sm_scale) for q in qs]
        if len(self.res) == self.nr + self.group:
            old = self.res[:self.group]
            self.res = self.res[self.group:]
            kw, ksc, kze = quant.quant_pack_channel(np.array([r[1] for r in old], F32),
                                                    self.k_bits, self.group)
            vw, vsc, vze = quant.quant_pack_token(np.array([r[2] for r in old], F32),
                                                  self.v_bits, self.group)
            self.kw = np.concatenate([self.kw, kw])
            self.ksc = np.concatenate([self.ksc, ksc])
            self.kze = np.concatenate([self.kze, kze])
            self.vw = np.concatenate([self.vw, vw])
            self.vsc = np.concatenate([self.vsc, vsc])
            self.vze = np.concatenate([self.vze, vze])
            self.ids += [r[0] for r in old]
            self._refresh()
        return np.array([o[0] for o in outs]), np.array([o[1] for o in outs])


# ---------------------------------------------------------------------------
# DiffKV
# ---------------------------------------------------------------------------

def diffkv_significance(colscore, T):
    """colscore [g, T] float32 -> float32 [T]: max over heads of colscore_hj / (T - j)."""
    cs = _f32(colscore)
    cnt = (F32(T) - np.arange(T).astype(F32)).astype(F32)
    return (cs / cnt[None, :]).astype(F32).max(axis=0)


class DiffKVUnit:
    def __init__(self, k, v, colscore, n_high, n_low, window, group, high_bits=(8, 4), low_bits=(4, 2)):
        """high_bits / low_bits: (key bits, value bits) of the two tiers; K8V4 / K4V2 as the
        DiffKV pages give them, other pairs for the codec variants (the K4V8 mirror the
        DiffKV verdict JSON lists among its negative results)."""
        T, d = k.shape
        self.W, self.group, self.d = window, group, d
        self.high = TokenTier(high_bits[0], high_bits[1], group, d)
        self.low = TokenTier(low_bits[0], low_bits[1], group, d)
        self.pruned = []
        nc = T - window
        sig = diffkv_significance(colscore, T)
        order = topk_order(sig, np.arange(nc))
        n_high = min(n_high, nc)
        n_low = min(n_low, nc - n_high)
        hi, lo, pr = order[:n_high], order[n_high:n_high + n_low], order[n_high + n_low:]
        self.alpha_h = F32(T) * sig[hi[-1]] if n_high else F32(np.inf)
        self.alpha_l = F32(T) * sig[lo[-1]] if n_low else self.alpha_h
        self.alpha_h, self.alpha_l = F32(self.alpha_h), F32(self.alpha_l)
        kf, vf = _f32(k), _f32(v)
        for t in hi:
            self.high.add_raw(t, kf[t], vf[t])
        for t in lo:
            self.low.add_raw(t, kf[t], vf[t])
        self.pruned = sorted(int(t) for t in pr)
        cs = _f32(colscore)
        # window entries: [token id, k, v, acc per head]
        self.win = [[j, kf[j], vf[j], cs[:, j].copy()] for j in range(nc, T)]

    def attend(self, pos, qs, k_new, v_new, sm_scale):
        """Append the new token to the window, attend, add the attention to the window sums."""
        g = qs.shape[0]
        self.win.append([int(pos), _f32(k_new), _f32(v_new), np.zeros(g, F32)])
        ids, kk, vv = [], [], []
        for tier in (self.high, self.low):
            for t in tier.ids():
                kh, vh = tier.dequant(t)
                ids.append(t)
                kk.append(kh)
                vv.append(vh)
        nq = len(ids)
        for w in self.win:
            ids.append(w[0])
            kk.append(w[1])
            vv.append(w[2])
        kk = np.array(kk, F32)
        vv = np.array(vv, F32)
        outs = [decode_head(q, kk, vv, sm_scale) for q in qs]
        for h in range(g):
            p = outs[h][2]
            for i, w in enumerate(self.win):
                w[3][h] = F32(w[3][h] + F32(p[nq + i]))
        return np.array([o[0] for o in outs]), np.array([o[1] for o in outs])

    def tail(self, N):
        """The oldest window token leaves (if the window overflows); N = sequence length."""
        if len(self.win) <= self.W:
            return None
        tc, kc, vc, acc = self.win.pop(0)
        score = (acc / F32(N - tc)).astype(F32).max()
        th_h = F32(self.alpha_h / F32(N))
        th_l = F32(self.alpha_l / F32(N))
        if score >= th_h:
            self.high.add_raw(tc, kc, vc)
            return (tc, "high")
        if score >= th_l:
            self.low.add_raw(tc, kc, vc)
            return (tc, "low")
        self.pruned.append(tc)
        return (tc, "pruned")

    def step(self, pos, qs, k_new, v_new, sm_scale):
        o, lse = self.attend(pos, qs, k_new, v_new, sm_scale)
        return o, lse, self.tail(pos + 1)


# ---------------------------------------------------------------------------
# MiKV
# ---------------------------------------------------------------------------

def mikv_cumulative(colscore):
    """colscore [g, T] float32 -> float32 [T]: sum over the GQA group in head order."""
    cs = _f32(colscore)
    acc = np.zeros(cs.shape[1], F32)
    for h in range(cs.shape[0]):
        acc = (acc + cs[h]).astype(F32)
    return acc


class MiKVUnit:
    def __init__(self, k, v, colscore, nr, group, hi_frac_den=5):
        T, d = k.shape
        self.nr, self.group, self.d, self.den = nr, group, d, hi_frac_den
        self.hi = TokenTier(4, 4, group, d)
        self.lo = TokenTier(2, 2, group, d)
        self.cs = {}
        acc = mikv_cumulative(colscore)
        for j in range(T):
            self.cs[j] = F32(acc[j])
        nq = max(T - nr, 0)
        kf, vf = _f32(k), _f32(v)
        order = topk_order(acc, np.arange(nq))
        n4 = nq // self.den
        for t in order[:n4]:
            self.hi.add_raw(t, kf[t], vf[t])
        for t in order[n4:]:
            self.lo.add_raw(t, kf[t], vf[t])
        self.res = [(j, kf[j], vf[j]) for j in range(nq, T)]
        self.demoted = []

    def attend(self, pos, qs, k_new, v_new, sm_scale):
        """Append the new token, attend, add this step's attention to every cumulative score."""
        g = qs.shape[0]
        self.res.append((int(pos), _f32(k_new), _f32(v_new)))
        self.cs[int(pos)] = F32(0)
        ids, kk, vv = [], [], []
        for tier in (self.hi, self.lo):
            for t in tier.ids():
                kh, vh = tier.dequant(t)
                ids.append(t)
                kk.append(kh)
                vv.append(vh)
        for r in self.res:
            ids.append(r[0])
            kk.append(r[1])
            vv.append(r[2])
        kk = np.array(kk, F32)
        vv = np.array(vv, F32)
        outs = [decode_head(q, kk, vv, sm_scale) for q in qs]
        contrib = np.zeros(len(ids), F32)
        for h in range(g):
            contrib = (contrib + outs[h][2].astype(F32)).astype(F32)
        for i, t in enumerate(ids):
            self.cs[t] = F32(self.cs[t] + contrib[i])
        return np.array([o[0] for o in outs]), np.array([o[1] for o in outs])

    def tail(self):
        """Residual exit, re-ranking and demotion; returns (entered, demoted)."""
        demoted = []
        entered = None
        if len(self.res) > self.nr:
            e, ke, ve = self.res.pop(0)
            pop = self.hi.ids() + self.lo.ids() + [e]
            sc = np.array([self.cs[t] for t in pop], F32)
            order = topk_by_id(sc, np.array(pop))
            top = set(int(t) for t in order[:len(pop) // self.den])
            if e in top:
                self.hi.add_raw(e, ke, ve)
                entered = (e, "int4")
            else:
                self.lo.add_raw(e, ke, ve)
                entered = (e, "int2")
            for t in self.hi.ids():
                if t not in top:
                    kh, vh = self.hi.dequant(t)
                    del self.hi.rows[t]
                    self.lo.add_raw(t, kh, vh)
                    demoted.append(t)
        self.demoted.append(demoted)
        return entered, demoted

    def step(self, pos, qs, k_new, v_new, sm_scale):
        o, lse = self.attend(pos, qs, k_new, v_new, sm_scale)
        entered, demoted = self.tail()
        return o, lse, entered, demoted
