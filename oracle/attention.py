"""Oracle: prefill attention (pass 1 and pass 2) and decode attention, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Prefill pass 1 (MiniKV review page, referee minor comment 2 on section 3.2,
and the verdict JSON ``key_machinery``): the attention output is the usual
FlashAttention-compatible softmax attention; here it is written out as its
definition, O_i = sum_{j<=i} softmax_j(sigma * q_i . k_j) v_j, with
sigma = 1/sqrt(D) and a causal mask (reading: the pages give neither; the
inputs are taken as already position-encoded).  The per-row log-sum-exp
lse_i = log sum_{j<=i} exp(sigma q_i . k_j) is returned with it.

Prefill pass 2 (same sources, "column-wise cumulative attention scores";
heavy-hitter assumption under "Assumptions & free parameters"; MiKV
rebuttal, answer on the importance policy: H2O cumulative attention):
colscore_j = sum_{i >= j} P_ij over every prompt query i.

Decode attention (MiKV rebuttal, section on the INTn x FP16 GEMV kernels;
MiniKV verdict JSON ``forward_implications``): the new query attends to every
cached token, each packed token through its dequantised value and the
residual tokens at full precision.  The oracle takes dequantised float32
tensors as input, so the result isolates the attention arithmetic from the
quantisation error.

Pins (tests/test_oracle_attention.py): a pure-Python triple loop on tiny
inputs, rows of P summing to 1, sum_j colscore_j = number of queries,
colscore_{T-1} = P_{T-1,T-1}, the closed form for a zero query (uniform
attention: O_i is the running mean of v and colscore_j = H_T - H_j with H
the harmonic numbers), permutation invariance of decode.  Observation-window
scores: w_obs = T gives the full column scores, w_obs = 1 the last query's
own attention row, and every window's scores sum to w_obs.
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


def _f64(x):
    return np.asarray(x).astype(F64)


def attention_matrix(q, k, sm_scale, causal=True):
    """P [Tq, Tk] for one head: row softmax of sigma * q k^T under the mask."""
    q = _f64(q)
    k = _f64(k)
    s = (q @ k.T) * F64(sm_scale)
    tq, tk = s.shape
    if causal:
        mask = np.arange(tk)[None, :] > np.arange(tq)[:, None]
        s = np.where(mask, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def prefill_head(q, k, v, sm_scale, causal=True):
    """One (batch, query head): returns (O [T, D] f64, lse [T] f64, colscore [T] f64)."""
    p, lse = attention_matrix(q, k, sm_scale, causal)
    o = p @ _f64(v)
    colscore = p.sum(axis=0)
    return o, lse, colscore


def prefill(q, k, v, sm_scale=None, causal=True):
    """Batched prefill over q [B, Hq, T, D], k/v [B, Hkv, T, D].

    Query head h reads KV head h // (Hq/Hkv).  Returns O, lse, colscore
    (float64, shapes [B,Hq,T,D], [B,Hq,T], [B,Hq,T]).
    """
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    o = np.zeros((B, Hq, T, D), F64)
    lse = np.zeros((B, Hq, T), F64)
    cs = np.zeros((B, Hq, T), F64)
    for b in range(B):
        for h in range(Hq):
            o[b, h], lse[b, h], cs[b, h] = prefill_head(q[b, h], k[b, h // g], v[b, h // g],
                                                        sm_scale, causal)
    return o, lse, cs


def prefill_rows(q, k, v, rows, sm_scale, causal=True):
    """O and lse of selected query rows of one head (each row is independent).

    Used where T is too large for the full matrix; returns (O [r, D], lse [r]).
    """
    rows = np.asarray(rows)
    qs = _f64(q)[rows]
    k = _f64(k)
    s = (qs @ k.T) * F64(sm_scale)
    if causal:
        s = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return (e / l) @ _f64(v), (m + np.log(l))[:, 0]


def lse_all_rows(q, k, sm_scale, causal=True, block=1024):
    """lse_i for every row of one head, one block of rows at a time."""
    T = q.shape[0]
    out = np.zeros(T, F64)
    k = _f64(k)
    for r0 in range(0, T, block):
        rows = np.arange(r0, min(T, r0 + block))
        s = (_f64(q[rows]) @ k.T) * F64(sm_scale)
        if causal:
            s = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        out[rows] = (m + np.log(np.exp(s - m).sum(axis=1, keepdims=True)))[:, 0]
    return out


def colscore_cols(q, k, cols, lse, sm_scale, causal=True):
    """colscore_j = sum_i exp(sigma q_i.k_j - lse_i) for selected key columns j."""
    cols = np.asarray(cols)
    s = (_f64(q) @ _f64(k)[cols].T) * F64(sm_scale)               # [T, c]
    p = np.exp(s - _f64(lse)[:, None])
    if causal:
        p = np.where(np.arange(q.shape[0])[:, None] < cols[None, :], 0.0, p)
    return p.sum(axis=0)


def window_colscore_head(q, k, sm_scale, w_obs, causal=True):
    """Column scores over an observation window (SnapKV-style selection; the MiniKV verdict
    JSON names SnapKV as a LongBench baseline without its mechanism, read as: keys scored
    by the attention of the last w_obs queries): colscore_j = sum over i >= T - w_obs of
    P_ij, P the full softmax of the prompt (rows keep their normalisation over all keys).
    One head: q, k [T, D]; returns [T] float64."""
    p, _ = attention_matrix(q, k, sm_scale, causal)
    T = p.shape[0]
    return p[T - w_obs:].sum(axis=0)


def decode_head(q, keys, values, sm_scale):
    """One query vector against N cached tokens: returns (o [D], lse, p [N]).

    ``keys``/``values`` are the dequantised (or full-precision) float tensors
    [N, D]; the order of tokens is irrelevant (permutation invariance).
    """
    s = (_f64(keys) @ _f64(q)) * F64(sm_scale)
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    p = e / l
    return p @ _f64(values), float(m + np.log(l)), p
