"""Pins of the oracle attention against textbook definitions and closed forms (no GPU)."""
import math

import numpy as np
import pytest

from oracle import attention as A


def _loops_attention(q, k, v, scale):
    """Textbook causal softmax attention written as plain Python loops."""
    T, D = len(q), len(q[0])
    out, lse = [], []
    for i in range(T):
        s = [scale * sum(q[i][c] * k[j][c] for c in range(D)) for j in range(i + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        l = sum(e)
        out.append([sum(e[j] / l * v[j][c] for j in range(i + 1)) for c in range(D)])
        lse.append(m + math.log(l))
    col = [0.0] * T
    for i in range(T):
        s = [scale * sum(q[i][c] * k[j][c] for c in range(D)) for j in range(i + 1)]
        for j in range(i + 1):
            col[j] += math.exp(s[j] - lse[i])
    return out, lse, col


def test_prefill_matches_python_loops():
    r = np.random.default_rng(0)
    T, D = 7, 5
    q, k, v = (r.normal(size=(T, D)) for _ in range(3))
    o, lse, cs = A.prefill_head(q, k, v, 0.37)
    o2, lse2, cs2 = _loops_attention(q.tolist(), k.tolist(), v.tolist(), 0.37)
    assert np.allclose(o, o2, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, lse2, rtol=1e-12, atol=1e-12)
    assert np.allclose(cs, cs2, rtol=1e-12, atol=1e-12)


def test_rows_sum_to_one_and_column_totals():
    r = np.random.default_rng(1)
    T, D = 96, 16
    q, k = r.normal(size=(T, D)), r.normal(size=(T, D)) * 3
    p, _ = A.attention_matrix(q, k, 1 / math.sqrt(D))
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(np.triu(p, 1) == 0)
    _, _, cs = A.prefill_head(q, k, r.normal(size=(T, D)), 1 / math.sqrt(D))
    assert abs(cs.sum() - T) <= 1e-9 * T
    assert cs[0] >= 1.0
    assert abs(cs[-1] - p[-1, -1]) < 1e-15


def test_zero_query_closed_form():
    """q = 0: every row attends uniformly, O_i = mean(v_0..v_i), colscore_j = H_T - H_j."""
    r = np.random.default_rng(2)
    T, D = 50, 8
    v = r.normal(size=(T, D))
    o, lse, cs = A.prefill_head(np.zeros((T, D)), r.normal(size=(T, D)), v, 0.125)
    run = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.allclose(o, run, atol=1e-13)
    assert np.allclose(lse, np.log(np.arange(1, T + 1)), atol=1e-13)
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, T + 1))])
    assert np.allclose(cs, H[T] - H[np.arange(T)], atol=1e-13)


def test_non_causal_total():
    r = np.random.default_rng(3)
    q, k, v = (r.normal(size=(20, 4)) for _ in range(3))
    _, _, cs = A.prefill_head(q, k, v, 0.5, causal=False)
    assert abs(cs.sum() - 20) < 1e-12


def test_gqa_head_mapping():
    """Query head h reads KV head h // g (a transposed mapping fails this)."""
    r = np.random.default_rng(4)
    B, Hq, Hkv, T, D = 1, 4, 2, 6, 3
    q = r.normal(size=(B, Hq, T, D))
    k = r.normal(size=(B, Hkv, T, D))
    v = r.normal(size=(B, Hkv, T, D))
    o, _, _ = A.prefill(q, k, v, 0.5)
    for h in range(Hq):
        o1, _, _ = A.prefill_head(q[0, h], k[0, h // 2], v[0, h // 2], 0.5)
        assert np.allclose(o[0, h], o1)
    o2, _, _ = A.prefill_head(q[0, 1], k[0, 1], v[0, 1], 0.5)
    assert not np.allclose(o[0, 1], o2)


def test_blocked_helpers_agree_with_full_matrix():
    r = np.random.default_rng(5)
    T, D = 300, 16
    q, k, v = (r.normal(size=(T, D)) for _ in range(3))
    o, lse, cs = A.prefill_head(q, k, v, 0.25)
    rows = np.array([0, 1, 17, 128, 299])
    o_r, lse_r = A.prefill_rows(q, k, v, rows, 0.25)
    assert np.allclose(o_r, o[rows], atol=1e-12)
    assert np.allclose(lse_r, lse[rows], atol=1e-12)
    assert np.allclose(A.lse_all_rows(q, k, 0.25, block=64), lse, atol=1e-12)
    cols = np.array([0, 5, 150, 299])
    assert np.allclose(A.colscore_cols(q, k, cols, lse, 0.25), cs[cols], atol=1e-12)


def test_decode_textbook_and_permutation():
    r = np.random.default_rng(6)
    N, D = 40, 8
    q, k, v = r.normal(size=D), r.normal(size=(N, D)), r.normal(size=(N, D))
    o, lse, p = A.decode_head(q, k, v, 0.3)
    s = [0.3 * float(np.dot(q, k[j])) for j in range(N)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    l = sum(e)
    o2 = [sum(e[j] / l * v[j][c] for j in range(N)) for c in range(D)]
    assert np.allclose(o, o2, atol=1e-13)
    assert abs(lse - (m + math.log(l))) < 1e-13
    perm = r.permutation(N)
    o3, lse3, p3 = A.decode_head(q, k[perm], v[perm], 0.3)
    assert np.allclose(o3, o, atol=1e-14) and abs(lse3 - lse) < 1e-14
    assert np.allclose(p3, p[perm])
    o4, lse4, _ = A.decode_head(np.zeros(D), k, v, 0.3)
    assert np.allclose(o4, v.mean(axis=0)) and abs(lse4 - math.log(N)) < 1e-13


def test_window_scores_pins():
    """Observation-window column scores: the last w queries only.  Brute force by loops for
    every window on tiny inputs (from the textbook loops' lse), w = T reduces to the full
    column scores, and every window sums to w."""
    r = np.random.default_rng(5)
    T, D = 9, 4
    q, k, v = (r.normal(size=(T, D)) for _ in range(3))
    _, lse, _ = _loops_attention(q.tolist(), k.tolist(), v.tolist(), 0.41)
    for w in range(1, T + 1):
        ref = [0.0] * T
        for i in range(T - w, T):
            for j in range(i + 1):
                ref[j] += math.exp(0.41 * sum(q[i][c] * k[j][c] for c in range(D)) - lse[i])
        got = A.window_colscore_head(q, k, 0.41, w)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14), w
        assert abs(got.sum() - w) < 1e-12
    _, _, cs = A.prefill_head(q, k, v, 0.41)
    assert np.allclose(A.window_colscore_head(q, k, 0.41, T), cs, rtol=0, atol=1e-14)


def test_window_scores_zero_query_closed_form():
    """q = 0: colscore_j = H_T - H_max(j, T-w) (uniform rows over the window)."""
    r = np.random.default_rng(6)
    T, D = 40, 8
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, T + 1))])
    for w in (1, 7, 40):
        got = A.window_colscore_head(np.zeros((T, D)), r.normal(size=(T, D)), 0.125, w)
        ref = H[T] - H[np.maximum(np.arange(T), T - w)]
        assert np.allclose(got, ref, atol=1e-13), w
