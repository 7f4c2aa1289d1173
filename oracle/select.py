"""Oracle: token budgets and heavy-hitter + recent-window selection.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

MiniKV review page, "Assumptions & free parameters": the cache keeps heavy
hitters (tokens with the largest cumulative attention score, chosen once at
the end of prefill) plus a recent window; the default budget is 25% heavy
hitters + 25% recent window; the pyramid variant lets the heavy-hitter budget
fall linearly with depth.  Figure 2 caption: heavy hitters alone or the
window alone collapse on some tasks, so both are always kept.

Readings taken:

* budgets are integers: w = floor(T * rw% / 100), k = floor(T * hh% / 100),
  then k is clamped to the T - w tokens outside the window;
* the pyramid schedule is the linear 40% -> 10% schedule of the 32-layer
  sweep workload, in the exact integer form
  k_l = floor(T * (hi*(L-1) - (hi-lo)*l) / (100*(L-1)));  the page's "pyramid
  depth d = 7" is left undefined by the pages and is not used;
* heavy hitters are the k largest scores among positions j < T - w, ordered
  by (score descending, position ascending), so equal scores go to the lower
  position; the output lists the chosen positions in ascending order.

Pins (tests/test_oracle_select.py): a full sort on every unit (brute force),
hh = 0 gives the window only, a 100% budget gives every position, ties
resolve to the lower index (tests/golden/select_ties.txt), the pyramid
end points 6553 and 1638 at T = 16384.
"""
from __future__ import annotations

import numpy as np


def budget(T, hh_pct, rw_pct):
    """(k, w) from percentages of the prompt length, clamped so k <= T - w."""
    w = (T * rw_pct) // 100
    w = min(w, T)
    k = (T * hh_pct) // 100
    return min(k, T - w), w


def pyramid_hh_budget(T, layer, n_layers, hi_pct=40, lo_pct=10):
    """Heavy-hitter budget of ``layer`` under the linear hi% -> lo% schedule."""
    if n_layers == 1:
        return (T * hi_pct) // 100
    num = T * (hi_pct * (n_layers - 1) - (hi_pct - lo_pct) * layer)
    return num // (100 * (n_layers - 1))


def topk_order(score, candidates):
    """Candidate positions sorted by (score descending, position ascending)."""
    candidates = np.asarray(candidates, dtype=np.int64)
    s = np.asarray(score)[candidates]
    order = np.lexsort((candidates, -s.astype(np.float64)))
    return candidates[order]


def select_unit(score, k, w):
    """Selected positions of one unit, ascending: top-k heavy hitters + last w."""
    T = len(score)
    k = min(k, T - w)
    hh = topk_order(score, np.arange(T - w))[:k]
    return np.concatenate([np.sort(hh), np.arange(T - w, T)]).astype(np.int32)


def select_tokens(score, k_per_unit, w):
    """score [B, H, T] float32, k_per_unit [B*H] -> list of index arrays per unit."""
    B, H, T = score.shape
    out = []
    for b in range(B):
        for h in range(H):
            out.append(select_unit(score[b, h], int(k_per_unit[b * H + h]), w))
    return out
