"""Comparison helpers shared by the parity tests (no method arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

# attention outputs at fp16/bf16: max-abs 2e-3 and relative 1e-2 per element
ATTN_ATOL, ATTN_RTOL = 2e-3, 1e-2
# cumulative scores: relative 1e-4 (plus a floor for values near zero)
SCORE_RTOL, SCORE_ATOL = 1e-4, 1e-7


def np_(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.float()
        return t.numpy()
    return np.asarray(t)


def u32(t):
    return np_(t).view(np.uint32)


def u16(t):
    a = np_(t)
    return a.view(np.uint16)


def assert_attn_close(gpu, ref, what=""):
    g = np_(gpu).astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    bad = err > ATTN_ATOL + ATTN_RTOL * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} elements outside tolerance, max abs err {err.max():.3e}"
    return float(err.max())


def assert_scores_close(gpu, ref, what=""):
    g = np_(gpu).astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    bad = err > SCORE_RTOL * np.abs(r) + SCORE_ATOL
    assert not bad.any(), (f"{what}: {bad.sum()} scores outside tolerance, max rel err "
                           f"{(err / np.maximum(np.abs(r), 1e-30)).max():.3e}")


def selection_agrees(gpu_sel, ref_sel, ref_scores, k, w):
    """True when identical; otherwise asserts the difference is a valid tie.

    A position may differ only if its (oracle) score lies within the score
    tolerance of the k-th largest candidate score, i.e. the two rankings
    differ by rounding at the boundary.
    """
    g, r = set(int(x) for x in gpu_sel), set(int(x) for x in ref_sel)
    if g == r:
        return True
    T = len(ref_scores)
    cand = np.asarray(ref_scores[: T - w], dtype=np.float64)
    bound = np.sort(cand)[::-1][k - 1]
    for j in g.symmetric_difference(r):
        assert j < T - w, f"window position {j} differs"
        assert abs(cand[j] - bound) <= SCORE_RTOL * abs(bound) + SCORE_ATOL, \
            f"position {j} (score {cand[j]}) differs far from the boundary {bound}"
    assert len(g) == len(r)
    return False


def gpu_tier_rows(tier, u):
    """{token id: (k codes, k scale, k zero, v codes, v scale, v zero)} of unit u of a
    per-token tier (fixed per-unit arrays or page pools), as uint32 / uint16 arrays."""
    rows = tier.rows_of(u).to(tier.token_id.device)
    c = len(rows)
    pick = lambda x: x.reshape(-1, *x.shape[2:]).index_select(0, rows)
    ids = pick(tier.token_id).cpu().numpy()
    kc, ks, kz = u32(pick(tier.k_codes)), u16(pick(tier.k_scale)), u16(pick(tier.k_zero))
    vc, vs, vz = u32(pick(tier.v_codes)), u16(pick(tier.v_scale)), u16(pick(tier.v_zero))
    return {int(ids[i]): (kc[i], ks[i], kz[i], vc[i], vs[i], vz[i]) for i in range(c)}


def oracle_tier_rows(tt):
    """Same view of an oracle TokenTier."""
    out = {}
    for tid, (kc, ks, kz, vc, vs, vz) in tt.rows.items():
        out[int(tid)] = (kc.view(np.uint32), ks.view(np.uint16), kz.view(np.uint16),
                         vc.view(np.uint32), vs.view(np.uint16), vz.view(np.uint16))
    return out


def assert_tiers_equal(gpu_rows, ref_rows, what=""):
    assert sorted(gpu_rows) == sorted(ref_rows), f"{what}: token sets differ"
    for tid, row in ref_rows.items():
        for a, b in zip(gpu_rows[tid], row):
            assert np.array_equal(a, b), f"{what}: token {tid} payload differs"
