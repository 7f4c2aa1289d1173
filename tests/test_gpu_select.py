"""select_tokens on the GPU: bit-exact with the oracle on identical float32 scores."""
import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import select as OS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,T,ties", [(1, 2, 256, 0), (2, 3, 1500, 8), (1, 4, 4096, 0),
                                         (2, 2, 3000, 3), (1, 1, 1, 0), (1, 2, 16384, 50)])
def test_select_bit_exact(B, H, T, ties):
    s = inputs.random_scores(B, H, T, seed=T + ties, ties=ties)
    r = np.random.default_rng(T)
    for w in sorted({0, T // 4, T}):
        ks = r.integers(0, T + 1, size=B * H).astype(np.int32)
        ks[0] = min(T, T // 4)
        idx, n = kvq.select_tokens(s.cuda(), torch.from_numpy(ks).cuda(), w, kmax=T)
        idx, n = idx.cpu().numpy(), n.cpu().numpy()
        for u in range(B * H):
            ref = OS.select_unit(s.view(B * H, T)[u].numpy(), int(ks[u]), w)
            assert n[u] == len(ref)
            assert np.array_equal(idx.reshape(B * H, -1)[u, :n[u]], ref), (u, w)
    assert kvq.device_status() == 0


def test_select_pyramid_layer_budgets():
    """Per-layer budgets of the 40% -> 10% schedule at T = 16384 with a 25% window."""
    T, L = 16384, 32
    s = inputs.random_scores(1, L, T, seed=5)
    ks = np.array([OS.pyramid_hh_budget(T, l, L) for l in range(L)], np.int32)
    k_, w = OS.budget(T, 0, 25)
    idx, n = kvq.select_tokens(s.cuda(), torch.from_numpy(ks).cuda(), w, kmax=int(ks.max()))
    idx, n = idx.cpu().numpy(), n.cpu().numpy()
    for l in range(L):
        ref = OS.select_unit(s[0, l].numpy(), int(ks[l]), w)
        assert np.array_equal(idx[0, l, :n[l]], ref)


def test_gqa_score_reduce():
    from oracle import policies as OP
    B, Hq, Hkv, T = 2, 8, 2, 300
    cs = inputs.random_scores(B, Hq, T, seed=9)
    got_sum = kvq.kvq_score_reduce(cs.cuda(), Hkv, 0).cpu().numpy()
    got_mm = kvq.kvq_score_reduce(cs.cuda(), Hkv, 1).cpu().numpy()
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            blk = cs[b, h * g:(h + 1) * g].numpy()
            assert np.array_equal(got_sum[b, h], OP.mikv_cumulative(blk))
            assert np.array_equal(got_mm[b, h], OP.diffkv_significance(blk, T))
