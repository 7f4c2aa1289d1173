"""prefill_attn_scores (tcgen05 two-pass kernel) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import attention as OA
from tests.helpers import assert_attn_close, assert_scores_close, np_

pytestmark = pytest.mark.gpu


def _run(B, Hq, Hkv, T, dtype=torch.float16, seed=0, outlier_scale=10.0, n_out=3, D=128):
    x = inputs.make_qkv(B, Hq, Hkv, T, D, dtype=dtype, seed=seed,
                        outliers=inputs.outlier_channels(Hkv, D, n_out, seed),
                        outlier_scale=outlier_scale)
    scale = 1.0 / math.sqrt(D)
    o, lse, cs = kvq.prefill_attn_scores(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    return x, scale, o, lse, cs


@pytest.mark.parametrize("B,Hq,Hkv,T,dtype", [
    (1, 2, 2, 256, torch.float16),       # two full tiles
    (2, 4, 2, 300, torch.float16),       # GQA, ragged tail of 44 rows
    (1, 4, 1, 200, torch.bfloat16),      # bf16, g = 4
    (1, 1, 1, 1, torch.float16),         # a single token
    (1, 5, 1, 129, torch.float16),       # g = 5, one row past a tile
])
def test_prefill_matches_oracle(B, Hq, Hkv, T, dtype):
    _check_all(*_run(B, Hq, Hkv, T, dtype), T)


@pytest.mark.parametrize("B,Hq,Hkv,T", [(1, 2, 2, 256), (1, 4, 2, 300)])
def test_prefill_head_dim_64(B, Hq, Hkv, T):
    """Head dim 64 (the tiny workload's) on both passes, ragged tail included."""
    _check_all(*_run(B, Hq, Hkv, T, D=64, n_out=2, outlier_scale=8.0), T)


def _check_all(x, scale, o, lse, cs, T):
    oo, ol, oc = OA.prefill(np_(x.q), np_(x.k), np_(x.v), scale)
    assert_attn_close(o, oo, "O")
    assert np.allclose(np_(lse), ol, atol=1e-4, rtol=1e-5), "lse"
    assert_scores_close(cs, oc, "colscore")
    # the column scores of each head add up to the number of queries
    assert np.allclose(np_(cs).sum(axis=-1), T, rtol=1e-5)


def test_prefill_4096_sampled():
    """The 32-head, 4096-token LLaMA2-7B-shaped layer: two heads checked in full."""
    B, H, T, D = 1, 32, 4096, 128
    x, scale, o, lse, cs = _run(B, H, H, T)
    for h in (0, 31):
        oo, ol, oc = OA.prefill_head(np_(x.q[0, h]), np_(x.k[0, h]), np_(x.v[0, h]), scale)
        assert_attn_close(o[0, h], oo, f"O head {h}")
        assert_scores_close(cs[0, h], oc, f"colscore head {h}")
    assert np.allclose(np_(cs).sum(axis=-1), T, rtol=1e-4)


def test_prefill_large_scores():
    """Outlier channels x40 push row maxima far apart (exercises the rescale path)."""
    x, scale, o, lse, cs = _run(1, 2, 2, 512, outlier_scale=40.0, n_out=6)
    oo, ol, oc = OA.prefill(np_(x.q), np_(x.k), np_(x.v), scale)
    assert_attn_close(o, oo, "O")
    assert_scores_close(cs, oc, "colscore")


@pytest.mark.parametrize("B,Hq,Hkv,T,w_obs,dtype,D", [
    (1, 2, 2, 300, 1, torch.float16, 128),      # the last query's own row
    (2, 4, 2, 300, 32, torch.float16, 128),     # inside the last (ragged) tile
    (1, 4, 1, 512, 200, torch.bfloat16, 128),   # a window start inside a middle tile, bf16, g = 4
    (1, 2, 2, 256, 256, torch.float16, 128),    # the whole prompt: the full column scores
    (1, 2, 2, 512, 128, torch.float16, 128),    # a window starting exactly on a tile boundary
    (1, 2, 2, 256, 100, torch.float16, 64),     # head dim 64
    (1, 2, 2, 4096, 1024, torch.float16, 128),  # the LLaMA-layer prompt: many key tiles skip ahead
])
def test_window_scores_match_oracle(B, Hq, Hkv, T, w_obs, dtype, D):
    """Observation-window column scores (pass 2 over the last w_obs queries) against the
    float64 definition, with the same tolerance as the full column scores."""
    x, scale, o, lse, cs = _run(B, Hq, Hkv, T, dtype, D=D)
    ws = kvq.prefill_window_scores(x.q.cuda(), x.k.cuda(), lse, w_obs, scale)
    torch.cuda.synchronize()
    assert kvq.device_status() == 0
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            ref = OA.window_colscore_head(np_(x.q[b, h]), np_(x.k[b, h // g]), scale, w_obs)
            assert_scores_close(ws[b, h], ref, f"window scores {b},{h}")
            assert abs(float(ws[b, h].double().sum()) - w_obs) <= 1e-4 * w_obs
