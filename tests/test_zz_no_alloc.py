"""decode_attn_qkv_static: the decode entry point for callers that cannot give the
library scratch memory (an engine whose allocator already owns all free device
memory, or C code without a device allocator).  It must produce what
decode_attn_qkv produces with a caller workspace, call after call.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from tests.helpers import ATTN_ATOL, ATTN_RTOL, np_

pytestmark = pytest.mark.gpu


def _cache(k, v, idx, n_sel, B, H, D, nr, cap):
    c = kvq.make_cache(B, H, H, D, 32, torch.float16, kvq.POLICY_MINIKV,
                       [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr)
    kvq.requant_demote(c, 0, k_src=k, v_src=v, sel_idx=idx, n_sel=n_sel)
    return c


def test_static_scratch_matches_caller_workspace():
    B, H, T, D, nr = 1, 4, 512, 128, 32
    x = inputs.make_qkv(B, H, H, T, D, seed=21, outliers=inputs.outlier_channels(H, D, 2, 21),
                        outlier_scale=8.0)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    scale = 1.0 / math.sqrt(D)
    _, _, cs = kvq.prefill_attn_scores(q, k, v, scale)
    k_hh, w = T // 4, T // 4
    idx, _ = kvq.select_tokens(cs, torch.full((B * H,), k_hh, dtype=torch.int32, device="cuda"), w)
    cap = 512
    with_ws = _cache(k, v, idx, k_hh + w, B, H, D, nr, cap)
    no_ws = _cache(k, v, idx, k_hh + w, B, H, D, nr, cap)
    need = kvq.lib().kvq_decode_workspace_bytes(ctypes.byref(no_ws.desc))
    assert need <= kvq.STATIC_SCRATCH_BYTES
    for t in range(2):                                   # two calls in a row
        qd, kd, vd = inputs.make_decode_step(B, H, H, D, t, seed=21)
        qd, kd, vd = qd.cuda(), kd.cuda(), vd.cuda()
        o_ref, l_ref = kvq.decode_attn_qkv(qd, kd, vd, with_ws, scale)
        o_st, l_st = kvq.decode_attn_qkv_static(qd, kd, vd, no_ws, scale)
        kvq.requant_demote(with_ws, t + 1)
        kvq.requant_demote(no_ws, t + 1)
        torch.cuda.synchronize()
        a, b = np_(o_st).astype(np.float64), np_(o_ref).astype(np.float64)
        assert np.all(np.abs(a - b) <= ATTN_ATOL + ATTN_RTOL * np.abs(b)), f"call {t}"
        assert np.allclose(np_(l_st), np_(l_ref), atol=1e-5)
    assert kvq.device_status() == 0
    assert torch.equal(with_ws.res_len, no_ws.res_len)
    assert torch.equal(with_ws.seq_len, no_ws.seq_len)


def test_static_scratch_rejects_a_cache_too_large():
    """A cache needing more scratch than is built in is refused before any launch."""
    B, Hq, Hkv, D = 1, 8, 1, 128
    slots = kvq.STATIC_SCRATCH_BYTES // (4 * Hq) + 4096      # per-token logits outgrow the array
    c = kvq.make_cache(B, Hq, Hkv, D, 32, torch.float16, kvq.POLICY_MIKV,
                       [kvq.TierSpec(4, 4, kvq.AXIS_TOKEN, 64), kvq.TierSpec(2, 2, kvq.AXIS_TOKEN, slots)],
                       nr=16, score_cap=64)
    need = kvq.lib().kvq_decode_workspace_bytes(ctypes.byref(c.desc))
    assert need > kvq.STATIC_SCRATCH_BYTES
    q = torch.zeros((B, Hq, D), dtype=torch.float16, device="cuda")
    kn = torch.zeros((B, Hkv, D), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attn_qkv_static(q, kn, kn, c, 0.1)
    assert e.value.status == kvq.KVQ_EWORKSPACE
    assert kvq.device_status() == 0
