"""Failure detection on the GPU without a fault: a decode launch whose first staged copy
is withheld (a barrier that nothing completes) runs out of its bounded waits, reports
KVQ_ETIMEOUT through the status word, leaves no copy in flight, and the launches after it
are correct again, with the cache state still in step with the oracle."""
import math

import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import policies as OP
from oracle import select as OS
from tests.helpers import assert_attn_close, np_

pytestmark = pytest.mark.gpu


def test_withheld_copy_times_out_and_the_context_survives():
    B, H, T, D, G, nr = 1, 2, 256, 128, 32, 0
    scale = 1.0 / math.sqrt(D)
    x = inputs.make_qkv(B, H, H, T, D, seed=11, device="cuda")
    k_hh, w = OS.budget(T, 25, 25)
    n_sel = k_hh + w
    cs = inputs.random_scores(B, H, T, seed=12)
    idx, _ = kvq.select_tokens(cs.cuda(), torch.full((B * H,), k_hh, dtype=torch.int32, device="cuda"), w)
    cap = ((n_sel + 8) // G + 1) * G
    cache = kvq.make_cache(B, H, H, D, G, torch.float16, kvq.POLICY_MINIKV,
                           [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr)
    kvq.requant_demote(cache, 0, k_src=x.k, v_src=x.v, sel_idx=idx, n_sel=n_sel)
    units = [OP.MiniKVUnit(np_(x.k[0, h]), np_(x.v[0, h]), OS.select_unit(np_(cs[0, h]), k_hh, w), nr, G)
             for h in range(H)]
    assert kvq.device_status() == 0
    for t in range(4):
        qd, kd, vd = inputs.make_decode_step(B, H, H, D, t, seed=11, device="cuda")
        kvq.debug_withhold_copy(t == 1)
        try:
            od, _ = kvq.decode_attn_qkv(qd, kd, vd, cache, scale)
            st = kvq.device_status()
        finally:
            kvq.debug_withhold_copy(False)
        for h in range(H):
            ro, _ = units[h].step(T + t, np_(qd[0, h:h + 1]), np_(kd[0, h]), np_(vd[0, h]), scale)
            if t == 1 and h == 0:
                continue                       # the unit whose copy was withheld: output undefined
            assert_attn_close(od[0, h], ro[0], f"step {t} head {h}")
        assert st == (kvq.KVQ_ETIMEOUT if t == 1 else 0), f"step {t}: status {st}"
