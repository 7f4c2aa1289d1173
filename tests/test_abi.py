"""The C ABI library builds, loads and exports every symbol include/kvq.h declares;
host-side validation rejects bad arguments before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_mixed_precision_gb300 import build, kvq
    build.build()
    return kvq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^(?:kvq_status|size_t|int|const char\*)\s+(\w+)\s*\(", src, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["kv_quant_pack", "prefill_attn_scores", "select_tokens", "requant_demote",
              "decode_attn_qkv"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_struct_layout_matches_header(tmp_path):
    """The binding's ctypes structs have the header's sizes and field offsets (compiled with
    the host C compiler from include/kvq.h)."""
    import shutil
    import subprocess
    from bit_mixed_precision_gb300 import kvq
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    inc = os.path.join(ROOT, "include")
    fields = {"kvq_tier": kvq.KvqTier, "kvq_cache": kvq.KvqCache, "kvq_policy_params": kvq.KvqPolicyParams}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kvq.h"', "int main(void) {"]
    for cname, py in fields.items():
        lines.append(f'printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", inc, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in fields.items():
        assert got[(cname, "sizeof")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)


def test_host_validation_without_gpu(L):
    from bit_mixed_precision_gb300 import kvq
    vp = ctypes.c_void_p(16)
    # null input
    assert L.kv_quant_pack(None, 0, 1, 1, 32, 128, None, 32, 2, 32, 0, vp, vp, vp, None) == kvq.KVQ_EINVAL
    assert L.kv_quant_pack(None, 0, 1, 1, 32, 128, None, 0, 2, 32, 0, None, None, None, None) == kvq.KVQ_OK
    assert b"null" in L.kvq_last_error()
    # 3-bit codes are not a format
    assert L.kv_quant_pack(vp, 0, 1, 1, 32, 128, None, 32, 3, 32, 0, vp, vp, vp, None) == kvq.KVQ_EINVAL
    # channel grouping needs whole groups of tokens
    assert L.kv_quant_pack(vp, 0, 1, 1, 40, 128, None, 40, 2, 32, 0, vp, vp, vp, None) == kvq.KVQ_EINVAL
    # prefill head dim other than 128 is not built
    assert L.prefill_attn_scores(vp, vp, vp, 0, 1, 2, 2, 64, 96, ctypes.c_float(0.1), 1, vp, vp,
                                 None, None, 0, None) == kvq.KVQ_EUNSUPPORTED
    # GQA needs Hq multiple of Hkv
    assert L.prefill_attn_scores(vp, vp, vp, 0, 1, 3, 2, 64, 128, ctypes.c_float(0.1), 1, vp, vp,
                                 None, None, 0, None) == kvq.KVQ_EINVAL
    # window larger than the prompt
    assert L.select_tokens(vp, 1, 1, 10, vp, 4, 11, vp, vp, None, 0, None) == kvq.KVQ_EINVAL
    # observation window outside [1, T], and a missing lse
    for w in (0, 65):
        assert L.prefill_window_scores(vp, vp, 0, 1, 2, 2, 64, 128, ctypes.c_float(0.1), vp, w, vp,
                                       None) == kvq.KVQ_EINVAL
    assert L.prefill_window_scores(vp, vp, 0, 1, 2, 2, 64, 128, ctypes.c_float(0.1), None, 8, vp,
                                   None) == kvq.KVQ_EINVAL
    assert b"prefill_window_scores" in L.kvq_last_error()
    # empty cache descriptor
    c = kvq.KvqCache()
    assert L.decode_attn_qkv(vp, vp, vp, ctypes.byref(c), ctypes.c_float(0.1), vp, None, vp, 1 << 20,
                             None) == kvq.KVQ_EINVAL
    assert L.kvq_decode_workspace_bytes(ctypes.byref(c)) == ctypes.c_size_t(-1).value
    assert L.kvq_decode_launches(ctypes.byref(c)) == -1
    assert L.kvq_version() == 100


def test_tier_byte_accounting(L):
    from bit_mixed_precision_gb300 import kvq
    out = (ctypes.c_size_t * 8)()
    # one unit, 32 tokens, INT2 keys per channel and values per token, D = 128, G = 32
    tot = L.kvq_tier_bytes(1, 128, 32, 2, 2, kvq.AXIS_CHANNEL, 32, out)
    per_token_payload = sum(out[:6]) / 32
    assert per_token_payload == 96             # 3 bits per scalar, keys + values
    assert tot == sum(out)
    assert L.kvq_tier_bytes(1, 128, 32, 2, 2, kvq.AXIS_CHANNEL, 40, out) == 0


def test_decode_cache_group_sizes(L):
    """The decode kernels take groups of 32; groups of 16 only on the single-head 2-bit
    MiniKV path (D = 128, Hq == Hkv): other caches are refused on the host (the descriptor
    is never dereferenced)."""
    from bit_mixed_precision_gb300 import kvq
    fake = 1 << 20                                  # aligned, never read
    size_max = ctypes.c_size_t(-1).value

    def cache(policy, tiers, nr, res_cap):
        c = kvq.KvqCache()
        c.B, c.Hq, c.Hkv, c.D, c.dtype, c.policy, c.n_tiers = 1, 4, 1, 128, kvq.F16, policy, len(tiers)
        for t, (kb, vb, ax) in enumerate(tiers):
            tr = c.tier[t]
            tr.k_bits, tr.v_bits, tr.k_axis, tr.cap = kb, vb, ax, 256
            for f in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero", "token_id", "count"):
                setattr(tr, f, fake)
        c.res_cap, c.nr = res_cap, nr
        for f in ("res_k", "res_v", "res_token_id", "res_start", "res_len", "seq_len", "cum_score"):
            setattr(c, f, fake)
        c.score_cap, c.hi_den = 1024, 5
        return c

    mikv = cache(kvq.POLICY_MIKV, [(4, 4, kvq.AXIS_TOKEN), (2, 2, kvq.AXIS_TOKEN)], 128, 192)
    minikv = cache(kvq.POLICY_MINIKV, [(2, 2, kvq.AXIS_CHANNEL)], 0, 128)
    for c in (mikv, minikv):
        c.G = 32
        assert L.kvq_decode_workspace_bytes(ctypes.byref(c)) != size_max, L.kvq_last_error()
        for G in (64, 16):
            c.G = G
            assert L.kvq_decode_workspace_bytes(ctypes.byref(c)) == size_max
            assert f"G = {G} is built for 2-bit MiniKV".encode() in L.kvq_last_error()
    minikv.Hq = 1                                   # one query head per KV head: groups of 16 built
    minikv.G = 16
    assert L.kvq_decode_workspace_bytes(ctypes.byref(minikv)) != size_max, L.kvq_last_error()
    minikv.G, minikv.Hq = 32, 4
    # workspace: MiniKV none; MiKV the step's logits [u][g][slots] (slots = tier caps + ring),
    # then (256-byte aligned) the lse per head [u][8] and the ring state [u][4]
    mikv.G = minikv.G = 32
    assert L.kvq_decode_workspace_bytes(ctypes.byref(minikv)) == 0
    slots = 256 + 256 + 192
    logits = 1 * 4 * slots * 4
    assert L.kvq_decode_workspace_bytes(ctypes.byref(mikv)) == (logits + 255) // 256 * 256 + 8 * 4 + 4 * 4
