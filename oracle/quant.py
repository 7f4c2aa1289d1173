"""Oracle: asymmetric low-bit quantisation, packing and dequantisation.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix (MiniKV verdict JSON, ``pith_extraction.key_machinery``
and ``supporting_citations`` for KIVI; MiniKV review page, "Core claim" and
Figure 1 caption): each group of scalars is stored as low-bit unsigned codes
with one FP16 scale and one FP16 zero-point; keys are grouped per channel
(a group runs along tokens), values per token (a group runs along channels);
16 INT2 codes share one 32-bit word.

What the pages leave open and the reading taken here:

* zero-point and scale: z = the largest fp16 not above min(x) (a zero
  minimum or maximum counts as +0.0);
  s = the smallest fp16 not below fp32(fp32(max(x) - z) / (2^b - 1)).
  The directed roundings keep z <= min and z + (2^b-1) s >= max, so the
  stored fp16 pair still covers the group and |x - x_hat| <= s/2.
* code: q = clamp(rint_half_even(fp32(fp32(x - z) / s)), 0, 2^b - 1); a group
  whose scale is 0 (all equal) gets code 0 everywhere and x_hat = z.
* dequantisation: x_hat = fp32(q * s + z).  q * s is exact in float32 (at most
  8 + 11 significant bits), so this single rounding equals fmaf(q, s, z).
* packing: code i of a word sits in bits [b*i, b*i + b), least significant
  first; 32/b codes per word.  Keys are packed along tokens (word w of
  channel c holds tokens w*32/b ...), values along channels.

Pins (tests/test_oracle_quant.py): directed-rounding definitions checked by
neighbour search, the s/2 error bound, brute-force nearest-code search over
every code value, exact round trip of on-grid inputs, the constant group,
hand-computed packed words (tests/golden/pack_int2.txt).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F16 = np.float16


def f16_round_down(x):
    """Largest float16 value that is <= x (x float32, finite)."""
    x = np.asarray(x, dtype=F32)
    h = x.astype(F16)
    over = h.astype(F32) > x
    if np.any(over):
        with np.errstate(over="ignore"):
            h = np.where(over, np.nextafter(h, F16(-np.inf)), h)
    return h.astype(F16)


def f16_round_up(x):
    """Smallest float16 value that is >= x (x float32, finite)."""
    x = np.asarray(x, dtype=F32)
    h = x.astype(F16)
    under = h.astype(F32) < x
    if np.any(under):
        with np.errstate(over="ignore"):
            h = np.where(under, np.nextafter(h, F16(np.inf)), h)
    return h.astype(F16)


def quantize_groups(x, bits):
    """Quantise each row of ``x`` (shape [..., G]) as one group.

    Returns (codes uint8 [..., G], scale fp16 [...], zero fp16 [...]).
    Follows the float32 sequence stated in the module docstring.
    """
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    x = np.asarray(x).astype(F32)          # fp16 / bf16 / fp32 -> fp32 is exact
    qmax = (1 << bits) - 1
    # + 0.0 turns a -0.0 extreme into +0.0: the sign of a zero minimum or
    # maximum is otherwise unspecified (IEEE min/max of signed zeros)
    mn = (x.min(axis=-1) + F32(0.0)).astype(F32)
    mx = (x.max(axis=-1) + F32(0.0)).astype(F32)
    zero = f16_round_down(mn)
    z32 = zero.astype(F32)
    span = (mx - z32).astype(F32)
    scale = f16_round_up((span / F32(qmax)).astype(F32))
    s32 = scale.astype(F32)
    safe = np.where(s32 == 0, F32(1), s32).astype(F32)
    t = ((x - z32[..., None]).astype(F32) / safe[..., None]).astype(F32)
    q = np.rint(t)                          # round half to even
    q = np.clip(q, 0, qmax)
    q = np.where((s32 == 0)[..., None], 0, q)
    return q.astype(np.uint8), scale, zero


def dequantize_groups(codes, scale, zero):
    """x_hat = fp32(q * s + z) per element; ``scale``/``zero`` broadcast on the last axis."""
    q = np.asarray(codes).astype(F32)
    s = np.asarray(scale).astype(F32)[..., None]
    z = np.asarray(zero).astype(F32)[..., None]
    return ((q * s).astype(F32) + z).astype(F32)


def pack_codes(codes, bits):
    """Pack codes along the last axis, 32/bits per uint32, least significant first."""
    codes = np.asarray(codes).astype(np.uint32)
    per = 32 // bits
    n = codes.shape[-1]
    if n % per:
        raise ValueError("last axis must be a multiple of 32/bits")
    c = codes.reshape(codes.shape[:-1] + (n // per, per))
    words = np.zeros(c.shape[:-1], dtype=np.uint32)
    for i in range(per):
        words |= (c[..., i] & np.uint32((1 << bits) - 1)) << np.uint32(bits * i)
    return words


def unpack_codes(words, bits):
    """Inverse of ``pack_codes``: uint32 [..., W] -> uint8 [..., W * 32/bits]."""
    words = np.asarray(words).astype(np.uint32)
    per = 32 // bits
    out = np.zeros(words.shape + (per,), dtype=np.uint8)
    for i in range(per):
        out[..., i] = (words >> np.uint32(bits * i)) & np.uint32((1 << bits) - 1)
    return out.reshape(words.shape[:-1] + (words.shape[-1] * per,))


# ---------------------------------------------------------------------------
# The two groupings.  One unit = one (batch, KV head); x is [n, D].
# ---------------------------------------------------------------------------

def quant_pack_channel(x, bits, group):
    """Keys: per-channel groups of ``group`` consecutive tokens.

    x [n, D] -> codes uint32 [n*bits/32, D], scale fp16 [n/group, D],
    zero fp16 [n/group, D].  Codes are packed along tokens.
    """
    x = np.asarray(x)
    n, d = x.shape
    if n % group:
        raise ValueError("token count must be a multiple of the group size")
    g = x.reshape(n // group, group, d).transpose(0, 2, 1)       # [ng, D, G]
    q, s, z = quantize_groups(g, bits)                            # q [ng, D, G]
    qt = q.transpose(1, 0, 2).reshape(d, n)                       # [D, n] tokens in order
    words = pack_codes(qt, bits)                                  # [D, n*bits/32]
    return words.T.copy(), s, z


def unpack_channel(words, scale, zero, bits, group):
    """Dequantise a per-channel packed block back to float32 [n, D]."""
    q = unpack_codes(np.asarray(words).T, bits)                   # [D, n]
    d, n = q.shape
    qg = q.reshape(d, n // group, group).transpose(1, 0, 2)       # [ng, D, G]
    xh = dequantize_groups(qg, scale, zero)                       # [ng, D, G]
    return xh.transpose(0, 2, 1).reshape(n, d)


def quant_pack_token(x, bits, group):
    """Values (and per-token keys): per-token groups of ``group`` channels.

    x [n, D] -> codes uint32 [n, D*bits/32], scale fp16 [n, D/group],
    zero fp16 [n, D/group].  Codes are packed along channels.
    """
    x = np.asarray(x)
    n, d = x.shape
    if d % group:
        raise ValueError("head dim must be a multiple of the group size")
    g = x.reshape(n, d // group, group)
    q, s, z = quantize_groups(g, bits)                            # q [n, D/G, G]
    words = pack_codes(q.reshape(n, d), bits)
    return words, s, z


def unpack_token(words, scale, zero, bits, group):
    """Dequantise a per-token packed block back to float32 [n, D]."""
    q = unpack_codes(words, bits)                                 # [n, D]
    n, d = q.shape
    xh = dequantize_groups(q.reshape(n, d // group, group), scale, zero)
    return xh.reshape(n, d)


def kv_quant_pack(x, bits, group, axis, gather_idx=None):
    """Batched form of the two groupings over [B, H, T, D] input.

    ``axis`` is "channel" (keys) or "token" (values).  With ``gather_idx``
    [B, H, n] the rows x[b, h, gather_idx[b, h, i]] are packed in that order.
    Returns (codes, scale, zero) with the unit axes [B, H] in front.
    """
    x = np.asarray(x)
    B, H = x.shape[:2]
    fn = quant_pack_channel if axis == "channel" else quant_pack_token
    outs = []
    for b in range(B):
        row = []
        for h in range(H):
            xs = x[b, h] if gather_idx is None else x[b, h][np.asarray(gather_idx)[b, h]]
            row.append(fn(xs, bits, group))
        outs.append(row)
    codes = np.stack([np.stack([r[0] for r in row]) for row in outs])
    scale = np.stack([np.stack([r[1] for r in row]) for row in outs])
    zero = np.stack([np.stack([r[2] for r in row]) for row in outs])
    return codes, scale, zero
