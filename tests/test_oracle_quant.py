"""Pins of the oracle quantiser against what the pages and arithmetic fix (no GPU)."""
import os

import numpy as np
import pytest

from oracle import quant

F32 = np.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def test_f16_directed_rounding_definition():
    r = _rng(1)
    x = np.concatenate([
        r.normal(size=20000).astype(F32) * F32(10.0),
        (r.normal(size=2000) * 1e-6).astype(F32),          # fp16 subnormal range
        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, -65504.0, 6e-8], F32),
        np.float16(r.normal(size=500)).astype(F32),         # exactly representable
    ])
    lo = quant.f16_round_down(x)
    hi = quant.f16_round_up(x)
    lo32 = lo.astype(F32)
    hi32 = hi.astype(F32)
    assert np.all(lo32 <= x) and np.all(hi32 >= x)
    # neighbour search: the next fp16 value beyond the result crosses x
    with np.errstate(over="ignore"):
        nlo = np.nextafter(lo, np.float16(np.inf)).astype(F32)
        nhi = np.nextafter(hi, np.float16(-np.inf)).astype(F32)
    assert np.all(nlo > x)
    assert np.all(nhi < x)
    exact = lo32 == x
    assert np.array_equal(exact, hi32 == x)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound_and_cover(bits):
    r = _rng(bits)
    x = r.normal(size=(4000, 32)).astype(np.float16).astype(F32)
    x[::7, 3] *= F32(10.0)                                  # outlier scalars
    q, s, z = quant.quantize_groups(x, bits)
    qmax = (1 << bits) - 1
    s32 = s.astype(F32)
    z32 = z.astype(F32)
    assert q.max() <= qmax
    assert np.all(z32 <= x.min(axis=1))
    cover = z32.astype(np.float64) + qmax * s32.astype(np.float64)
    assert np.all(cover >= x.max(axis=1) * (1 - 2e-7) - 1e-30)
    xh = quant.dequantize_groups(q, s, z)
    err = np.abs(xh.astype(np.float64) - x)
    tol = s32[:, None] * (0.5 + 2.0 ** -20) + np.spacing(np.abs(x)).astype(np.float64)
    assert np.all(err <= tol)


@pytest.mark.parametrize("bits", [2, 4])
def test_nearest_code_by_enumeration(bits):
    """Every code is the nearest of all 2^b codes to t = (x - z)/s; ties go to even."""
    r = _rng(10 + bits)
    x = r.normal(size=(3000, 32)).astype(np.float16).astype(F32)
    q, s, z = quant.quantize_groups(x, bits)
    s32 = s.astype(F32)[:, None]
    z32 = z.astype(F32)[:, None]
    t = ((x - z32).astype(F32) / s32).astype(F32).astype(np.float64)
    cand = np.arange(1 << bits, dtype=np.float64)
    dist = np.abs(t[..., None] - cand)
    best = dist.min(axis=-1)
    nearest = np.abs(dist - best[..., None]) == 0
    # among equally near codes, the even one
    pick = np.where(nearest.sum(-1) > 1,
                    np.argmax(nearest & (cand % 2 == 0), axis=-1),
                    np.argmax(nearest, axis=-1))
    assert np.array_equal(pick, q.astype(np.int64))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_on_grid_round_trip(bits):
    """x = q*s + z exactly, with codes 0 and 2^b-1 present, is recovered exactly."""
    r = _rng(20 + bits)
    qmax = (1 << bits) - 1
    n = 500
    s = np.float16(2.0 ** r.integers(-8, 0, size=n) * (1 + r.integers(0, 64, size=n) / 64.0))
    z = np.float16(-r.integers(1, 200, size=n) / 16.0)
    q = r.integers(0, qmax + 1, size=(n, 32))
    q[:, 0] = 0
    q[:, 1] = qmax
    x = (q * s.astype(np.float64)[:, None] + z.astype(np.float64)[:, None])
    assert np.array_equal(x.astype(F32).astype(np.float64), x)   # exactly representable
    x = x.astype(F32)
    qq, ss, zz = quant.quantize_groups(x, bits)
    assert np.array_equal(zz, z)
    assert np.array_equal(ss, s)
    assert np.array_equal(qq, q.astype(np.uint8))
    assert np.array_equal(quant.dequantize_groups(qq, ss, zz), x)


def test_constant_group():
    x = np.full((3, 32), np.float16(0.7109375), F32)
    x[1] = F32(-3.5)
    x[2] = F32(0.0)
    for bits in (2, 4, 8):
        q, s, z = quant.quantize_groups(x, bits)
        assert np.all(q == 0) and np.all(s == 0)
        assert np.array_equal(quant.dequantize_groups(q, s, z), x)


def _golden_pack():
    rows = []
    with open(os.path.join(GOLDEN, "pack_int2.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            codes, word = line.split(";")
            rows.append(([int(c) for c in codes.split()], int(word.strip(), 16)))
    return rows


def test_pack_golden():
    for codes, word in _golden_pack():
        got = quant.pack_codes(np.array([codes]), 2)
        assert got.shape == (1, 1) and int(got[0, 0]) == word
        assert list(quant.unpack_codes(got, 2)[0]) == codes


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_round_trip(bits):
    r = _rng(30 + bits)
    c = r.integers(0, 1 << bits, size=(7, 64)).astype(np.uint8)
    w = quant.pack_codes(c, bits)
    assert w.shape == (7, 64 * bits // 32)
    assert np.array_equal(quant.unpack_codes(w, bits), c)


def test_channel_grouping_layout():
    """Keys: a group is G consecutive tokens of one channel, packed along tokens."""
    G = 32
    x = np.zeros((64, 4), F32)
    # channel 1: tokens 0..31 take values 0..3 cyclically -> codes 0..3, s = 1, z = 0
    x[:32, 1] = np.arange(32) % 4
    # channel 2, second group: 10 + the same pattern
    x[32:, 2] = 10 + np.arange(32) % 4
    w, s, z = quant.quant_pack_channel(x, 2, G)
    assert w.shape == (4, 4) and s.shape == (2, 4) and z.shape == (2, 4)
    assert float(s[0, 1]) == 1.0 and float(z[0, 1]) == 0.0
    assert float(s[1, 2]) == 1.0 and float(z[1, 2]) == 10.0
    # tokens 0..15 of channel 1 live in word row 0: codes 0,1,2,3,... -> 0xe4e4e4e4
    assert int(w[0, 1]) == 0xE4E4E4E4 and int(w[1, 1]) == 0xE4E4E4E4
    assert int(w[2, 2]) == 0xE4E4E4E4 and int(w[2, 1]) == 0
    back = quant.unpack_channel(w, s, z, 2, G)
    assert np.array_equal(back, x)


def test_token_grouping_layout():
    """Values: a group is G consecutive channels of one token, packed along channels."""
    x = np.zeros((2, 64), F32)
    x[0, 32:] = 5 + 2 * (np.arange(32) % 4)                 # s = 2, z = 5
    w, s, z = quant.quant_pack_token(x, 2, 32)
    assert w.shape == (2, 4) and s.shape == (2, 2)
    assert float(s[0, 1]) == 2.0 and float(z[0, 1]) == 5.0
    assert int(w[0, 2]) == 0xE4E4E4E4 and int(w[0, 0]) == 0
    assert np.array_equal(quant.unpack_token(w, s, z, 2, 32), x)


def test_signed_zero_extremes_are_canonical():
    """A group whose minimum/maximum is -0.0 stores the same z/s bits as +0.0."""
    a = np.zeros((2, 32), F32)
    a[0, 5] = F32(-0.0)
    a[1, :] = F32(-0.0)
    a[0, 7] = F32(1.5)
    q, s, z = quant.quantize_groups(a, 2)
    assert z.view(np.uint16).tolist() == [0, 0]
    assert s.view(np.uint16)[1] == 0
    assert np.all(q[1] == 0)
