"""Pins of the oracle selection and budgets (no GPU)."""
import os

import numpy as np

from oracle import select as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute(score, k, w):
    T = len(score)
    cand = sorted(range(T - w), key=lambda j: (-float(score[j]), j))
    return sorted(cand[:min(k, T - w)]) + list(range(T - w, T))


def test_brute_force_sort():
    r = np.random.default_rng(0)
    for trial in range(200):
        T = int(r.integers(1, 90))
        w = int(r.integers(0, T + 1))
        k = int(r.integers(0, T + 1))
        sc = r.integers(0, 6, size=T).astype(np.float32) / 4  # many ties
        assert list(S.select_unit(sc, k, w)) == _brute(sc, k, w)


def test_golden_ties():
    with open(os.path.join(GOLDEN, "select_ties.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            head, sc, exp = line.split(";")
            T, k, w = (int(x) for x in head.split())
            sc = np.array([float(x) for x in sc.split()], np.float32)
            assert len(sc) == T
            assert list(S.select_unit(sc, k, w)) == [int(x) for x in exp.split()]


def test_window_only_and_full_budget():
    sc = np.random.default_rng(1).random(64).astype(np.float32)
    assert list(S.select_unit(sc, 0, 16)) == list(range(48, 64))
    k, w = S.budget(64, 100, 0)
    assert list(S.select_unit(sc, k, w)) == list(range(64))
    k, w = S.budget(64, 50, 50)
    assert list(S.select_unit(sc, k, w)) == list(range(64))


def test_budgets():
    assert S.budget(256, 25, 25) == (64, 64)
    assert S.budget(4096, 25, 25) == (1024, 1024)
    assert S.budget(100, 90, 25) == (75, 25)       # clamped to T - w
    ks = [S.pyramid_hh_budget(16384, l, 32) for l in range(32)]
    assert ks[0] == 6553 and ks[31] == 1638      # floor(0.4 T), floor(0.1 T)
    assert all(a >= b for a, b in zip(ks, ks[1:]))
    # linear: second differences of the unfloored schedule vanish
    exact = [16384 * (40 * 31 - 30 * l) / 3100 for l in range(32)]
    assert all(abs(k - e) < 1 for k, e in zip(ks, exact))
