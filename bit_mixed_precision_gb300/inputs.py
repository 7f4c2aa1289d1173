"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and value structure of the workloads (Gaussian queries,
keys and values, a few outlier key channels scaled up, per-channel key
standard deviations, Dirichlet tier fractions).  Everything is drawn with a
torch.Generator seeded by the caller, on the CPU (small cases that the
oracle also sees) or on the GPU (full-size cases, where the oracle receives
device-to-host copies of the units it checks).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass
class QKV:
    q: torch.Tensor          # [B, Hq, T, D]
    k: torch.Tensor          # [B, Hkv, T, D]
    v: torch.Tensor          # [B, Hkv, T, D]


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def outlier_channels(n_heads, head_dim, count, seed):
    """Per-head list of ``count`` distinct outlier channels (CPU, deterministic)."""
    g = _gen(seed + 7919, "cpu")
    rows = [torch.randperm(head_dim, generator=g)[:count].sort().values for _ in range(n_heads)]
    return torch.stack(rows) if count else torch.zeros((n_heads, 0), dtype=torch.long)


def make_qkv(B, Hq, Hkv, T, D, dtype=torch.float16, seed=0, device="cpu",
             outliers=None, outlier_scale=1.0, key_std=None):
    """Gaussian Q, K, V.

    ``outliers``: [Hkv, c] channel indices scaled by ``outlier_scale`` in K
    (the same channels for every batch element).  ``key_std``: optional
    [Hkv, D] per-channel standard deviation of K.  Values are drawn in
    float32 and rounded once to ``dtype``.
    """
    g = _gen(seed, device)
    q = torch.randn((B, Hq, T, D), generator=g, device=device, dtype=torch.float32)
    k = torch.randn((B, Hkv, T, D), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((B, Hkv, T, D), generator=g, device=device, dtype=torch.float32)
    if key_std is not None:
        k.mul_(key_std.to(device=device, dtype=torch.float32)[None, :, None, :])
    if outliers is not None and outliers.numel():
        mult = torch.ones((Hkv, D), dtype=torch.float32)
        for h in range(Hkv):
            mult[h, outliers[h]] = float(outlier_scale)
        k.mul_(mult.to(device)[None, :, None, :])
    return QKV(q.to(dtype), k.to(dtype), v.to(dtype))


def make_decode_step(B, Hq, Hkv, D, step, dtype=torch.float16, seed=0, device="cpu",
                     outliers=None, outlier_scale=1.0, key_std=None):
    """New query and new key/value of decode step ``step`` (position T + step)."""
    g = _gen(seed * 1000003 + 17 + step, device)
    q = torch.randn((B, Hq, D), generator=g, device=device, dtype=torch.float32)
    k = torch.randn((B, Hkv, D), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((B, Hkv, D), generator=g, device=device, dtype=torch.float32)
    if key_std is not None:
        k.mul_(key_std.to(device=device, dtype=torch.float32)[None])
    if outliers is not None and outliers.numel():
        mult = torch.ones((Hkv, D), dtype=torch.float32)
        for h in range(Hkv):
            mult[h, outliers[h]] = float(outlier_scale)
        k.mul_(mult.to(device)[None])
    return q.to(dtype), k.to(dtype), v.to(dtype)


def lognormal_key_std(n_heads, head_dim, sigma=0.5, seed=0):
    """Per-(head, channel) key standard deviation drawn from LogNormal(0, sigma)."""
    g = _gen(seed + 104729, "cpu")
    return torch.exp(torch.randn((n_heads, head_dim), generator=g) * sigma)


def dirichlet_fractions(n_units, alpha=(2.0, 5.0, 3.0), seed=0):
    """[n_units, 3] float64 fractions (high, low, prune) from Dirichlet(alpha)."""
    rng = np.random.default_rng(int(seed) + 15485863)
    return rng.dirichlet(alpha, size=n_units)


def random_scores(B, H, T, seed=0, device="cpu", ties=0):
    """Non-negative float32 scores shaped like column scores, optionally with ties.

    ``ties`` > 0 rounds the scores to that many distinct levels so that many
    positions share a value.
    """
    g = _gen(seed + 31, device)
    s = torch.rand((B, H, T), generator=g, device=device, dtype=torch.float32)
    s = s * s * 4.0
    if ties:
        s = torch.floor(s * ties) / ties
    return s
