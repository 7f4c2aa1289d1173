"""Thin Python binding of libkvq.so (ctypes over torch CUDA tensors).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  The functions keep the C names; tensors are torch tensors on
the current CUDA device and the work is enqueued on torch's current stream
(or the ``stream`` given).  If the library has not been built the first call
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_ECUDA, KVQ_ETIMEOUT, KVQ_EWORKSPACE, KVQ_EDEVICE = range(7)
F16, BF16 = 0, 1
AXIS_CHANNEL, AXIS_TOKEN = 0, 1
POLICY_MINIKV, POLICY_DIFFKV, POLICY_MIKV = 0, 1, 2
MAX_TIERS = 2

EXPORTS = ["kv_quant_pack", "prefill_attn_scores", "prefill_window_scores", "kvq_score_reduce", "select_tokens",
           "minikv_prefill_build", "requant_demote", "decode_attn_qkv", "decode_attn_qkv_static",
           "kvq_pages_init", "kvq_pages_release",
           "kvq_decode_workspace_bytes", "kvq_decode_launches", "kvq_tier_bytes",
           "kvq_last_error", "kvq_device_status", "kvq_debug_withhold_copy", "kvq_version"]


class KvqError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"kvq status {status}: {msg}")
        self.status = status


class KvqTier(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("k_axis", ctypes.c_int32), ("cap", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("k_zero", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p),
                ("token_id", ctypes.c_void_p), ("count", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("page_owner", ctypes.c_void_p),
                ("free_ring", ctypes.c_void_p), ("ring_ctr", ctypes.c_void_p),
                ("max_pages", ctypes.c_int32), ("n_pages", ctypes.c_int32)]


class KvqCache(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("G", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("policy", ctypes.c_int32), ("n_tiers", ctypes.c_int32),
                ("tier", KvqTier * MAX_TIERS),
                ("res_cap", ctypes.c_int32), ("nr", ctypes.c_int32),
                ("res_k", ctypes.c_void_p), ("res_v", ctypes.c_void_p),
                ("res_token_id", ctypes.c_void_p), ("res_start", ctypes.c_void_p),
                ("res_len", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
                ("win_acc", ctypes.c_void_p), ("alpha", ctypes.c_void_p),
                ("cum_score", ctypes.c_void_p), ("score_cap", ctypes.c_int32),
                ("hi_den", ctypes.c_int32)]


class KvqPolicyParams(ctypes.Structure):
    _fields_ = [("k_src", ctypes.c_void_p), ("v_src", ctypes.c_void_p), ("T", ctypes.c_int32),
                ("sel_idx", ctypes.c_void_p), ("n_sel", ctypes.c_int32),
                ("colscore", ctypes.c_void_p), ("n_high", ctypes.c_void_p),
                ("n_low", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -c 'import __graft_entry__ as g; "
                               "g.build()'` (nvcc, sm_103a) first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.kv_quant_pack.argtypes = [vp, i32, i32, i32, i32, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.prefill_attn_scores.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, vp,
                                          vp, vp, sz, vp]
        L.prefill_window_scores.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, i32, vp, vp]
        L.kvq_score_reduce.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp]
        L.select_tokens.argtypes = [vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, sz, vp]
        L.requant_demote.argtypes = [ctypes.POINTER(KvqCache), i32, ctypes.POINTER(KvqPolicyParams),
                                     i32, vp]
        L.minikv_prefill_build.argtypes = [ctypes.POINTER(KvqCache), vp, vp, i32, vp, vp, i32, i32, vp, vp]
        L.kvq_pages_init.argtypes = [ctypes.POINTER(KvqCache), vp]
        L.kvq_pages_release.argtypes = [ctypes.POINTER(KvqCache), vp, vp]
        L.decode_attn_qkv.argtypes = [vp, vp, vp, ctypes.POINTER(KvqCache), f32, vp, vp, vp, sz, vp]
        L.decode_attn_qkv_static.argtypes = [vp, vp, vp, ctypes.POINTER(KvqCache), f32, vp, vp, vp]
        L.decode_attn_qkv_static.restype = ctypes.c_int
        L.kvq_decode_workspace_bytes.argtypes = [ctypes.POINTER(KvqCache)]
        L.kvq_decode_workspace_bytes.restype = sz
        L.kvq_decode_launches.argtypes = [ctypes.POINTER(KvqCache)]
        L.kvq_decode_launches.restype = ctypes.c_int
        L.kvq_tier_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
        L.kvq_tier_bytes.restype = sz
        L.kvq_last_error.restype = ctypes.c_char_p
        L.kvq_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.kvq_debug_withhold_copy.argtypes = [i32]
        for name in ["kv_quant_pack", "prefill_attn_scores", "prefill_window_scores", "kvq_score_reduce", "select_tokens",
                     "minikv_prefill_build", "requant_demote", "kvq_pages_init", "kvq_pages_release", "decode_attn_qkv", "kvq_device_status", "kvq_debug_withhold_copy"]:
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status):
    if status != KVQ_OK:
        raise KvqError(status, lib().kvq_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t):
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("activations must be float16 or bfloat16")


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# --------------------------------------------------------------------- ops

def kv_quant_pack(x, bits, group, axis, gather_idx=None, n=None, out=None, stream=None):
    """Quantise + pack x [B, H, T, D]; returns (codes, scale, zero)."""
    _cuda(x, gather_idx)
    B, H, T, D = x.shape
    if n is None:
        n = gather_idx.shape[-1] if gather_idx is not None else T
    if out is None:
        dev = x.device
        if axis == AXIS_CHANNEL:
            codes = torch.empty((B, H, n * bits // 32, D), dtype=torch.int32, device=dev)
            scale = torch.empty((B, H, n // group, D), dtype=torch.int16, device=dev)
        else:
            codes = torch.empty((B, H, n, D * bits // 32), dtype=torch.int32, device=dev)
            scale = torch.empty((B, H, n, D // group), dtype=torch.int16, device=dev)
        zero = torch.empty_like(scale)
    else:
        codes, scale, zero = out
    _check(lib().kv_quant_pack(_ptr(x), _dt(x), B, H, T, D, _ptr(gather_idx), n, bits, group, axis,
                               _ptr(codes), _ptr(scale), _ptr(zero), _stream(stream)))
    return codes, scale, zero


def _check_qk(q, k, v=None):
    """q [B, Hq, T, D] and k (v) [B, Hkv, T, D] of one dtype, Hq a multiple of Hkv: the
    kernels build their tensor maps from q's sizes, so a shorter k would be read past
    its end."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k must be [B, H, T, D]")
    B, Hq, T, D = q.shape
    for x in (k, v):
        if x is None:
            continue
        if x.dtype != q.dtype:
            raise TypeError("q, k and v must share one dtype")
        if x.shape[0] != B or x.shape[2:] != (T, D) or x.shape[1] != k.shape[1]:
            raise ValueError(f"k/v shape {tuple(x.shape)} does not match q {tuple(q.shape)}")
    if k.shape[1] == 0 or Hq % k.shape[1]:
        raise ValueError("Hq must be a multiple of Hkv")


def _check_lse(lse, q):
    B, Hq, T, _ = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, T):
        raise ValueError(f"lse must be float32 [{B}, {Hq}, {T}]")


def prefill_attn_scores(q, k, v, sm_scale=None, colscore=True, out=None, stream=None):
    """Two-pass prefill: returns (o [B,Hq,T,D], lse [B,Hq,T], colscore [B,Hq,T] or None)."""
    _cuda(q, k, v)
    _check_qk(q, k, v)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
        cs = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if colscore else None
    else:
        o, lse, cs = out
        _cuda(o, lse, cs)
        if o.shape != q.shape or o.dtype != q.dtype:
            raise ValueError("o must have q's shape and dtype")
        _check_lse(lse, q)
        if cs is not None:
            _check_lse(cs, q)
    _check(lib().prefill_attn_scores(_ptr(q), _ptr(k), _ptr(v), _dt(q), B, Hq, Hkv, T, D,
                                     float(sm_scale), 1, _ptr(o), _ptr(lse), _ptr(cs), None, 0,
                                     _stream(stream)))
    return o, lse, cs


def prefill_window_scores(q, k, lse, w_obs, sm_scale=None, out=None, stream=None):
    """Column scores over the last w_obs queries (lse from prefill_attn_scores): [B, Hq, T]."""
    _cuda(q, k, lse)
    _check_qk(q, k)
    _check_lse(lse, q)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    _cuda(out)
    _check_lse(out, q)
    _check(lib().prefill_window_scores(_ptr(q), _ptr(k), _dt(q), B, Hq, Hkv, T, D, float(sm_scale), _ptr(lse),
                                       int(w_obs), _ptr(out), _stream(stream)))
    return out


def kvq_score_reduce(colscore, Hkv, mode, out=None, stream=None):
    """[B, Hq, T] -> [B, Hkv, T]; mode 0 = sum over the group, 1 = max of cs/(T-j)."""
    _cuda(colscore)
    B, Hq, T = colscore.shape
    if out is None:
        out = torch.empty((B, Hkv, T), dtype=torch.float32, device=colscore.device)
    _check(lib().kvq_score_reduce(_ptr(colscore), B, Hq, Hkv, T, mode, _ptr(out), _stream(stream)))
    return out


def select_tokens(score, k_hh, w_recent, kmax=None, out=None, stream=None):
    """Heavy hitters + recent window; returns (idx [B, H, kmax + w], n [B*H])."""
    _cuda(score, k_hh)
    B, H, T = score.shape
    if kmax is None:
        kmax = int(k_hh.max().item()) if k_hh.numel() else 0
    if out is None:
        idx = torch.empty((B, H, kmax + w_recent), dtype=torch.int32, device=score.device)
        n = torch.empty((B * H,), dtype=torch.int32, device=score.device)
    else:
        idx, n = out
    _check(lib().select_tokens(_ptr(score), B, H, T, _ptr(k_hh), kmax, w_recent, _ptr(idx),
                               _ptr(n), None, 0, _stream(stream)))
    return idx, n


def debug_withhold_copy(on):
    """Failure-detection check: while on, decode launches withhold one staged copy of unit 0
    so that its bounded waits run out and device_status() reports KVQ_ETIMEOUT."""
    _check(lib().kvq_debug_withhold_copy(1 if on else 0))


def device_status(stream=None):
    """Synchronises and returns (and clears) the device status word (0 = fine)."""
    v = ctypes.c_uint32(0)
    _check(lib().kvq_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)


# --------------------------------------------------------------------- cache

@dataclass
class TierSpec:
    k_bits: int
    v_bits: int
    k_axis: int
    cap: int


PAGE_TOKENS = 128


@dataclass
class Tier:
    spec: TierSpec
    k_codes: torch.Tensor
    k_scale: torch.Tensor
    k_zero: torch.Tensor
    v_codes: torch.Tensor
    v_scale: torch.Tensor
    v_zero: torch.Tensor
    token_id: torch.Tensor
    count: torch.Tensor
    # paged tiers (DiffKV): the arrays above are [n_pages, PAGE_TOKENS, ...]
    page_table: torch.Tensor = None     # [units, max_pages] int32
    page_owner: torch.Tensor = None     # [n_pages] int32
    free_ring: torch.Tensor = None      # [n_pages] int32
    ring_ctr: torch.Tensor = None       # [2] (head, tail)
    max_pages: int = 0
    n_pages: int = 0

    def rows_of(self, u):
        """Flat row indices (into the arrays viewed as [rows, ...]) of unit u's slots 0..count-1."""
        c = int(self.count[u].item())
        if self.page_table is None:
            return torch.arange(u * self.spec.cap, u * self.spec.cap + c)
        pt = self.page_table[u].cpu()
        s = torch.arange(c)
        return pt[s // PAGE_TOKENS].long() * PAGE_TOKENS + s % PAGE_TOKENS


@dataclass
class Cache:
    """Device memory of one layer's compressed cache plus its C descriptor."""
    B: int
    Hq: int
    Hkv: int
    D: int
    G: int
    dtype: torch.dtype
    policy: int
    tiers: list
    nr: int
    res_cap: int
    res_k: torch.Tensor
    res_v: torch.Tensor
    res_token_id: torch.Tensor
    res_start: torch.Tensor
    res_len: torch.Tensor
    seq_len: torch.Tensor
    win_acc: torch.Tensor = None
    alpha: torch.Tensor = None
    cum_score: torch.Tensor = None
    score_cap: int = 0
    hi_den: int = 5
    desc: KvqCache = field(default=None, repr=False)
    ws: torch.Tensor = field(default=None, repr=False)

    @property
    def units(self):
        return self.B * self.Hkv

    def _make_desc(self):
        d = KvqCache()
        d.B, d.Hq, d.Hkv, d.D, d.G = self.B, self.Hq, self.Hkv, self.D, self.G
        d.dtype = F16 if self.dtype == torch.float16 else BF16
        d.policy = self.policy
        d.n_tiers = len(self.tiers)
        for i, t in enumerate(self.tiers):
            s = t.spec
            pg = t.page_table is not None
            d.tier[i] = KvqTier(s.k_bits, s.v_bits, s.k_axis, s.cap, t.k_codes.data_ptr(),
                                t.k_scale.data_ptr(), t.k_zero.data_ptr(), t.v_codes.data_ptr(),
                                t.v_scale.data_ptr(), t.v_zero.data_ptr(), t.token_id.data_ptr(),
                                t.count.data_ptr(),
                                t.page_table.data_ptr() if pg else None, t.page_owner.data_ptr() if pg else None,
                                t.free_ring.data_ptr() if pg else None, t.ring_ctr.data_ptr() if pg else None,
                                t.max_pages, t.n_pages)
        d.res_cap, d.nr = self.res_cap, self.nr
        d.res_k, d.res_v = self.res_k.data_ptr(), self.res_v.data_ptr()
        d.res_token_id = self.res_token_id.data_ptr()
        d.res_start, d.res_len = self.res_start.data_ptr(), self.res_len.data_ptr()
        d.seq_len = self.seq_len.data_ptr()
        d.win_acc = self.win_acc.data_ptr() if self.win_acc is not None else None
        d.alpha = self.alpha.data_ptr() if self.alpha is not None else None
        d.cum_score = self.cum_score.data_ptr() if self.cum_score is not None else None
        d.score_cap, d.hi_den = self.score_cap, self.hi_den
        self.desc = d
        nbytes = lib().kvq_decode_workspace_bytes(ctypes.byref(d))
        if nbytes == ctypes.c_size_t(-1).value:
            raise KvqError(KVQ_EINVAL, lib().kvq_last_error().decode())
        self.ws = (torch.empty((nbytes + 255) // 4, dtype=torch.int32, device=self.res_k.device)
                   if nbytes else None)

    def tier_nbytes(self):
        """Bytes held by the packed tiers (codes + scale/zero + ids), all units."""
        tot = 0
        for t in self.tiers:
            for x in (t.k_codes, t.k_scale, t.k_zero, t.v_codes, t.v_scale, t.v_zero):
                tot += x.numel() * x.element_size()
        return tot


def _alloc_paged_tier(units, D, G, spec, n_pages, device):
    """A tier whose slots live in a pool of n_pages pages of PAGE_TOKENS slots shared by the units."""
    max_pages = (spec.cap + PAGE_TOKENS - 1) // PAGE_TOKENS
    spec = TierSpec(spec.k_bits, spec.v_bits, spec.k_axis, max_pages * PAGE_TOKENS)
    pool = _alloc_tier(n_pages, D, G, TierSpec(spec.k_bits, spec.v_bits, spec.k_axis, PAGE_TOKENS), device)
    i32 = torch.int32
    return Tier(spec, pool.k_codes, pool.k_scale, pool.k_zero, pool.v_codes, pool.v_scale, pool.v_zero,
                pool.token_id, torch.zeros((units,), dtype=i32, device=device),
                page_table=torch.full((units, max_pages), -1, dtype=i32, device=device),
                page_owner=torch.full((n_pages,), -1, dtype=i32, device=device),
                free_ring=torch.arange(n_pages, dtype=i32, device=device),
                ring_ctr=torch.tensor([0, n_pages], dtype=torch.int32, device=device),
                max_pages=max_pages, n_pages=n_pages)


def _alloc_tier(units, D, G, spec, device):
    spec = TierSpec(spec.k_bits, spec.v_bits, spec.k_axis, (spec.cap + 31) // 32 * 32)
    cap = spec.cap
    i32, i16 = torch.int32, torch.int16
    if spec.k_axis == AXIS_CHANNEL:
        kc = torch.zeros((units, cap * spec.k_bits // 32, D), dtype=i32, device=device)
        ks = torch.zeros((units, cap // G, D), dtype=i16, device=device)
    else:
        kc = torch.zeros((units, cap, D * spec.k_bits // 32), dtype=i32, device=device)
        ks = torch.zeros((units, cap, D // G), dtype=i16, device=device)
    vc = torch.zeros((units, cap, D * spec.v_bits // 32), dtype=i32, device=device)
    vs = torch.zeros((units, cap, D // G), dtype=i16, device=device)
    return Tier(spec, kc, ks, torch.zeros_like(ks), vc, vs, torch.zeros_like(vs),
                torch.full((units, cap), -1, dtype=i32, device=device),
                torch.zeros((units,), dtype=i32, device=device))


def make_cache(B, Hq, Hkv, D, G, dtype, policy, tiers, nr, res_cap=None, score_cap=0, hi_den=5,
               device="cuda", pages=None):
    """Allocates every array of a cache (torch device memory) and its descriptor.  `pages`
    (DiffKV): a pool size in pages per tier (None for a fixed per-unit tier); a paged
    tier's spec.cap is then the most slots one unit may hold.  Paged caches are emptied
    with pages_init before their first build."""
    units = B * Hkv
    if res_cap is None:
        res_cap = nr + G if policy == POLICY_MINIKV else nr + 1
    pages = pages or [None] * len(tiers)
    c = Cache(B=B, Hq=Hq, Hkv=Hkv, D=D, G=G, dtype=dtype, policy=policy,
              tiers=[_alloc_tier(units, D, G, s, device) if n is None
                     else _alloc_paged_tier(units, D, G, s, n, device) for s, n in zip(tiers, pages)],
              nr=nr, res_cap=res_cap,
              res_k=torch.zeros((units, res_cap, D), dtype=dtype, device=device),
              res_v=torch.zeros((units, res_cap, D), dtype=dtype, device=device),
              res_token_id=torch.full((units, res_cap), -1, dtype=torch.int32, device=device),
              res_start=torch.zeros((units,), dtype=torch.int32, device=device),
              res_len=torch.zeros((units,), dtype=torch.int32, device=device),
              seq_len=torch.zeros((B * Hkv,), dtype=torch.int32, device=device),
              score_cap=score_cap, hi_den=hi_den)
    if policy == POLICY_DIFFKV:
        c.win_acc = torch.zeros((B * Hq, res_cap), dtype=torch.float32, device=device)
        c.alpha = torch.zeros((units, 2), dtype=torch.float32, device=device)
    if policy == POLICY_MIKV:
        c.cum_score = torch.zeros((units, score_cap), dtype=torch.float32, device=device)
    c._make_desc()
    return c


def pages_init(cache, stream=None):
    """Empties every paged tier (free ring 0 .. n_pages-1, no owners, no table entries)."""
    _check(lib().kvq_pages_init(ctypes.byref(cache.desc), _stream(stream)))


def pages_release(cache, mask, stream=None):
    """Returns every page of the units with mask[u] != 0 (int32 [B*Hkv] CUDA tensor)."""
    _cuda(mask)
    if mask.dtype != torch.int32 or mask.numel() != cache.units:
        raise ValueError("mask must be int32 [B * Hkv]")
    _check(lib().kvq_pages_release(ctypes.byref(cache.desc), _ptr(mask), _stream(stream)))


def requant_demote(cache, step, k_src=None, v_src=None, sel_idx=None, n_sel=0, colscore=None,
                   n_high=None, n_low=None, stream=None):
    """Policy tail (step > 0) or cache build at the end of prefill (step == 0)."""
    p = None
    if step == 0:
        _cuda(k_src, v_src, sel_idx, colscore, n_high, n_low)
        p = KvqPolicyParams(k_src.data_ptr(), v_src.data_ptr(), k_src.shape[2],
                            sel_idx.data_ptr() if sel_idx is not None else None, n_sel,
                            colscore.data_ptr() if colscore is not None else None,
                            n_high.data_ptr() if n_high is not None else None,
                            n_low.data_ptr() if n_low is not None else None)
    _check(lib().requant_demote(ctypes.byref(cache.desc), cache.policy,
                                ctypes.byref(p) if p is not None else None, step, _stream(stream)))


def minikv_prefill_build(cache, k, v, score, k_hh, w_recent, kmax=None, idx_out=None, stream=None):
    """MiniKV prefill-end build in one launch: heavy hitters + window from score [B, Hkv, T],
    packed into tier 0 with the residual filled (select_tokens + requant_demote(step 0))."""
    _cuda(k, v, score, k_hh, idx_out)
    B, H, T, D = k.shape
    if v.shape != k.shape or v.dtype != k.dtype or k.dtype != cache.dtype:
        raise ValueError("k and v must share the cache's dtype and one shape")
    if tuple(score.shape) != (B, H, T) or score.dtype != torch.float32:
        raise ValueError(f"score must be float32 [{B}, {H}, {T}]")
    if (B, H, D) != (cache.B, cache.Hkv, cache.D):
        raise ValueError("k does not match the cache's B / Hkv / D")
    if k_hh.dtype != torch.int32 or k_hh.numel() != B * H:
        raise ValueError("k_hh must be int32 [B * Hkv]")
    if kmax is None:
        kmax = int(k_hh.max().item()) if k_hh.numel() else 0
    if idx_out is not None and (idx_out.dtype != torch.int32 or idx_out.numel() != B * H * (kmax + w_recent)):
        raise ValueError("idx_out must be int32 [B, Hkv, kmax + w_recent]")
    _check(lib().minikv_prefill_build(ctypes.byref(cache.desc), _ptr(k), _ptr(v), T, _ptr(score), _ptr(k_hh),
                                      int(kmax), int(w_recent), _ptr(idx_out), _stream(stream)))
    return idx_out


def decode_attn_qkv(q, k_new, v_new, cache, sm_scale=None, o=None, lse=None, stream=None):
    """One decode step; returns (o [B, Hq, D], lse [B, Hq])."""
    _cuda(q, k_new, v_new)
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().decode_attn_qkv(_ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(cache.desc),
                                 float(sm_scale), _ptr(o), _ptr(lse), _ptr(cache.ws),
                                 0 if cache.ws is None else cache.ws.numel() * 4, _stream(stream)))
    return o, lse


STATIC_SCRATCH_BYTES = 16 << 20


def decode_launches(cache):
    """Kernel launches one decode_attn_qkv call makes for the cache on the current device."""
    n = lib().kvq_decode_launches(ctypes.byref(cache.desc))
    if n < 0:
        raise KvqError(KVQ_EINVAL, lib().kvq_last_error().decode())
    return n


def decode_attn_qkv_static(q, k_new, v_new, cache, sm_scale=None, o=None, lse=None, stream=None):
    """decode_attn_qkv for callers that cannot provide scratch memory.

    The library uses its own built-in device array (STATIC_SCRATCH_BYTES)
    instead of ``cache.ws``; nothing is allocated by the call.  Calls whose
    GPU work overlaps share that array and must not run concurrently.
    """
    _cuda(q, k_new, v_new)
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().decode_attn_qkv_static(_ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(cache.desc),
                                        float(sm_scale), _ptr(o), _ptr(lse), _stream(stream)))
    return o, lse
