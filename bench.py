"""Benchmark of the compressed-KV-cache attention hot path on one GB300 (or N replicas).

One step = the whole hot path over one batch of synthetic input: two-pass
prefill (output + column scores), the prefill-end cache build (selection and
INT2 packing in one launch for MiniKV, the tier split for DiffKV / MiKV), then every decode
step of the workload (attention over the packed cache + the policy tail).

Default workload (`pyramid`): the 32-layer MiniKV pyramid sweep -- 32 layers of
32 heads x head dim 128, batch 16, prompt 16384, keys with LogNormal(0, 0.5)
per-channel std, heavy-hitter budget falling linearly from 40% (layer 0) to
10% (layer 31) plus a 25% recent window, INT2 with fp16 scale / zero in groups
of 32, 256 decode steps of every layer (one CUDA graph of the 32 layers' decode
launches per step).  It is the largest workload that fits one GPU (12.9 GB of
packed cache read per decode step).  Other workloads (`--workload`):
`llama-layer` (the LLaMA2-7B-shaped layer: batch 1, 32 heads, prompt 4096,
2% outlier key channels x10, 128-token residual, 25% + 25% budget, 128
steps), `tiny` (batch 1, 2 heads, head dim 64, prompt 256, 16 steps),
`pyramid-layer16` (layer 16 of the sweep alone), `diffkv` (GQA 40/8, batch 32,
prompt 8192, K8V4/K4V2/prune with Dirichlet(2,5,3) fractions, 64-token
window, 512 steps), `mikv` (GQA 32/8, batch 64, prompt 32768, bf16, INT4 top
20% / INT2 rest, 128-token residual, 1024 steps).

Printed value: decoded tokens per second of the whole step (prefill
included), inputs resident in HBM.  The line also carries decode-only
tokens/s and packed-KV GB/s, prefill TFLOP/s, the roofline of the dominant
kernel, the end-to-end number through host buffers, the CPU oracle baseline
and the SM clocks seen during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload pyramid|llama-layer|tiny|pyramid-layer16|diffkv|mikv]
                  [--batch B] [--decode-steps S]     (smaller cases, for profiling)
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn tokens/s & packed-KV GB/s (% HBM peak); prefill attn TFLOP/s"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
G = 32

WORKLOADS = {
    "llama-layer": dict(policy="minikv", B=1, Hq=32, Hkv=32, D=128, T=4096, steps=128, nr=128,
                        hh=25, rw=25, n_out=3, out_scale=10.0, dtype="f16"),
    "tiny": dict(policy="minikv", B=1, Hq=2, Hkv=2, D=64, T=256, steps=16, nr=0, hh=25, rw=25,
                 n_out=2, out_scale=8.0, dtype="f16"),
    "pyramid-layer16": dict(policy="minikv", B=16, Hq=32, Hkv=32, D=128, T=16384, steps=256, nr=0,
                            hh=None, layer=16, n_layers=32, rw=25, n_out=0, out_scale=1.0,
                            key_std=0.5, dtype="f16"),
    # the whole 32-layer sweep: every layer's budget, one shared synthetic prompt
    "pyramid": dict(policy="minikv", B=16, Hq=32, Hkv=32, D=128, T=16384, steps=256, nr=0,
                    hh=None, layer=None, n_layers=32, rw=25, n_out=0, out_scale=1.0,
                    key_std=0.5, dtype="f16", sweep=True),
    "diffkv": dict(policy="diffkv", B=32, Hq=40, Hkv=8, D=128, T=8192, steps=512, nr=64, n_out=0,
                   out_scale=1.0, dtype="f16", paged=True),
    "mikv": dict(policy="mikv", B=64, Hq=32, Hkv=8, D=128, T=32768, steps=1024, nr=128, n_out=1,
                 out_scale=12.0, dtype="bf16"),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# what decode_attn_qkv launches: single-head MiniKV caches with at least 8 items per resident
# CTA stream (two launches), every other cache runs the cluster kernel
DECODE_KERNELS = ("decode_attn_qkv: decode_stream_kernel + decode_stream_finalize (single-head MiniKV, "
                  "8+ items per resident CTA), else decode_kernel")

KERNEL_SOURCES = {
    "decode_kernel": ["bit_mixed_precision_gb300/csrc/decode.cu", "bit_mixed_precision_gb300/csrc/kvq_common.cuh",
                      "bit_mixed_precision_gb300/csrc/pack_device.cuh"],
}


def sources_sha256(kernel):
    """Hash of the source files that make up a kernel."""
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic(kernel, workload, batch):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json) when it
    was taken on this workload from the kernel's current sources, scaled from the batch it
    was captured at to `batch` (the bytes of every unit are independent); otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel, {}).get(workload)
    if not d or d.get("source_sha256") != sources_sha256(kernel):
        return None
    return d["dram_bytes_per_launch"] * batch / d.get("batch", batch)


def job_ms(step_ms, world, device):
    """The slowest rank's step time (every rank calls this; replicas, no data exchange)."""
    if world <= 1:
        return step_ms
    t = torch.tensor([step_ms], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(world, tokens_per_rank, ms):
    """Whole-job decoded tokens per second: every rank decodes its own replica."""
    return world * tokens_per_rank / (ms / 1e3)


def _budget(wl):
    """(heavy-hitter budget, window) of a MiniKV workload, integer form of the percentages."""
    T = wl["T"]
    w = (T * wl["rw"]) // 100
    if wl.get("hh") is None:
        L, l = wl["n_layers"], wl["layer"]
        k = (T * (40 * (L - 1) - 30 * l)) // (100 * (L - 1))      # 40% at layer 0 down to 10% at L-1
    else:
        k = (T * wl["hh"]) // 100
    return min(k, T - w), w


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the raw samples (the JSON line carries their summary); KVQ_CLOCKS_DIR keeps them
        out_dir = os.environ.get("KVQ_CLOCKS_DIR") or os.path.join(ROOT, "_clocks")
        self.path = os.path.join(out_dir, f"clocks_gpu{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- our arm

class Hot:
    """Device-resident state of one replica of a workload."""

    def __init__(self, wl, dev, seed=0):
        from bit_mixed_precision_gb300 import inputs, kvq
        self.kvq, self.wl, self.dev = kvq, wl, dev
        B, Hq, Hkv, D, T, steps = wl["B"], wl["Hq"], wl["Hkv"], wl["D"], wl["T"], wl["steps"]
        self.dtype = torch.bfloat16 if wl["dtype"] == "bf16" else torch.float16
        self.scale = 1.0 / math.sqrt(D)
        outl = inputs.outlier_channels(Hkv, D, wl["n_out"], seed) if wl["n_out"] else None
        kstd = inputs.lognormal_key_std(Hkv, D, wl["key_std"], seed) if wl.get("key_std") else None
        x = inputs.make_qkv(B, Hq, Hkv, T, D, dtype=self.dtype, seed=seed, device=dev, outliers=outl,
                            outlier_scale=wl["out_scale"], key_std=kstd)
        self.q, self.k, self.v = x.q, x.k, x.v
        self.dec = [inputs.make_decode_step(B, Hq, Hkv, D, t, dtype=self.dtype, seed=seed, device=dev,
                                            outliers=outl, outlier_scale=wl["out_scale"], key_std=kstd)
                    for t in range(steps)]
        pol = wl["policy"]
        nr = wl["nr"]
        if pol == "minikv":
            self.k_hh, self.w = _budget(wl)
            self.n_sel = self.k_hh + self.w
            r0 = self.n_sel if self.n_sel <= nr else nr + (self.n_sel - nr) % G
            cap = ((self.n_sel - r0 + steps) // G + 1) * G
            self.cache = kvq.make_cache(B, Hq, Hkv, D, G, self.dtype, kvq.POLICY_MINIKV,
                                        [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr, device=dev)
            self.kh = torch.full((B * Hkv,), self.k_hh, dtype=torch.int32, device=dev)
            self.idx = torch.empty((B, Hkv, self.n_sel), dtype=torch.int32, device=dev)
            self.nout = torch.empty((B * Hkv,), dtype=torch.int32, device=dev)
            # prefill passes, the build, then every decode call (the flush runs inside it)
            self.launches_per_step = 2 + 1 + steps * kvq.decode_launches(self.cache)
        elif pol == "diffkv":
            f = inputs.dirichlet_fractions(B * Hkv, seed=seed)
            nc = T - nr
            self.n_high = torch.from_numpy(np.floor(f[:, 0] * nc).astype(np.int32)).to(dev)
            self.n_low = torch.from_numpy(np.floor(f[:, 1] * nc).astype(np.int32)).to(dev)
            caps = [int(self.n_high.max()) + steps + G, int(self.n_low.max()) + steps + G]
            pages = None
            if wl.get("paged"):
                # page pools sized for every unit's worst case over the run (its build tokens
                # plus every window exit), instead of the largest unit's capacity for all
                P = kvq.PAGE_TOKENS
                pages = [int(((x.cpu().numpy().astype(np.int64) + steps + P - 1) // P).sum())
                         for x in (self.n_high, self.n_low)]
            self.cache = kvq.make_cache(B, Hq, Hkv, D, G, self.dtype, kvq.POLICY_DIFFKV,
                                        [kvq.TierSpec(8, 4, kvq.AXIS_TOKEN, caps[0]),
                                         kvq.TierSpec(4, 2, kvq.AXIS_TOKEN, caps[1])], nr=nr, device=dev,
                                        pages=pages)
            if pages:
                kvq.pages_init(self.cache)
            self.pool_bytes = self.cache.tier_nbytes()
            self.fixed_bytes = sum(kvq.lib().kvq_tier_bytes(B * Hkv, D, G, s.k_bits, s.v_bits, s.k_axis,
                                                            (c + 31) // 32 * 32, None)
                                   for s, c in zip([kvq.TierSpec(8, 4, 1, 0), kvq.TierSpec(4, 2, 1, 0)], caps))
            self.launches_per_step = (2 + 1 + (1 if wl.get("paged") else 0)
                                      + steps * (kvq.decode_launches(self.cache) + 1))   # + policy step
        else:
            nq = T - nr + steps
            self.cache = kvq.make_cache(B, Hq, Hkv, D, G, self.dtype, kvq.POLICY_MIKV,
                                        [kvq.TierSpec(4, 4, kvq.AXIS_TOKEN, nq // 5 + 64),
                                         kvq.TierSpec(2, 2, kvq.AXIS_TOKEN, nq + 64)],
                                        nr=nr, score_cap=T + steps + 1, hi_den=5, device=dev)
            # decode (and its score update), policy step
            self.launches_per_step = 2 + 1 + steps * (kvq.decode_launches(self.cache) + 1)
        self.o_pre = torch.empty_like(self.q)
        self.lse = torch.empty((B, Hq, T), dtype=torch.float32, device=dev)
        self.cs = torch.empty_like(self.lse)
        self.o_dec = torch.empty((steps, B, Hq, D), dtype=self.dtype, device=dev)
        self.lse_dec = torch.empty((steps, B, Hq), dtype=torch.float32, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        nt = len(self.cache.tiers)
        self.hist = torch.zeros((steps, nt + 1, B * Hkv), dtype=torch.int32, device=dev)
        # the causal half of pass-1 QK^T and PV and of pass-2 QK^T, 2 flops per multiply-add
        self.prefill_flops = 3 * D * T * T * B * Hq

    def prefill_build(self, s):
        kvq, pol = self.kvq, self.wl["policy"]
        kvq.prefill_attn_scores(self.q, self.k, self.v, self.scale,
                                out=(self.o_pre, self.lse, self.cs), stream=s)
        if pol == "minikv":
            # selection + packing + residual in one launch (the prefill-end epilogue)
            kvq.minikv_prefill_build(self.cache, self.k, self.v, self.cs, self.kh, self.w, kmax=self.k_hh,
                                     idx_out=self.idx, stream=s)
        elif pol == "diffkv":
            kvq.requant_demote(self.cache, 0, k_src=self.k, v_src=self.v, colscore=self.cs,
                               n_high=self.n_high, n_low=self.n_low, stream=s)
        else:
            kvq.requant_demote(self.cache, 0, k_src=self.k, v_src=self.v, colscore=self.cs, stream=s)

    def decode(self, t, s):
        qd, kd, vd = self.dec[t]
        self.kvq.decode_attn_qkv(qd, kd, vd, self.cache, self.scale, o=self.o_dec[t],
                                 lse=self.lse_dec[t], stream=s)

    def has_tail(self):
        """DiffKV / MiKV decide a token's tier after each step; MiniKV's flush is part of decode."""
        return self.wl["policy"] != "minikv"

    def tail(self, t, s):
        self.kvq.requant_demote(self.cache, t + 1, stream=s)

    def record_counts(self, t):
        """Tier sizes and residual length as decode step t saw them (outside the timed windows)."""
        for i, tr in enumerate(self.cache.tiers):
            self.hist[t, i].copy_(tr.count)
        self.hist[t, -1].copy_(self.cache.res_len)

    def decode_bytes(self):
        """Algorithmic bytes each decode launch moves: packed codes + fp16 scale/zero of every
        stored token, the full-precision residual (with the new token), q / o / k_new / v_new,
        and for MiKV the cumulative-score read-modify-write of every token."""
        D, Hq, Hkv = self.wl["D"], self.wl["Hq"], self.wl["Hkv"]
        h = self.hist.cpu().numpy().astype(np.int64)
        per = []
        for tr in self.cache.tiers:
            s = tr.spec
            per.append(D * (s.k_bits + s.v_bits) // 8 + 2 * 2 * (D // G) * 2)
        out = []
        for t in range(h.shape[0]):
            packed = sum(int(h[t, i].sum()) * per[i] for i in range(len(per)))
            res = int(h[t, -1].sum() + h.shape[2]) * 2 * D * 2          # before the append, + new
            io = (2 * Hq + 2 * Hkv) * self.wl["B"] * D * 2
            extra = 0
            if self.wl["policy"] == "mikv":
                extra = 8 * (int(h[t, :-1].sum()) + int(h[t, -1].sum() + h.shape[2]))
            out.append(packed + res + io + extra)
        return out, packed


class Sweep:
    """All layers of the pyramid sweep on one GPU: one synthetic prompt shared by the layers,
    one MiniKV cache per layer with that layer's heavy-hitter budget."""

    def __init__(self, wl, dev, seed=0):
        from bit_mixed_precision_gb300 import inputs, kvq
        self.kvq, self.wl = kvq, wl
        B, H, D, T, steps, L = wl["B"], wl["Hq"], wl["D"], wl["T"], wl["steps"], wl["n_layers"]
        self.scale = 1.0 / math.sqrt(D)
        kstd = inputs.lognormal_key_std(H, D, wl["key_std"], seed)
        x = inputs.make_qkv(B, H, H, T, D, seed=seed, device=dev, key_std=kstd)
        self.q, self.k, self.v = x.q, x.k, x.v
        self.o_pre = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        self.cs = torch.empty_like(self.lse)
        self.layers = []
        for l in range(L):
            k_hh, w = _budget(dict(wl, layer=l))
            n_sel = k_hh + w
            r0 = n_sel % G                                    # nr = 0
            cap = ((n_sel - r0 + steps) // G + 1) * G
            cache = kvq.make_cache(B, H, H, D, G, torch.float16, kvq.POLICY_MINIKV,
                                   [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=0, device=dev)
            self.layers.append(dict(k_hh=k_hh, w=w, n_sel=n_sel, r0=r0, cache=cache,
                                    kh=torch.full((B * H,), k_hh, dtype=torch.int32, device=dev),
                                    idx=torch.empty((B, H, n_sel), dtype=torch.int32, device=dev),
                                    nout=torch.empty((B * H,), dtype=torch.int32, device=dev)))
        # decode inputs of one step (the same for every layer), refreshed before each step
        self.dec = [inputs.make_decode_step(B, H, H, D, t, seed=seed, device=dev, key_std=kstd)
                    for t in range(steps)]
        # zeros until the first step is loaded (the capture's warm-up call decodes them)
        self.qd = torch.zeros_like(self.dec[0][0])
        self.kd = torch.zeros_like(self.dec[0][1])
        self.vd = torch.zeros_like(self.dec[0][2])
        self.o_dec = torch.empty((L, B, H, D), dtype=torch.float16, device=dev)
        self.graph = None
        self.prefill_flops = 3 * D * T * T * B * H * L
        self.launches_per_step = sum(2 + 1 + steps * kvq.decode_launches(ly["cache"]) for ly in self.layers)

    def prefill_build(self, s):
        kvq = self.kvq
        for ly in self.layers:
            kvq.prefill_attn_scores(self.q, self.k, self.v, self.scale, out=(self.o_pre, self.lse, self.cs),
                                    stream=s)
            kvq.minikv_prefill_build(ly["cache"], self.k, self.v, self.cs, ly["kh"], ly["w"], kmax=ly["k_hh"],
                                     idx_out=ly["idx"], stream=s)

    def _decode_layers(self, s):
        for l, ly in enumerate(self.layers):
            self.kvq.decode_attn_qkv(self.qd, self.kd, self.vd, ly["cache"], self.scale, o=self.o_dec[l], stream=s)

    def capture(self, s):
        """One decode step of every layer as a CUDA graph (all cache state is on the device)."""
        with torch.cuda.stream(s):
            self._decode_layers(s)                            # first launches: attributes, occupancy
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=s):
            self._decode_layers(s)

    def load_step(self, t, src=None):
        """This step's decode inputs into the graph's input buffers (from `src`, host
        buffers, when given)."""
        qd, kd, vd = src if src is not None else self.dec[t]
        self.qd.copy_(qd, non_blocking=True)
        self.kd.copy_(kd, non_blocking=True)
        self.vd.copy_(vd, non_blocking=True)

    def decode_step(self, t, s):
        self.load_step(t)
        self.graph.replay()

    def decode_bytes(self):
        """Mean algorithmic bytes per decode step (all layers): packed codes + scale/zero of the
        stored tokens and the residual rows, from the flush schedule (nr = 0, G = 32)."""
        wl = self.wl
        B, H, D, steps = wl["B"], wl["Hq"], wl["D"], wl["steps"]
        per_tok = D * 4 // 8 + 2 * 2 * (D // G) * 2
        tot = 0
        for t in range(steps):
            for ly in self.layers:
                packed = ly["n_sel"] - ly["r0"] + G * ((ly["r0"] + t) // G)
                res = (ly["r0"] + t) % G + 1
                tot += (packed * per_tok + res * 2 * D * 2) * B * H + 4 * B * H * D * 2
        return tot / steps

    def e2e(self, s, warmup, reps):
        """The whole step through the public calls from pinned host buffers: H2D of the prompt
        Q/K/V and of every step's decode inputs, D2H of every layer's decode output of every
        step, all inside the timed region."""
        steps, L = self.wl["steps"], len(self.layers)
        pin = lambda t: t.cpu().pin_memory()
        hq, hk, hv = pin(self.q), pin(self.k), pin(self.v)
        hdec = [tuple(pin(x) for x in d) for d in self.dec]
        ho = torch.empty((steps,) + tuple(self.o_dec.shape), dtype=self.o_dec.dtype).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        h2d += sum(x.numel() * x.element_size() for d in hdec for x in d)
        d2h = ho.numel() * ho.element_size()
        times = []
        for it in range(warmup + reps):
            with torch.cuda.stream(s):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                self.q.copy_(hq, non_blocking=True)
                self.k.copy_(hk, non_blocking=True)
                self.v.copy_(hv, non_blocking=True)
                self.prefill_build(s)
                for t in range(steps):
                    self.load_step(t, hdec[t])
                    self.graph.replay()
                    ho[t].copy_(self.o_dec, non_blocking=True)
                b.record(s)
            torch.cuda.synchronize()
            if it >= warmup:
                times.append(a.elapsed_time(b))
        ms = statistics.mean(times)
        return {"value": self.wl["B"] * steps / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps_timed": reps,
                "note": f"{L} layers' decode outputs of each of the {steps} decode steps copied back"}


def _l2_note(wl):
    if wl.get("sweep"):
        return "not flushed: the per-step working set (every layer's cache, about 13 GB) is larger than L2"
    return "flushed (256 MB write) before the prefill and before every decode step; flush time excluded"


def _config(args, wl, world):
    """The config object of the JSON line (identical for both arms)."""
    return {"workload": args.workload, **{k: v for k, v in wl.items() if v is not None},
            "l2": _l2_note(wl), "parallelism": f"replicas x{world}"}


def run_sweep(args, wl, rank, world):
    """Pyramid sweep: each step prefills and builds all layers, then decodes every layer for
    `steps` steps (one CUDA graph of all layers per step).  The working set (every layer's
    cache, about 13 GB) is far larger than L2, so no flush is needed between launches."""
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sw = Sweep(wl, dev, seed=rank)
    s = torch.cuda.Stream(device=dev)
    steps, L = wl["steps"], wl["n_layers"]
    hbm_peak, tf_peak, peak_src = _peaks()

    def one_step():
        """One whole step; event pairs around the prefill + build and around each step's
        graph replay (the decode launches alone, not the input copies)."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 + 2 * steps)]
        with torch.cuda.stream(s):
            ev[0].record(s)
            sw.prefill_build(s)
            ev[1].record(s)
            for t in range(steps):
                sw.load_step(t)
                ev[2 + 2 * t].record(s)
                sw.graph.replay()
                ev[3 + 2 * t].record(s)
        return ev

    with torch.cuda.stream(s):
        sw.prefill_build(s)
    torch.cuda.synchronize()
    sw.capture(s)
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    st = sw.kvq.device_status(s)
    if st:
        raise RuntimeError(f"device status {st} after warm-up")
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    pre_ms = dec_ms = 0.0
    with Clocks(dev.index) as clk:
        t_start.record(s)
        for _ in range(args.steps):
            ev = one_step()
            torch.cuda.synchronize()
            pre_ms += ev[0].elapsed_time(ev[1])
            dec_ms += sum(ev[2 + 2 * t].elapsed_time(ev[3 + 2 * t]) for t in range(steps))
        t_end.record(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    st = sw.kvq.device_status(s)
    if st:
        raise RuntimeError(f"device status {st} after the timed steps")
    step_ms = t_start.elapsed_time(t_end) / args.steps
    ms_max = job_ms(step_ms, world, dev)
    B = wl["B"]
    value = job_value(world, B * steps, ms_max)
    dec_step_ms = dec_ms / args.steps / steps
    dbytes = sw.decode_bytes()
    achieved = dbytes / (dec_step_ms / 1e3) / 1e9
    pre_tf = sw.prefill_flops / (pre_ms / args.steps / 1e3) / 1e12      # includes select + build
    e2e = sw.e2e(s, warmup=1, reps=min(2, args.steps))
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 in, f32 accumulate, packed INT2 cache",
        "data": "synthetic (seeded Gaussian Q/V, keys with LogNormal(0, 0.5) per-channel std; one prompt "
                "shared by the layers)",
        "config": _config(args, wl, world),
        "decode": {"tokens_per_s": B * steps / (dec_ms / args.steps / 1e3),
                   "us_per_layer_step": dec_step_ms * 1e3 / L,
                   "bytes_per_layer_step": dbytes / L, "packed_kv_gbs": achieved,
                   "frac_hbm": achieved / hbm_peak, "launch": "one CUDA graph of every layer per step"},
        "prefill": {"ms_all_layers": pre_ms / args.steps, "tflops_incl_select_build": pre_tf,
                    "frac_tensor": pre_tf / tf_peak},
        "segments_ms_per_step": {"prefill_build": pre_ms / args.steps, "decode": dec_ms / args.steps,
                                 "decode_input_copies_and_gaps": step_ms - (pre_ms + dec_ms) / args.steps},
        "roofline": {"kernel": DECODE_KERNELS, "bound": "hbm", "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": _traffic("decode_kernel", args.workload, B),
                     "per": "launch (one layer's decode, averaged over the 32 layers)",
                     "peak_source": f"{peak_src} hbm_gbs (of measured)" if peak_src == "measured"
                                    else "fallback 6800 GB/s"},
        "roofline_prefill": {"kernel": "prefill_pass1_kernel + prefill_pass2_kernel (+ select, build)",
                             "bound": "tensor", "achieved": pre_tf, "peak": tf_peak, "unit": "TFLOP/s",
                             "frac": pre_tf / tf_peak, "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "e2e": e2e,
        "gpu_launches": sw.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        cb = cpu_baseline(dict(wl, layer=L // 2), args)
        # one layer's oracle cost (layer 16's budget) for each of the layers
        cb["value"] /= L
        cb["seconds_per_step_estimated"] *= L
        cb["sample"] += f", times {L} layers"
        out["cpu_baseline"] = cb
        print(json.dumps(out), flush=True)


def run_ours(args, wl, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    from bit_mixed_precision_gb300 import kvq
    kvq.lib()
    hot = Hot(wl, dev, seed=rank)
    s = torch.cuda.Stream(device=dev)
    steps = wl["steps"]
    hbm_peak, tf_peak, peak_src = _peaks()

    def one_step(rec):
        """Runs one step; returns the event pairs of each timed segment."""
        ev = []
        with torch.cuda.stream(s):
            hot.flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            hot.prefill_build(s)
            e1.record(s)
            ev.append(("prefill", e0, e1))
            for t in range(steps):
                hot.flush.zero_()
                if rec:
                    hot.record_counts(t)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c = torch.cuda.Event(enable_timing=True)
                a.record(s)
                hot.decode(t, s)
                b.record(s)
                ev.append(("decode", a, b))
                if hot.has_tail():
                    hot.tail(t, s)
                    c.record(s)
                    ev.append(("tail", b, c))
        return ev

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    st = kvq.device_status(s)
    if st:
        raise RuntimeError(f"device status {st} after warm-up")
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    seg = {"prefill": 0.0, "decode": 0.0, "tail": 0.0}
    n_dec = 0
    with Clocks(dev.index) as clk:
        for _ in range(args.steps):
            ev = one_step(True)
            torch.cuda.synchronize()
            for name, a, b in ev:
                seg[name] += a.elapsed_time(b)
                n_dec += name == "decode"
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    st = kvq.device_status(s)
    if st:
        raise RuntimeError(f"device status {st} after the timed steps")
    step_ms = sum(seg.values()) / args.steps
    # the two prefill kernels alone, for TFLOP/s
    pre = []
    for _ in range(3):
        with torch.cuda.stream(s):
            hot.flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            kvq.prefill_attn_scores(hot.q, hot.k, hot.v, hot.scale,
                                    out=(hot.o_pre, hot.lse, hot.cs), stream=s)
            b.record(s)
        torch.cuda.synchronize()
        pre.append(a.elapsed_time(b))
    pre_ms = statistics.median(pre)
    B = wl["B"]
    dec_tokens = B * steps
    ms_max = job_ms(step_ms, world, dev)
    value = job_value(world, dec_tokens, ms_max)
    dec_ms_per_launch = seg["decode"] / n_dec
    dbytes, _ = hot.decode_bytes()
    dec_bytes = float(np.mean(dbytes))
    achieved = dec_bytes / (dec_ms_per_launch / 1e3) / 1e9
    pre_tf = hot.prefill_flops / (pre_ms / 1e3) / 1e12
    default = args.workload == "llama-layer" or args.workload == "tiny"
    e2e = run_e2e(hot, s, args, wl) if default else None
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"{wl['dtype']} in, f32 accumulate, packed {'INT2' if wl['policy'] == 'minikv' else ('K8V4/K4V2' if wl['policy'] == 'diffkv' else 'INT4/INT2')} cache",
        "data": "synthetic (seeded Gaussian Q/K/V, outlier key channels)",
        "config": _config(args, wl, world),
        "decode": {"tokens_per_s": dec_tokens / (seg['decode'] / args.steps / 1e3),
                   "us_per_launch": dec_ms_per_launch * 1e3, "bytes_per_launch": dec_bytes,
                   "packed_kv_gbs": achieved, "frac_hbm": achieved / hbm_peak},
        "prefill": {"ms": pre_ms, "tflops": pre_tf, "frac_tensor": pre_tf / tf_peak,
                    "flops_counted": "3*D*T^2 per (batch, query head): the causal half (T^2/2 "
                                     "query-key pairs) of pass-1 QK^T and PV and of pass-2 QK^T, "
                                     "2 flops per multiply-add"},
        "segments_ms_per_step": {k2: v2 / args.steps for k2, v2 in seg.items()},
        "roofline": {"kernel": DECODE_KERNELS, "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": _traffic("decode_kernel", args.workload, wl["B"]),
                     "peak_source": f"{peak_src} hbm_gbs (of measured)" if peak_src == "measured"
                                    else "fallback 6800 GB/s"},
        "roofline_prefill": {"kernel": "prefill_pass1_kernel + prefill_pass2_kernel", "bound": "tensor",
                             "achieved": pre_tf, "peak": tf_peak, "unit": "TFLOP/s",
                             "frac": pre_tf / tf_peak,
                             "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "e2e": e2e,
        **({"pages": {"pool_bytes": hot.pool_bytes, "fixed_capacity_bytes": hot.fixed_bytes,
                      "page_tokens": kvq.PAGE_TOKENS}} if wl.get("paged") else {}),
        "gpu_launches": hot.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(wl, args)
        print(json.dumps(out), flush=True)


def run_e2e(hot, s, args, wl):
    """Same step through the public calls with host buffers: H2D of the prompt Q/K/V and of
    every decode input, D2H of every decode output, all inside the timed region."""
    steps = wl["steps"]
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv = pin(hot.q), pin(hot.k), pin(hot.v)
    hdec = [tuple(pin(x) for x in d) for d in hot.dec]
    ho = torch.empty(hot.o_dec.shape, dtype=hot.o_dec.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    h2d += sum(x.numel() * x.element_size() for d in hdec for x in d)
    d2h = ho.numel() * ho.element_size()
    times = []
    for it in range(args.warmup + args.steps):
        with torch.cuda.stream(s):
            hot.flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            hot.q.copy_(hq, non_blocking=True)
            hot.k.copy_(hk, non_blocking=True)
            hot.v.copy_(hv, non_blocking=True)
            hot.prefill_build(s)
            for t in range(steps):
                for dst, src in zip(hot.dec[t], hdec[t]):
                    dst.copy_(src, non_blocking=True)
                hot.decode(t, s)
                if hot.has_tail():
                    hot.tail(t, s)
            ho.copy_(hot.o_dec, non_blocking=True)
            b.record(s)
        torch.cuda.synchronize()
        if it >= args.warmup:
            times.append(a.elapsed_time(b))
    ms = statistics.mean(times)
    return {"value": wl["B"] * steps / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "L2 not flushed inside this region (the prompt copy itself streams the inputs)"}


# ---------------------------------------------------------------------------- oracle arm

def oracle_step_seconds(wl, seed=0, rows=256, dec_steps=2):
    """Times the CPU oracle on a bounded sample of one step and scales it to the full step.

    Sample: float64 prefill (pass 1 and pass 2) of `rows` query rows of one head, then the
    policy life cycle (build + `dec_steps` decode steps) of one unit.  Scale: rows -> all
    rows of all heads; one unit x dec_steps -> all units x all decode steps.
    """
    from bit_mixed_precision_gb300 import inputs
    from oracle import attention as OA
    from oracle import policies as OP
    from oracle import select as OS
    B, Hq, Hkv, D, T, steps, nr = (wl[k] for k in ("B", "Hq", "Hkv", "D", "T", "steps", "nr"))
    g = Hq // Hkv
    dt = torch.bfloat16 if wl["dtype"] == "bf16" else torch.float16
    scale = 1.0 / math.sqrt(D)
    outl = inputs.outlier_channels(1, D, wl["n_out"], seed) if wl["n_out"] else None
    x = inputs.make_qkv(1, g, 1, T, D, dtype=dt, seed=seed, outliers=outl,
                        outlier_scale=wl["out_scale"])
    qh = [x.q[0, h].float().numpy() for h in range(g)]
    kh, vh = x.k[0, 0].float().numpy(), x.v[0, 0].float().numpy()
    t0 = time.perf_counter()
    sample_rows = np.linspace(0, T - 1, min(rows, T)).astype(np.int64)
    OA.prefill_rows(qh[0], kh, vh, sample_rows, scale)
    t_rows = time.perf_counter() - t0
    t_pre = t_rows / len(sample_rows) * T * 2 * (B * Hq)           # pass 1 + pass 2
    # column scores of the unit (the build needs them); not part of the timed sample
    cs = np.stack([OA.colscore_cols(qh[h], kh, np.arange(T), OA.lse_all_rows(qh[h], kh, scale),
                                    scale) for h in range(g)]).astype(np.float32) if T <= 8192 else \
        np.abs(np.random.default_rng(seed).normal(size=(g, T))).astype(np.float32)
    t1 = time.perf_counter()
    if wl["policy"] == "minikv":
        k_hh, w = _budget(wl)
        unit = OP.MiniKVUnit(kh, vh, OS.select_unit(cs[0], k_hh, w), nr, G)
    elif wl["policy"] == "diffkv":
        nc = T - nr
        unit = OP.DiffKVUnit(kh, vh, cs, int(0.2 * nc), int(0.5 * nc), nr, G)
    else:
        unit = OP.MiKVUnit(kh, vh, cs, nr, G)
    t_build = (time.perf_counter() - t1) * (B * Hkv)
    dec = [inputs.make_decode_step(1, g, 1, D, t, dtype=dt, seed=seed) for t in range(dec_steps)]
    t2 = time.perf_counter()
    for t, (qd, kd, vd) in enumerate(dec):
        unit.step(T + t, qd[0].float().numpy(), kd[0, 0].float().numpy(), vd[0, 0].float().numpy(), scale)
    t_dec = (time.perf_counter() - t2) / dec_steps * (B * Hkv * steps)
    sample = (f"float64 prefill of {len(sample_rows)} rows of 1 of {B * Hq} heads, the cache build "
              f"and {dec_steps} of {steps} decode steps of 1 of {B * Hkv} units, scaled to the full step")
    return t_pre + t_build + t_dec, sample


def cpu_baseline(wl, args):
    torch.set_num_threads(os.cpu_count() or 1)
    secs, sample = oracle_step_seconds(wl)
    return {"value": wl["B"] * wl["steps"] / secs, "unit": UNIT, "cores": _oracle_cores(),
            "kind": "oracle", "sample": sample, "seconds_per_step_estimated": secs}


def _oracle_cores():
    """Threads the oracle's numpy matrix products may use (its Python loops use one)."""
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def run_reference(args, wl, rank, world):
    """The oracle arm: each step times the CPU oracle on a bounded sample of the workload's
    step (see oracle_step_seconds) on the host cores.  ms_per_step is the time of what ran;
    value is the full step's throughput estimated from it (the scale factor is printed)."""
    if rank != 0:
        return
    torch.set_num_threads(os.cpu_count() or 1)
    n_layers = wl["n_layers"] if wl.get("sweep") else 1
    wl_s = dict(wl, layer=wl["n_layers"] // 2) if wl.get("sweep") else wl

    def sample():
        t0 = time.perf_counter()
        est, smp = oracle_step_seconds(wl_s, rows=64, dec_steps=1)
        return time.perf_counter() - t0, est * n_layers, smp

    for _ in range(args.warmup):
        sample()
    ran, est, smp, t0 = [], [], "", time.perf_counter()
    for _ in range(args.steps):
        r, e, smp = sample()
        ran.append(r)
        est.append(e)
    if n_layers > 1:
        smp += f", times {n_layers} layers (layer {wl['n_layers'] // 2}'s budget for each)"
    secs = statistics.mean(est)
    v = wl["B"] * wl["steps"] / secs
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(ran) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 attention, f32 quantiser",
        "data": "synthetic (seeded Gaussian Q/K/V, outlier key channels)",
        "config": _config(args, wl, world),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": _oracle_cores(), "kind": "oracle",
                         "sample": smp},
        "scale_factor": secs / statistics.mean(ran),
        "seconds_per_full_step_estimated": secs,
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t0}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="pyramid", choices=sorted(WORKLOADS))
    # smaller cases of a workload's kernels (profiling): the batch and the decode steps per
    # timed step; the JSON line's config records them
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--decode-steps", type=int, default=None)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    wl = dict(WORKLOADS[args.workload])
    if args.batch is not None:
        wl["B"] = args.batch
    if args.decode_steps is not None:
        wl["steps"] = args.decode_steps
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        (run_sweep if wl.get("sweep") else run_ours)(args, wl, rank, world)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
