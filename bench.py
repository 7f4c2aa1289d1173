"""Benchmark of the compressed-KV-cache attention hot path on one GB300 (or N replicas).

One step = the whole hot path over one batch of synthetic input: two-pass
prefill (output + column scores), heavy-hitter + recent-window selection, the
prefill-end cache build (INT2 packing), then `decode_steps` decode steps
(attention over the packed cache + residual flush).  Default workload: the
LLaMA2-7B-shaped layer (batch 1, 32 heads, head dim 128, prompt 4096, fp16,
2% outlier key channels x10, INT2 groups of 32, 128-token residual, 25% heavy
hitters + 25% window, 128 decode steps).

Printed value: decoded tokens per second of the whole step (prefill included),
inputs resident in HBM.  The line also carries decode-only tokens/s and
packed-KV GB/s, prefill TFLOP/s, the roofline of the dominant kernel, the
end-to-end number through host buffers, the CPU oracle baseline and the SM
clocks seen during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama-layer|pyramid-sweep|diffkv|mikv]
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

WORKLOADS = {
    # name: B, H, D, T, steps, nr, hh%, rw%, outlier channels, outlier scale
    "llama-layer": dict(B=1, H=32, D=128, T=4096, steps=128, nr=128, hh=25, rw=25, n_out=3,
                        out_scale=10.0),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{index}.csv")

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
    """Device-resident state of one replica of the workload."""

    def __init__(self, wl, dev, seed=0):
        from bit_mixed_precision_gb300 import inputs, kvq
        self.kvq = kvq
        self.wl = wl
        B, H, D, T = wl["B"], wl["H"], wl["D"], wl["T"]
        self.scale = 1.0 / math.sqrt(D)
        self.outl = inputs.outlier_channels(H, D, wl["n_out"], seed)
        x = inputs.make_qkv(B, H, H, T, D, seed=seed, device=dev, outliers=self.outl,
                            outlier_scale=wl["out_scale"])
        self.q, self.k, self.v = x.q, x.k, x.v
        self.k_hh = (T * wl["hh"]) // 100
        self.w = (T * wl["rw"]) // 100
        self.n_sel = self.k_hh + self.w
        G, nr, steps = 32, wl["nr"], wl["steps"]
        r0 = self.n_sel if self.n_sel <= nr else nr + (self.n_sel - nr) % G
        cap = ((self.n_sel - r0 + steps) // G + 1) * G
        self.cache = kvq.make_cache(B, H, H, D, G, torch.float16, kvq.POLICY_MINIKV,
                                    [kvq.TierSpec(2, 2, kvq.AXIS_CHANNEL, cap)], nr=nr, device=dev)
        self.kh = torch.full((B * H,), self.k_hh, dtype=torch.int32, device=dev)
        self.dec = [inputs.make_decode_step(B, H, H, D, t, seed=seed, device=dev,
                                            outliers=self.outl, outlier_scale=wl["out_scale"])
                    for t in range(steps)]
        self.o_pre = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        self.cs = torch.empty_like(self.lse)
        self.idx = torch.empty((B, H, self.k_hh + self.w), dtype=torch.int32, device=dev)
        self.nout = torch.empty((B * H,), dtype=torch.int32, device=dev)
        self.o_dec = torch.empty((steps, B, H, D), dtype=torch.float16, device=dev)
        self.lse_dec = torch.empty((steps, B, H), dtype=torch.float32, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        # packed-cache bytes each decode launch reads, from the flush schedule
        self.dec_bytes = []
        n_p, r = self.n_sel - r0, r0
        per_tok = D * (2 + 2) // 8 + 2 * 2 * (D // G) * 2   # INT2 K+V codes + fp16 s/z
        for t in range(steps):
            r += 1
            self.dec_bytes.append(B * H * (n_p * per_tok + r * 2 * D * 2 + 4 * D * 2))
            if r == nr + G:
                n_p, r = n_p + G, r - G
        self.prefill_flops = 3 * D * T * T * B * H            # QK^T + PV (pass 1) + QK^T (pass 2)
        self.launches_per_step = 2 + 1 + 3 + 2 * steps

    def prefill_select_build(self, s):
        kvq = self.kvq
        kvq.prefill_attn_scores(self.q, self.k, self.v, self.scale,
                                out=(self.o_pre, self.lse, self.cs), stream=s)
        kvq.select_tokens(self.cs, self.kh, self.w, kmax=self.k_hh, out=(self.idx, self.nout),
                          stream=s)
        kvq.requant_demote(self.cache, 0, k_src=self.k, v_src=self.v, sel_idx=self.idx,
                           n_sel=self.n_sel, stream=s)

    def decode(self, t, s):
        qd, kd, vd = self.dec[t]
        self.kvq.decode_attn_qkv(qd, kd, vd, self.cache, self.scale, o=self.o_dec[t],
                                 lse=self.lse_dec[t], stream=s)

    def tail(self, t, s):
        self.kvq.requant_demote(self.cache, t + 1, stream=s)


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
        """Runs one step; when rec, returns the event pairs of each timed segment."""
        ev = []
        with torch.cuda.stream(s):
            hot.flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            hot.prefill_select_build(s)
            e1.record(s)
            ev.append(("prefill", e0, e1))
            for t in range(steps):
                hot.flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c = torch.cuda.Event(enable_timing=True)
                a.record(s)
                hot.decode(t, s)
                b.record(s)
                hot.tail(t, s)
                c.record(s)
                ev.append(("decode", a, b))
                ev.append(("tail", b, c))
        return ev

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    st = kvq.device_status(s)
    if st:
        raise RuntimeError(f"device status {st} after warm-up")
    # separate prefill-kernel timing for the prefill roofline
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
    if world > 1:
        torch.distributed.barrier()
    step_ms = sum(seg.values()) / args.steps
    # prefill kernels alone (both passes), for TFLOP/s
    pre = []
    for _ in range(5):
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
    ms_max = step_ms
    if world > 1:
        t = torch.tensor([step_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_max = float(t.item())
    value = world * dec_tokens / (ms_max / 1e3)
    dec_ms_per_launch = seg["decode"] / n_dec
    dec_bytes = float(np.mean(hot.dec_bytes))
    achieved = dec_bytes / (dec_ms_per_launch / 1e3) / 1e9
    e2e = run_e2e(hot, s, args, wl)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16 in, fp32 accumulate, INT2 cache",
        "data": "synthetic (seeded Gaussian Q/K/V, outlier key channels)",
        "config": {"workload": args.workload, "batch": B, "heads": wl["H"], "head_dim": wl["D"],
                   "prompt": wl["T"], "decode_steps": steps, "kv_bits": 2, "group": 32,
                   "residual": wl["nr"], "budget": f"{wl['hh']}% heavy hitters + {wl['rw']}% window",
                   "l2": "flushed (256 MB write) before the prefill and before every decode step; "
                         "flush time excluded", "parallelism": f"replicas x{world}"},
        "decode": {"tokens_per_s": dec_tokens / (seg['decode'] / args.steps / 1e3),
                   "us_per_launch": dec_ms_per_launch * 1e3, "packed_kv_gbs": achieved,
                   "frac_hbm": achieved / hbm_peak},
        "prefill": {"ms": pre_ms, "tflops": hot.prefill_flops / (pre_ms / 1e3) / 1e12,
                    "frac_tensor": hot.prefill_flops / (pre_ms / 1e3) / 1e12 / tf_peak,
                    "flops_counted": "3*D*T^2 per (batch, head): pass-1 QK^T and PV, pass-2 QK^T "
                                     "(dense count, the causal half is not subtracted)"},
        "segments_ms_per_step": {k2: v2 / args.steps for k2, v2 in seg.items()},
        "roofline": {"kernel": "decode_kernel (decode_attn_qkv)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": None,
                     "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": e2e,
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
            hot.prefill_select_build(s)
            for t in range(steps):
                for dst, src in zip(hot.dec[t], hdec[t]):
                    dst.copy_(src, non_blocking=True)
                hot.decode(t, s)
                hot.tail(t, s)
            ho.copy_(hot.o_dec, non_blocking=True)
            b.record(s)
        torch.cuda.synchronize()
        if it >= args.warmup:
            times.append(a.elapsed_time(b))
    ms = statistics.mean(times)
    return {"value": wl["B"] * steps / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "L2 not flushed inside this region (the prompt copy itself streams 100 MB)"}


# ---------------------------------------------------------------------------- oracle arm

def oracle_step_seconds(wl, seed=0, heads=2, dec_units=2, dec_steps=8):
    """Times the CPU oracle on a bounded sample of one step and scales it to the full step.

    Sample: prefill (both passes, float64) of `heads` heads, then the MiniKV life cycle of
    `dec_units` units for `dec_steps` decode steps.  Scale: heads -> all heads; units x steps ->
    all units x all decode steps.
    """
    from bit_mixed_precision_gb300 import inputs
    from oracle import attention as OA
    from oracle import policies as OP
    from oracle import select as OS
    B, H, D, T, steps, nr = wl["B"], wl["H"], wl["D"], wl["T"], wl["steps"], wl["nr"]
    scale = 1.0 / math.sqrt(D)
    outl = inputs.outlier_channels(H, D, wl["n_out"], seed)
    x = inputs.make_qkv(1, heads, heads, T, D, seed=seed, outliers=outl[:heads],
                        outlier_scale=wl["out_scale"])
    k_hh, w = OS.budget(T, wl["hh"], wl["rw"])
    t0 = time.perf_counter()
    sels = []
    for h in range(heads):
        _, _, cs = OA.prefill_head(x.q[0, h].float().numpy(), x.k[0, h].float().numpy(),
                                   x.v[0, h].float().numpy(), scale)
        sels.append(OS.select_unit(cs.astype(np.float32), k_hh, w))
    t_pre = (time.perf_counter() - t0) / heads * (B * H)
    dec_in = [inputs.make_decode_step(1, heads, heads, D, t, seed=seed) for t in range(dec_steps)]
    t_build = t_dec = 0.0
    for u in range(dec_units):
        h = u % heads
        t1 = time.perf_counter()
        unit = OP.MiniKVUnit(x.k[0, h].float().numpy(), x.v[0, h].float().numpy(), sels[h], nr, 32)
        t2 = time.perf_counter()
        for t in range(dec_steps):
            qd, kd, vd = dec_in[t]
            unit.step(T + t, qd[0, h:h + 1].float().numpy(), kd[0, h].float().numpy(),
                      vd[0, h].float().numpy(), scale)
        t_build += t2 - t1
        t_dec += time.perf_counter() - t2
    t_build = t_build / dec_units * (B * H)
    t_dec = t_dec / (dec_units * dec_steps) * (B * H * steps)
    sample = (f"float64 prefill of {heads} of {B * H} heads + MiniKV decode of {dec_units} units x "
              f"{dec_steps} of {steps} steps, scaled to the full step")
    return t_pre + t_build + t_dec, sample


def cpu_baseline(wl, args):
    torch.set_num_threads(os.cpu_count() or 1)
    secs, sample = oracle_step_seconds(wl)
    return {"value": wl["B"] * wl["steps"] / secs, "unit": UNIT, "cores": torch.get_num_threads(),
            "kind": "oracle", "sample": sample, "seconds_per_step_estimated": secs}


def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    torch.set_num_threads(os.cpu_count() or 1)
    for _ in range(args.warmup):
        oracle_step_seconds(wl, heads=1, dec_units=1, dec_steps=2)
    est, t0 = [], time.perf_counter()
    sample = ""
    for _ in range(args.steps):
        s, sample = oracle_step_seconds(wl, heads=1, dec_units=1, dec_steps=2)
        est.append(s)
    secs = statistics.mean(est)
    v = wl["B"] * wl["steps"] / secs
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 quantiser",
        "data": "synthetic (seeded Gaussian Q/K/V, outlier key channels)",
        "config": {"workload": args.workload, **{k: wl[k] for k in ("B", "H", "D", "T", "steps", "nr")}},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": torch.get_num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t0}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama-layer", choices=sorted(WORKLOADS))
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
    else:
        run_ours(args, wl, rank, world)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
