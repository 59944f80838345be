#!/usr/bin/env python3
"""Benchmark: FP8 paged decode attention on the Llama-3.1-8B-shaped 128K
workload -- KV GB/s (% of HBM peak) and us/step vs context length.

One step = one decode step of a 32-layer Llama-3.1-8B-shaped model at batch
1 and 131,072 tokens of context: for each layer, the new token's K/V is
quantized into that layer's paged FP8 cache and paged decode attention
(split-KV partial + LSE combine) reads the whole cache, in one
kvq_paged_decode_attention_append call.  Each layer has its own cache
(32 x 256 MiB = 8 GiB), so every step streams from HBM (inputs larger than
L2).  Inputs are seeded synthetic bf16 N(0,1) with 4 outlier channels per
KV head (x20) and amax/448 scales.

Beside the headline, a single-GPU run measures the other decode
configurations (tiny 512-token latency floor; batch 8 at ~20K tokens;
the 24-layer hybrid full / sliding-window stack), chunked prefill, a
context sweep, the BF16 / E5M2 / per-token cache formats, the
accumulation ablation, and the CPU oracle on every configuration; each leg
carries the SM clocks sampled while it ran.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) the KV heads are sharded over the ranks (rank r
holds KV heads [8r/N, 8(r+1)/N) and their query heads, of N sequences, so
each rank streams the single-GPU step's bytes); there is no collective on
the data path, and rank 0 prints the whole-job throughput over the slowest
rank.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 paged decode attn: KV GB/s (% HBM peak) and µs/step vs context length"
LAYERS = 32
CONTEXT = 131072
HQ, HKV, D, P = 32, 8, 128, 16
FALLBACK_HBM_GBS = 6800.0
# cache layout of every leg: one paired allocation per layer (each (block,
# KV head) pair's K page followed by its V page), or, with
# --separate-caches, separate K and V allocations
PAIRED = True


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-e5m2", action="store_true")
    ap.add_argument("--no-per-token", action="store_true")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the tiny, concurrency-8 and hybrid legs")
    ap.add_argument("--prefill-head-dim", type=int, choices=[128, 256], default=128,
                    help="head dim of the prefill leg (256 runs single-level accumulation)")
    ap.add_argument("--separate-caches", action="store_true",
                    help="separate K and V allocations instead of the paired layout")
    ap.add_argument("--layers", type=int, default=32,
                    help="layers per step (fewer only for small profiling runs; the metric uses 32)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(ms, dist=None, device="cpu"):
    """The slowest rank's duration: the job is done when every rank is."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, step_bytes, steps, total_ms):
    """Whole-job GB/s: every rank's steps (weak scaling) over the slowest rank's time."""
    return world * step_bytes * steps / (total_ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def decode_traffic():
    """DRAM bytes per partial-kernel launch from the committed ncu record,
    or None when the kernel source changed since the counters were taken or
    they were taken on the other cache layout."""
    import hashlib
    tf = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        rec = json.load(open(tf))
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    except (OSError, ValueError, KeyError):
        return None
    if hashlib.sha256(src).hexdigest() != rec.get("source_sha256"):
        return None
    if rec.get("cache_layout") != ("paired" if PAIRED else "separate"):
        return None
    return rec.get("traffic_bytes_per_launch")


def decode_bytes(context, batch=1, hq=HQ, hkv=HKV, d=D):
    """Algorithmic bytes of one decode call: FP8 K + V of the attended
    tokens, per-head K and V scales, q and out (bf16)."""
    return 2 * batch * context * hkv * d + 2 * hkv * 4 + 2 * batch * hq * d * 2


def decode_bytes_lengths(lengths, hq, hkv, d, window=-1, esize=1):
    """Algorithmic bytes of one decode call over sequences of the given
    lengths: K and V of the attended tokens (the last `window` of each for a
    sliding-window layer) at `esize` bytes per element, the per-head K and V
    scales of an FP8 cache (none for BF16), q read and out written (bf16)."""
    attended = sum(min(L, window) if window > 0 else L for L in lengths)
    scales = 2 * hkv * 4 if esize == 1 else 0
    return 2 * attended * hkv * d * esize + scales + 2 * len(lengths) * hq * d * 2


def hybrid_step_bytes(batch=8, context=32768, hq=64, hkv=8, d=64, layers=24, window=128):
    """One decode step of the hybrid stack: layers alternate sliding-window
    BF16 (even) and full-attention FP8 (odd)."""
    full = decode_bytes_lengths([context] * batch, hq, hkv, d)
    sw = decode_bytes_lengths([context] * batch, hq, hkv, d, window=window, esize=2)
    return (layers // 2) * (full + sw), full, sw


def cache_write_bytes(tokens, hkv=HKV, d=D):
    """One token's K and V in (bf16) and out (FP8)."""
    return tokens * hkv * d * (2 * 2 + 2 * 1)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ setup ---
def build_workload(device, seed, batch=1, q_heads=HQ, kv_heads=HKV):
    """32 layer caches of `batch` sequences of 131,072 cached tokens (the
    last one is re-written by every step) over `kv_heads` KV heads, per-layer
    q and new-token K/V, one shared block table.  One rank of a head-sharded
    job holds its KV heads of every sequence: batch N with 8 / N heads keeps
    the bytes per rank (8 GiB) of the single-GPU workload (batch 1, 8 heads)."""
    import torch

    import fp8_kv_cache_reshape_gb300 as kvq
    import workloads as W

    g = W.generator(seed)
    bt, num_blocks = W.paged_layout([CONTEXT] * batch, P, g)
    bt_d = bt.to(device)
    pos = torch.arange(CONTEXT, dtype=torch.int64)
    slots = [W.slots_for(bt, b, pos, P).to(device) for b in range(batch)]
    layers = []
    chunk = 16384
    st = torch.zeros(1, dtype=torch.int32, device=device)
    for l in range(LAYERS):
        gl = W.generator(seed * 1000 + l, device=device)
        ch = W.outlier_channels(kv_heads, D, 4, W.generator(seed * 1000 + l))
        kd, vd = kvq.alloc_kv_cache(num_blocks, kv_heads, D, device=device, fill=0, paired=PAIRED)
        seqs = []
        amax_k = torch.zeros(kv_heads, device=device)
        amax_v = torch.zeros(kv_heads, device=device)
        for b in range(batch):
            k = W.apply_outliers(W.randn_bf16((CONTEXT, kv_heads, D), gl, device=device), ch)
            v = W.apply_outliers(W.randn_bf16((CONTEXT, kv_heads, D), gl, device=device), ch)
            amax_k = torch.maximum(amax_k, k.float().abs().amax(dim=(0, 2)))
            amax_v = torch.maximum(amax_v, v.float().abs().amax(dim=(0, 2)))
            seqs.append((k, v))
        ks = (amax_k / W.E4M3_MAX).contiguous()  # caller-side calibration: amax / 448 per head
        vs = (amax_v / W.E4M3_MAX).contiguous()
        for b, (k, v) in enumerate(seqs):
            for t0 in range(0, CONTEXT - 1, chunk):
                t1 = min(CONTEXT - 1, t0 + chunk)
                kvq.kvq_reshape_and_cache(k[t0:t1].contiguous(), v[t0:t1].contiguous(),
                                          slots[b][t0:t1].contiguous(), kd, vd, ks, vs, dev_status=st)
        layers.append(dict(kd=kd, vd=vd, ks=ks, vs=vs,
                           k_new=torch.stack([k[CONTEXT - 1] for k, _ in seqs]).contiguous(),
                           v_new=torch.stack([v[CONTEXT - 1] for _, v in seqs]).contiguous(),
                           q=W.randn_bf16((batch, q_heads, D), gl, device=device),
                           out=torch.empty((batch, q_heads, D), dtype=torch.bfloat16, device=device)))
        del seqs
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "cache fill reported a device fault"
    # a step's inputs (every layer's q and new K/V) and outputs live in one
    # staging buffer each, as a serving loop would keep them, so that the
    # end-to-end step moves them with one copy each way; the layers' tensors
    # are views into them (offsets multiples of 2 KiB)
    names_in = ("q", "k_new", "v_new")
    n_in = sum(layers[0][n].numel() for n in names_in)
    io_in = torch.empty(LAYERS * n_in, dtype=torch.bfloat16, device=device)
    io_out = torch.empty(LAYERS * layers[0]["out"].numel(), dtype=torch.bfloat16, device=device)
    off_in = off_out = 0
    for ly in layers:
        for n in names_in:
            t = ly[n]
            view = io_in[off_in:off_in + t.numel()].view(t.shape)
            view.copy_(t)
            ly[n] = view
            off_in += t.numel()
        o = ly["out"]
        ly["out"] = io_out[off_out:off_out + o.numel()].view(o.shape)
        off_out += o.numel()
    ws_bytes = kvq.kvq_decode_workspace_size(batch, q_heads, kv_heads, D, bt.shape[1])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    return dict(layers=layers, bt=bt_d, num_blocks=num_blocks, io_in=io_in, io_out=io_out,
                slot_new=torch.stack([sl[CONTEXT - 1] for sl in slots]).contiguous(),
                seq=torch.full((batch,), CONTEXT, dtype=torch.int32, device=device), ws=ws, status=st,
                batch=batch, q_heads=q_heads, kv_heads=kv_heads)


def run_step(wl, seq=None, decode_only=False, two_calls=False):
    """One decode step over all layers (enqueued on the current stream): per
    layer the new token's cache write and the decode call, fused into
    kvq_paged_decode_attention_append (two_calls: kvq_reshape_and_cache, then
    kvq_paged_decode_attention; decode_only: the decode call alone)."""
    import fp8_kv_cache_reshape_gb300 as kvq
    seq = wl["seq"] if seq is None else seq
    for ly in wl["layers"]:
        if not (decode_only or two_calls):
            kvq.kvq_paged_decode_attention_append(ly["q"], ly["k_new"], ly["v_new"], wl["slot_new"], ly["kd"],
                                                  ly["vd"], ly["ks"], ly["vs"], wl["bt"], seq, ly["out"],
                                                  num_blocks=wl["num_blocks"], sm_scale=1.0 / math.sqrt(D),
                                                  workspace=wl["ws"], dev_status=wl["status"])
            continue
        if two_calls:
            kvq.kvq_reshape_and_cache(ly["k_new"], ly["v_new"], wl["slot_new"], ly["kd"], ly["vd"], ly["ks"],
                                      ly["vs"], dev_status=wl["status"])
        kvq.kvq_paged_decode_attention(ly["q"], ly["kd"], ly["vd"], ly["ks"], ly["vs"], wl["bt"], seq, ly["out"],
                                       num_blocks=wl["num_blocks"], sm_scale=1.0 / math.sqrt(D),
                                       workspace=wl["ws"], dev_status=wl["status"])


def capture(fn):
    """CUDA graph of everything fn() enqueues (run once eagerly first)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, reps):
    """Milliseconds for `reps` back-to-back replays (CUDA events on the
    current stream, synchronized on both sides)."""
    import torch
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(reps):
        g.replay()
    ev1.record()
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


def time_eager(fn, reps):
    import torch
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(reps):
        fn()
    ev1.record()
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


def e2e_setup(wl):
    """Pinned host copies of the step's inputs (every layer's q and new K/V,
    one staging buffer) and outputs, and the step with its host<->device
    copies: one host-to-device copy before the layers, one device-to-host
    copy after them."""
    import torch
    host_in = wl["io_in"].cpu().pin_memory()
    host_out = torch.empty(wl["io_out"].shape, dtype=wl["io_out"].dtype).pin_memory()
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()

    def one():
        wl["io_in"].copy_(host_in, non_blocking=True)
        run_step(wl)
        host_out.copy_(wl["io_out"], non_blocking=True)

    return one, h2d, d2h


def context_sweep(wl, g_dec, reps=10):
    """us per layer of the decode call at shorter contexts over the same
    caches (seq_len = L attends to the first L cached tokens)."""
    rows = []
    for L in (4096, 8192, 16384, 32768, 65536, 131072):
        wl["seq"].fill_(L)
        g_dec.replay()
        us = time_graph(g_dec, reps) * 1e3 / (reps * LAYERS)
        rows.append({"context": L, "us_per_layer_decode": round(us, 3),
                     "kv_gbs": round(decode_bytes(L) / (us * 1e-6) / 1e9, 1)})
    wl["seq"].fill_(CONTEXT)
    xs = [r["context"] for r in rows]
    ys = [r["us_per_layer_decode"] for r in rows]
    n = len(xs)
    mx, my = sum(xs) / n, sum(ys) / n
    slope = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sum((x - mx) ** 2 for x in xs)
    icpt = my - slope * mx
    return {"points": rows, "fit_us_per_token": slope, "fit_intercept_us": round(icpt, 3),
            "slope_kv_gbs": round(2 * HKV * D / (slope * 1e-6) / 1e9, 1)}


# ------------------------------------------------- BF16 cache comparison ---
BF16_LAYERS = 8


def format_compare(fp8_sweep, device, cache_dtype, reps=20, per_token=False, accumulation=None):
    """The same decode on another cache format over 8 distinct 128K layer
    caches: us per layer vs context, the linear fit, and the slope ratio and
    break-even context against the FP8 E4M3 sweep.  For the BF16 cache (the
    "skip layers" format) this is the vLLM blog's ITL-slope comparison at
    kernel level; the E5M2 cache reads the same bytes as E4M3.  per_token:
    dynamic per-token scales (kvq_reshape_and_cache_per_token and the
    matching decode; the scales ride in the V pages' tails); the scale
    bytes count toward GB/s.  accumulation:
    "single_level" for the accumulation ablation."""
    import torch
    import fp8_kv_cache_reshape_gb300 as kvq
    import workloads as W
    esz = 2 if cache_dtype == "bf16" else 1
    g = W.generator(501)
    bt, nb = W.paged_layout([CONTEXT], P, g)
    slots = W.slots_for(bt, 0, torch.arange(CONTEXT, dtype=torch.int64), P).to(device)
    layers = []
    for l in range(BF16_LAYERS):
        gl = W.generator(502 * 1000 + l, device=device)
        kd, vd = kvq.alloc_kv_cache(nb, HKV, D, cache_dtype=cache_dtype, device=device, fill=0,
                                    per_token=per_token, paired=PAIRED)
        ks = vs = None
        if esz == 1 and not per_token:  # unit-variance data: per-head scale amax / M taken from one chunk
            probe = W.randn_bf16((16384, HKV, D), gl, device=device)
            ks = W.calibrate_amax(probe, W.E5M2_MAX if cache_dtype == "fp8_e5m2" else W.E4M3_MAX).to(device)
            vs = ks.clone()
        for t0 in range(0, CONTEXT, 16384):
            k = W.randn_bf16((16384, HKV, D), gl, device=device)
            v = W.randn_bf16((16384, HKV, D), gl, device=device)
            if per_token:
                kvq.kvq_reshape_and_cache_per_token(k, v, slots[t0:t0 + 16384].contiguous(), kd, vd,
                                                    cache_dtype=cache_dtype)
            else:
                kvq.kvq_reshape_and_cache(k, v, slots[t0:t0 + 16384].contiguous(), kd, vd, ks, vs,
                                          cache_dtype=cache_dtype)
        layers.append(dict(kd=kd, vd=vd, ks=ks, vs=vs, q=W.randn_bf16((1, HQ, D), gl, device=device),
                           out=torch.empty((1, HQ, D), dtype=torch.bfloat16, device=device)))
    btd = bt.to(device)
    seq = torch.tensor([CONTEXT], dtype=torch.int32, device=device)
    ws = torch.empty(kvq.kvq_decode_workspace_size(1, HQ, HKV, D, bt.shape[1]), dtype=torch.uint8, device=device)

    def run():
        for ly in layers:
            if per_token:
                kvq.kvq_paged_decode_attention_per_token(ly["q"], ly["kd"], ly["vd"], btd, seq, ly["out"],
                                                         num_blocks=nb, sm_scale=1.0 / math.sqrt(D),
                                                         cache_dtype=cache_dtype, workspace=ws)
            else:
                kvq.kvq_paged_decode_attention(ly["q"], ly["kd"], ly["vd"], ly["ks"], ly["vs"], btd, seq, ly["out"],
                                               num_blocks=nb, sm_scale=1.0 / math.sqrt(D), cache_dtype=cache_dtype,
                                               workspace=ws, accumulation=accumulation)

    gr = capture(run)
    rows = []
    for L in (4096, 8192, 16384, 32768, 65536, 131072):
        seq.fill_(L)
        gr.replay()
        us = time_graph(gr, reps) * 1e3 / (reps * BF16_LAYERS)
        kvb = 2 * L * HKV * (D * esz + (4 if per_token else 0))
        rows.append({"context": L, "us_per_layer_decode": round(us, 3), "kv_gbs": round(kvb / (us * 1e-6) / 1e9, 1)})
    xs = [r["context"] for r in rows]
    ys = [r["us_per_layer_decode"] for r in rows]
    n = len(xs)
    mx, my = sum(xs) / n, sum(ys) / n
    slope = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sum((x - mx) ** 2 for x in xs)
    icpt = my - slope * mx
    out = {"cache_dtype": cache_dtype, "per_token_scales": per_token, "accumulation": accumulation or "two_level",
           "points": rows, "fit_us_per_token": slope,
           "fit_intercept_us": round(icpt, 3),
           "slope_kv_gbs": round(2 * HKV * (D * esz + (4 if per_token else 0)) / (slope * 1e-6) / 1e9, 1)}
    if fp8_sweep:
        s8, i8 = fp8_sweep["fit_us_per_token"], fp8_sweep["fit_intercept_us"]
        out["slope_ratio_fp8_over_this"] = round(s8 / slope, 4)
        out["break_even_tokens"] = round((i8 - icpt) / (slope - s8)) if slope > s8 else None
    return out


# -------------------------------------------------------------- prefill ---
PF_NEW, PF_CACHED = 4096, 28672


def prefill_flops(new=PF_NEW, cached=PF_CACHED, hq=HQ, d=D):
    """4 * D FLOPs (QK^T and P.V, 2 each) per attended (query, key) pair;
    query i attends to cached + i + 1 keys."""
    pairs = new * cached + new * (new + 1) // 2
    return pairs * hq * 4 * d


def prefill_leg(device, reps=10, accumulation=None, head_dim=D, cache_dtype="fp8_e4m3", per_token=False):
    """Chunked causal prefill of 4,096 new tokens on 28,672 cached FP8
    tokens (32/8 heads, head_dim 128, or 256; E4M3 or E5M2 cache; per-head
    or, with per_token, per-token scales): TFLOP/s of kvq_prefill_attention
    (kvq_prefill_attention_per_token)."""
    import torch
    import fp8_kv_cache_reshape_gb300 as kvq
    import workloads as W
    g = W.generator(77)
    L = PF_NEW + PF_CACHED
    bt, nb = W.paged_layout([L], P, g)
    slots = W.slots_for(bt, 0, torch.arange(L), P).to(device)
    gd = W.generator(78, device=device)
    k = W.randn_bf16((L, HKV, head_dim), gd, device=device)
    v = W.randn_bf16((L, HKV, head_dim), gd, device=device)
    q = W.randn_bf16((PF_NEW, HQ, head_dim), gd, device=device)
    fmt_max = W.E5M2_MAX if cache_dtype == "fp8_e5m2" else W.E4M3_MAX
    ks, vs = W.calibrate_amax(k, fmt_max), W.calibrate_amax(v, fmt_max)
    qs = (q.float().abs().amax() / 448.0).reshape(1).to(torch.float32)
    kd, vd = kvq.alloc_kv_cache(nb, HKV, head_dim, cache_dtype=cache_dtype, device=device, fill=0,
                                per_token=per_token, paired=PAIRED)
    if per_token:
        kvq.kvq_reshape_and_cache_per_token(k, v, slots, kd, vd, cache_dtype=cache_dtype)
    else:
        kvq.kvq_reshape_and_cache(k, v, slots, kd, vd, ks, vs, cache_dtype=cache_dtype)
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=device)
    kvq.kvq_quantize_query(q, q8, qs)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=device)
    btd = bt.to(device)
    cu = torch.tensor([0, PF_NEW], dtype=torch.int32, device=device)
    sl = torch.tensor([L], dtype=torch.int32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)

    def call():
        if per_token:
            kvq.kvq_prefill_attention_per_token(q8, qs, kd, vd, btd, cu, sl, out, max_q_tokens=PF_NEW,
                                                sm_scale=1.0 / math.sqrt(head_dim), cache_dtype=cache_dtype,
                                                dev_status=st)
            return
        kvq.kvq_prefill_attention(q8, qs, kd, vd, ks, vs, btd, cu, sl, out, max_q_tokens=PF_NEW,
                                  sm_scale=1.0 / math.sqrt(head_dim), dev_status=st, accumulation=accumulation,
                                  cache_dtype=cache_dtype)

    for _ in range(3):
        call()
    ms = time_eager(call, reps) / reps
    assert int(st.item()) == 0, "prefill reported a device fault"
    peaks, src = measured_peaks()
    bf16 = float(peaks.get("bf16_tflops", 1900.0))
    fp8_peak = 2.0 * bf16  # nominal FP8:BF16 dense ratio 4.5 : 2.25
    flops = prefill_flops(d=head_dim)
    tf = flops / (ms * 1e-3) / 1e12
    name = ("llama31_8b_chunked_prefill_4k_on_28k" + ("" if head_dim == 128 else f"_head_dim_{head_dim}") +
            ("" if cache_dtype == "fp8_e4m3" else "_" + cache_dtype) + ("_per_token_scales" if per_token else ""))
    return {"workload": name, "ms": round(ms, 4), "flops": flops, "head_dim": head_dim, "cache_dtype": cache_dtype,
            "per_token_scales": per_token,
            "accumulation": accumulation or ("two_level" if head_dim == 128 else "single_level"),
            "bound": "tensor", "achieved": round(tf, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
            "frac": round(tf / fp8_peak, 4),
            "peak_source": f"{src} bf16_tflops x 2 (nominal FP8:BF16 dense ratio)",
            "exps": PF_NEW * PF_CACHED * HQ + PF_NEW * (PF_NEW + 1) // 2 * HQ}


# --------------------------------------------- the other decode configurations ---
def clocked(gpu, fn, *a, **kw):
    """Run one bench leg under its own clock sampler; the leg's dict gets the
    sampled clocks and, per timed figure, time x median SM MHz (so that legs
    measured at different clocks can be compared)."""
    with ClockSampler(gpu) as clk:
        out = fn(*a, **kw)
    if isinstance(out, dict):
        c = clk.summary()
        out["clocks"] = c
        if c.get("sm_mhz"):
            for key in ("us_per_call", "us_per_step", "ms"):
                if out.get(key) is not None:
                    out[key + "_x_mhz"] = round(out[key] * c["sm_mhz"], 1)
    return out


def _hbm_peak():
    peaks, src = measured_peaks()
    return float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS)), src


def _fill_decode_cache(kvq, lengths, bt, num_blocks, hkv, d, gen, device, cache_dtype="fp8_e4m3",
                       unit_scales=False):
    """A paged cache holding every position of every sequence (K, V ~ N(0,1)
    rounded to bf16 on the device; FP8: per-head amax/448 scales, or 1.0
    with unit_scales)."""
    import torch
    import workloads as W
    kd, vd = kvq.alloc_kv_cache(num_blocks, hkv, d, cache_dtype=cache_dtype, device=device, fill=0,
                                paired=PAIRED)
    ks = vs = None
    chunks = []
    for b, L in enumerate(lengths):
        pos = torch.arange(L, dtype=torch.int64)
        chunks.append((W.slots_for(bt, b, pos, P).to(device), L))
    if cache_dtype != "bf16":  # caller-side calibration over the whole layer
        amax_k = torch.zeros(hkv, device=device)
        amax_v = torch.zeros(hkv, device=device)
    data = []
    for slots, L in chunks:
        k = W.randn_bf16((L, hkv, d), gen, device=device)
        v = W.randn_bf16((L, hkv, d), gen, device=device)
        data.append((slots, k, v))
        if cache_dtype != "bf16":
            amax_k = torch.maximum(amax_k, k.float().abs().amax(dim=(0, 2)))
            amax_v = torch.maximum(amax_v, v.float().abs().amax(dim=(0, 2)))
    if cache_dtype != "bf16":
        ks = (amax_k / W.E4M3_MAX).float().contiguous()
        vs = (amax_v / W.E4M3_MAX).float().contiguous()
        if unit_scales:
            ks = torch.ones_like(ks)
            vs = torch.ones_like(vs)
    for slots, k, v in data:
        kvq.kvq_reshape_and_cache(k, v, slots, kd, vd, ks, vs, cache_dtype=cache_dtype)
    return kd, vd, ks, vs


def tiny_leg(device, calls=64, reps=50):
    """The tiny configuration (1 sequence of 512 tokens, 4 query / 1 KV head,
    head_dim 64, scales 1.0): the latency floor of one decode call.  Its
    66.6 KB stay in L2, so GB/s is reported but not against HBM."""
    import torch
    import fp8_kv_cache_reshape_gb300 as kvq
    import workloads as W
    cfg = W.TINY
    L, hq, hkv, d = cfg.context, cfg.q_heads, cfg.kv_heads, cfg.head_dim
    g = W.generator(W.config_seed(cfg.name) * 1000)
    bt, nb = W.paged_layout([L], P, g)
    kd, vd, one, _ = _fill_decode_cache(kvq, [L], bt, nb, hkv, d, W.generator(11, device=device), device,
                                        unit_scales=True)
    q = W.randn_bf16((1, hq, d), W.generator(12, device=device), device=device)
    out = torch.empty_like(q)
    btd, seq = bt.to(device), torch.tensor([L], dtype=torch.int32, device=device)
    ws = torch.empty(kvq.kvq_decode_workspace_size(1, hq, hkv, d, bt.shape[1]), dtype=torch.uint8, device=device)

    def run():
        for _ in range(calls):
            kvq.kvq_paged_decode_attention(q, kd, vd, one, one, btd, seq, out, num_blocks=nb, sm_scale=d ** -0.5,
                                           workspace=ws)

    gr = capture(run)
    for _ in range(3):
        gr.replay()
    us = time_graph(gr, reps) * 1e3 / (reps * calls)
    byts = decode_bytes_lengths([L], hq, hkv, d)
    return {"workload": cfg.name, "us_per_call": round(us, 3), "bytes_per_call": byts,
            "kv_gbs": round(byts / (us * 1e-6) / 1e9, 1), "l2_resident": True,
            "timing": f"{reps} replays of a CUDA graph of {calls} decode calls (partial + combine) on one cache"}


def conc8_leg(device, layers=4, reps=20):
    """The concurrency-8 configuration: batch 8, lengths uniform in [16384,
    24576] (seeded), 32 query / 8 KV heads, head_dim 128, pages shuffled
    across sequences.  `layers` distinct caches (about 1.4 GB, larger than
    L2) are read in turn, one decode call each."""
    import torch
    import fp8_kv_cache_reshape_gb300 as kvq
    import workloads as W
    cfg = W.CONC8
    hq, hkv, d = cfg.q_heads, cfg.kv_heads, cfg.head_dim
    lengths = W.decode_lengths(cfg)
    bt, nb = W.paged_layout(lengths, P, W.case_generator(cfg))
    btd = bt.to(device)
    seq = torch.tensor(lengths, dtype=torch.int32, device=device)
    caches = []
    for l in range(layers):
        gl = W.generator(W.config_seed(cfg.name) * 1000 + 100 + l, device=device)
        kd, vd, ks, vs = _fill_decode_cache(kvq, lengths, bt, nb, hkv, d, gl, device)
        caches.append((kd, vd, ks, vs, W.randn_bf16((len(lengths), hq, d), gl, device=device)))
    out = torch.empty((len(lengths), hq, d), dtype=torch.bfloat16, device=device)
    ws = torch.empty(kvq.kvq_decode_workspace_size(len(lengths), hq, hkv, d, bt.shape[1]), dtype=torch.uint8,
                     device=device)

    def run():
        for kd, vd, ks, vs, q in caches:
            kvq.kvq_paged_decode_attention(q, kd, vd, ks, vs, btd, seq, out, num_blocks=nb, sm_scale=d ** -0.5,
                                           workspace=ws)

    gr = capture(run)
    for _ in range(3):
        gr.replay()
    us = time_graph(gr, reps) * 1e3 / (reps * layers)
    byts = decode_bytes_lengths(lengths, hq, hkv, d)
    peak, src = _hbm_peak()
    gbs = byts / (us * 1e-6) / 1e9
    return {"workload": cfg.name, "lengths": lengths, "us_per_call": round(us, 3), "bytes_per_call": byts,
            "kv_gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4), "peak_gbs": peak, "peak_source": src,
            "splits": kvq.kvq_decode_num_splits(len(lengths), hkv, bt.shape[1], head_dim=d),
            "timing": f"{reps} replays of a CUDA graph of {layers} decode calls on distinct caches"}


def hybrid_leg(device, reps=10):
    """The hybrid gpt-oss-20b-shaped step: 24 layers, even layers sliding
    window 128 over a BF16 cache, odd layers full attention over an FP8
    cache; 64 query / 8 KV heads, head_dim 64, batch 8, context 32,768.  One
    step = 24 decode calls (12 full caches of 268 MB: 3.2 GB, larger than
    L2).  The sliding-window layers' caches hold their windows' pages; their
    time is also measured at shorter contexts, where it must stay flat."""
    import torch
    import fp8_kv_cache_reshape_gb300 as kvq
    import workloads as W
    cfg = W.HYBRID
    B, L, hq, hkv, d, win = cfg.batch, cfg.context, cfg.q_heads, cfg.kv_heads, cfg.head_dim, cfg.window
    lengths = [L] * B
    g = W.case_generator(cfg)
    bt, nb = W.paged_layout(lengths, P, g)
    btd = bt.to(device)
    seq = torch.tensor(lengths, dtype=torch.int32, device=device)
    # sliding-window caches: 8 pages per sequence, mapped cyclically so that any
    # window position reads written pages
    sw_pages = (win + P - 1) // P
    sw_bt = (torch.arange(B, dtype=torch.int32)[:, None] * sw_pages +
             torch.arange(bt.shape[1], dtype=torch.int32)[None, :] % sw_pages).to(device)
    layers = []
    for l in range(cfg.layers):
        gl = W.generator(W.config_seed(cfg.name) * 1000 + 200 + l, device=device)
        q = W.randn_bf16((B, hq, d), gl, device=device)
        if l % 2 == 0:  # sliding window, BF16
            kd, vd = kvq.alloc_kv_cache(B * sw_pages, hkv, d, cache_dtype="bf16", device=device, fill=0,
                                        paired=PAIRED)
            for b in range(B):
                pos = torch.arange(sw_pages * P, dtype=torch.int64)
                slots = (b * sw_pages + pos // P) * P + pos % P
                kvq.kvq_reshape_and_cache(W.randn_bf16((pos.numel(), hkv, d), gl, device=device),
                                          W.randn_bf16((pos.numel(), hkv, d), gl, device=device), slots.to(device),
                                          kd, vd, cache_dtype="bf16")
            layers.append(dict(sw=True, kd=kd, vd=vd, ks=None, vs=None, q=q, nb=B * sw_pages))
        else:
            kd, vd, ks, vs = _fill_decode_cache(kvq, lengths, bt, nb, hkv, d, gl, device)
            layers.append(dict(sw=False, kd=kd, vd=vd, ks=ks, vs=vs, q=q, nb=nb))
    out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=device)
    ws = torch.empty(kvq.kvq_decode_workspace_size(B, hq, hkv, d, bt.shape[1]), dtype=torch.uint8, device=device)

    def call(ly):
        if ly["sw"]:
            kvq.kvq_paged_decode_attention(ly["q"], ly["kd"], ly["vd"], None, None, sw_bt, seq, out, num_blocks=ly["nb"],
                                           sm_scale=d ** -0.5, window=win, cache_dtype="bf16", workspace=ws)
        else:
            kvq.kvq_paged_decode_attention(ly["q"], ly["kd"], ly["vd"], ly["ks"], ly["vs"], btd, seq, out,
                                           num_blocks=ly["nb"], sm_scale=d ** -0.5, workspace=ws)

    g_step = capture(lambda: [call(ly) for ly in layers])
    g_full = capture(lambda: [call(ly) for ly in layers if not ly["sw"]])
    g_sw = capture(lambda: [call(ly) for ly in layers if ly["sw"]])
    for _ in range(3):
        g_step.replay()
    step_us = time_graph(g_step, reps) * 1e3 / reps
    full_us = time_graph(g_full, reps) * 1e3 / (reps * (cfg.layers // 2))
    sw_rows = []
    for ctx in (4096, 8192, 16384, 32768):
        seq.fill_(ctx)
        g_sw.replay()
        sw_rows.append({"context": ctx, "us_per_sw_layer": round(time_graph(g_sw, 5 * reps) * 1e3 /
                                                                 (5 * reps * (cfg.layers // 2)), 3)})
    seq.fill_(L)
    step_b, full_b, sw_b = hybrid_step_bytes(B, L, hq, hkv, d, cfg.layers, win)
    peak, src = _hbm_peak()
    gbs = step_b / (step_us * 1e-6) / 1e9
    sw_us = [r["us_per_sw_layer"] for r in sw_rows]
    return {"workload": cfg.name, "us_per_step": round(step_us, 2), "bytes_per_step": step_b,
            "kv_gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4), "peak_gbs": peak, "peak_source": src,
            "us_per_full_layer": round(full_us, 3), "bytes_per_full_layer": full_b,
            "full_layer_frac_hbm": round(full_b / (full_us * 1e-6) / 1e9 / peak, 4),
            "bytes_per_sw_layer": sw_b, "sw_layer_vs_context": sw_rows,
            "sw_flatness": round(max(sw_us) / min(sw_us), 3),
            "timing": f"{reps} replays of a CUDA graph of the 24-layer step; full and sliding-window layers also "
                      f"timed alone"}


# ---------------------------------------------------------- CPU baseline ---
# The oracle (oracle/, float64 numpy), as it stands, timed on the host cores
# on each configuration: its decode runs per (sequence, KV head) unit -- the
# unit the method's arithmetic is independent over -- one after the other on
# one core, and over a process pool on all cores.  These functions run in a
# child process that hides the GPU (CUDA_VISIBLE_DEVICES="") and never
# initialises CUDA, so its pool may fork: the workers inherit the inputs.
_CPU_PROBLEM = None


def _oracle_decode_problem(cfg, layer=0, window=None, cache_dtype="fp8_e4m3", only_window_tokens=False):
    """Inputs of one decode layer of `cfg` and the oracle's own cache of them."""
    import numpy as np
    import workloads as W
    from oracle import kv_cache
    case = W.decode_case(cfg, layer=layer, window=window, cache_dtype=cache_dtype,
                         only_window_tokens=only_window_tokens)
    d, hkv = cfg.head_dim, cfg.kv_heads
    bf = cache_dtype == "bf16"
    kc = np.zeros((case.num_blocks, hkv, P, d), np.uint16 if bf else np.uint8)
    vc = np.zeros((case.num_blocks, hkv, d, P), np.uint16 if bf else np.uint8)
    kv_cache.reshape_and_cache(case.k.float().numpy(), case.v.float().numpy(), case.slot_mapping.numpy(), kc, vc,
                               case.k_scale.numpy(), case.v_scale.numpy(), cache_dtype)
    return dict(q=case.q.float().numpy(), kc=kc, vc=vc, ks=case.k_scale.numpy(), vs=case.v_scale.numpy(),
                bt=case.block_table.numpy(), sl=case.seq_lens.numpy(), sm=case.sm_scale, window=case.window,
                dtype=cache_dtype, g=cfg.q_heads // hkv,
                units=[(b, h) for b in range(case.q.shape[0]) for h in range(hkv)],
                bytes=decode_bytes_lengths(case.seq_lens.tolist(), cfg.q_heads, hkv, d, window=case.window,
                                           esize=2 if bf else 1))


def _oracle_decode_unit(i):
    """The oracle's decode (mirrored mode) of unit i of the current problem:
    one sequence and one KV head with its query-head group."""
    from oracle import attention
    pr = _CPU_PROBLEM
    b, h = pr["units"][i]
    g = pr["g"]
    attention.paged_decode(pr["q"][b:b + 1, h * g:(h + 1) * g], pr["kc"][:, h:h + 1], pr["vc"][:, h:h + 1],
                           pr["ks"][h:h + 1], pr["vs"][h:h + 1], pr["bt"][b:b + 1], pr["sl"][b:b + 1], pr["sm"],
                           window=pr["window"], cache_dtype=pr["dtype"])
    return i


def _oracle_prefill_problem(rows_per_unit=8, n_rows=256):
    """The chunked-prefill configuration for the oracle, with a stated sample
    of n_rows (query token, head) rows spread over the chunk."""
    import numpy as np
    import workloads as W
    from oracle import kv_cache
    pc = W.prefill_case(W.PREFILL)
    cfg = pc.cfg
    kc = np.zeros((pc.num_blocks, cfg.kv_heads, P, cfg.head_dim), np.uint8)
    vc = np.zeros((pc.num_blocks, cfg.kv_heads, cfg.head_dim, P), np.uint8)
    kv_cache.reshape_and_cache(pc.k.float().numpy(), pc.v.float().numpy(), pc.slot_mapping.numpy(), kc, vc,
                               pc.k_scale.numpy(), pc.v_scale.numpy())
    qs = np.float32(pc.q_scale.item())
    q8 = kv_cache.quantize_query(pc.q.float().numpy(), qs)
    rng = np.random.default_rng(4)
    flat = rng.choice(cfg.new_tokens * cfg.q_heads, n_rows, replace=False)
    rows = sorted((int(f // cfg.q_heads), int(f % cfg.q_heads)) for f in flat)
    # units: rows of one KV head together (the oracle gathers a head's keys once per call)
    g = cfg.q_heads // cfg.kv_heads
    rows.sort(key=lambda r: (r[1] // g, r[0]))
    units = [rows[i:i + rows_per_unit] for i in range(0, len(rows), rows_per_unit)]
    return dict(q8=q8, qs=qs, kc=kc, vc=vc, ks=pc.k_scale.numpy(), vs=pc.v_scale.numpy(),
                bt=pc.block_table.numpy(), cu=pc.cu_seqlens_q.numpy(), sl=pc.seq_lens.numpy(),
                sm=float(np.float32(pc.sm_scale)), units=units, n_rows=n_rows,
                total_rows=cfg.new_tokens * cfg.q_heads)


def _oracle_prefill_unit(i):
    from oracle import attention
    pr = _CPU_PROBLEM
    attention.prefill(pr["q8"], pr["qs"], pr["kc"], pr["vc"], pr["ks"], pr["vs"], pr["bt"], pr["cu"], pr["sl"],
                      pr["sm"], rows=pr["units"][i])
    return i


def _time_units(fn, n_units, pool, min_seconds):
    """Seconds for one pass over all units: on one core (pool None) or over
    the pool; repeated until min_seconds have passed, the mean taken."""
    reps, t0 = 0, time.perf_counter()
    while True:
        if pool is None:
            for i in range(n_units):
                fn(i)
        else:
            pool.map(fn, range(n_units), chunksize=1)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            return (time.perf_counter() - t0) / reps, reps


def cpu_baselines_run(configs=("tiny", "llama", "conc8", "hybrid", "prefill"), min_seconds=1.0):
    """The oracle timed per configuration, on one core and on every core of
    this host (the caller pins BLAS to one thread per process).  Returns
    {config: {...}} with seconds per call / layer / step and the metric."""
    import multiprocessing as mp
    import workloads as W
    global _CPU_PROBLEM
    ncpu = os.cpu_count() or 1
    ctx = mp.get_context("fork")  # this process has no CUDA context (see above)
    out = {"nproc": ncpu}

    def run(name, fn, n_units):
        one, r1 = _time_units(fn, n_units, None, min_seconds)
        with ctx.Pool(min(ncpu, n_units)) as pool:
            pool.map(fn, range(min(ncpu, n_units)))  # workers started and warm
            allc, ra = _time_units(fn, n_units, pool, min_seconds)
        return {"one_core_s": one, "all_core_s": allc, "threads": min(ncpu, n_units), "units": n_units,
                "reps_one_core": r1, "reps_all_core": ra}

    if "tiny" in configs:
        _CPU_PROBLEM = _oracle_decode_problem(W.TINY)
        r = run("tiny", _oracle_decode_unit, len(_CPU_PROBLEM["units"]))
        r.update(workload=W.TINY.name, per="decode call", bytes=_CPU_PROBLEM["bytes"],
                 sample="the whole call (1 sequence, 1 KV head)")
        out["tiny"] = r
    if "llama" in configs:
        _CPU_PROBLEM = _oracle_decode_problem(W.LLAMA_128K)
        r = run("llama", _oracle_decode_unit, len(_CPU_PROBLEM["units"]))
        r.update(workload=W.LLAMA_128K.name, per="decode layer (a step is 32 of them)", bytes=_CPU_PROBLEM["bytes"],
                 sample="one whole layer: 8 KV-head units of 131,072 tokens")
        out["llama"] = r
    if "conc8" in configs:
        _CPU_PROBLEM = _oracle_decode_problem(W.CONC8)
        r = run("conc8", _oracle_decode_unit, len(_CPU_PROBLEM["units"]))
        r.update(workload=W.CONC8.name, per="decode call", bytes=_CPU_PROBLEM["bytes"],
                 sample="the whole call: 8 sequences x 8 KV-head units")
        out["conc8"] = r
    if "hybrid" in configs:
        _CPU_PROBLEM = _oracle_decode_problem(W.HYBRID, layer=1, window=-1)
        full = run("hybrid_full", _oracle_decode_unit, len(_CPU_PROBLEM["units"]))
        full_b = _CPU_PROBLEM["bytes"]
        _CPU_PROBLEM = _oracle_decode_problem(W.HYBRID, layer=0, window=W.HYBRID.window, cache_dtype="bf16",
                                              only_window_tokens=True)
        sw = run("hybrid_sw", _oracle_decode_unit, len(_CPU_PROBLEM["units"]))
        n = W.HYBRID.layers // 2
        out["hybrid"] = {"workload": W.HYBRID.name, "per": "decode step of 24 layers",
                         "one_core_s": n * (full["one_core_s"] + sw["one_core_s"]),
                         "all_core_s": n * (full["all_core_s"] + sw["all_core_s"]),
                         "threads": full["threads"], "bytes": n * (full_b + _CPU_PROBLEM["bytes"]),
                         "sample": "one full-attention and one sliding-window layer (64 units each), "
                                   "times 12 each", "full_layer": full, "sw_layer": sw}
    if "prefill" in configs:
        _CPU_PROBLEM = _oracle_prefill_problem()
        r = run("prefill", _oracle_prefill_unit, len(_CPU_PROBLEM["units"]))
        f = _CPU_PROBLEM["total_rows"] / _CPU_PROBLEM["n_rows"]
        r.update(workload=W.PREFILL.name, per="chunked prefill call (extrapolated from the row sample)",
                 flops=prefill_flops(), one_core_s=r["one_core_s"] * f, all_core_s=r["all_core_s"] * f,
                 sample=f"{_CPU_PROBLEM['n_rows']} of {_CPU_PROBLEM['total_rows']} (query token, head) rows, "
                        f"spread at random over the chunk; times scaled by {f:.0f}")
        out["prefill"] = r
    _CPU_PROBLEM = None
    for k, r in out.items():
        if isinstance(r, dict) and "bytes" in r:
            r["gbs_one_core"] = r["bytes"] / r["one_core_s"] / 1e9
            r["gbs_all_core"] = r["bytes"] / r["all_core_s"] / 1e9
        if isinstance(r, dict) and "flops" in r:
            r["tflops_all_core"] = r["flops"] / r["all_core_s"] / 1e12
            r["tflops_one_core"] = r["flops"] / r["one_core_s"] / 1e12
    return out


def _cpu_child(args, timeout=1800):
    """Run `bench.py --_cpu-child <json args>` with the GPU hidden and one
    BLAS thread per process; returns its last JSON line."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--_cpu-child", json.dumps(args)], env=env,
                       capture_output=True, text=True, timeout=timeout)
    for line in r.stdout.splitlines()[::-1]:
        if line.startswith("{"):
            return json.loads(line)
    return {"error": r.stderr[-400:]}


def cpu_baselines(min_seconds=1.0):
    """The per-configuration oracle times and, for the JSON line's
    cpu_baseline, the Llama 128K layer on every core."""
    res = _cpu_child({"what": "configs", "min_seconds": min_seconds})
    if "llama" not in res:
        return {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle",
                "sample": "failed: " + str(res.get("error"))}, res
    r = res["llama"]
    head = {"value": round(r["gbs_all_core"], 4), "unit": "GB/s", "cores": r["threads"], "kind": "oracle",
            "sample": f"one decode layer of the 128K workload (8 KV-head units of 131,072 tokens) over "
                      f"{r['threads']} processes of {res['nproc']} host cores; float64 numpy",
            "seconds_per_layer": round(r["all_core_s"], 4), "one_core_seconds_per_layer": round(r["one_core_s"], 4),
            "nproc": res["nproc"]}
    return head, res


# ----------------------------------------------------------------- arms ---
def reference_arm(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, timed on the host
    cores on the same metric, unit and workload; each step is the oracle's
    decode of one whole layer of the 128K workload (8 KV-head units of
    131,072 tokens) over every core (a bounded sample of the 32-layer step).
    Under torchrun only rank 0 runs it."""
    if rank != 0:
        return
    res = _cpu_child({"what": "reference", "steps": args.steps, "warmup": args.warmup})
    if "seconds_per_step" not in res:
        print(json.dumps({"impl": "reference", "unavailable": "oracle run failed: " + str(res.get("error"))[-200:]}),
              flush=True)
        return
    sec, byts = res["seconds_per_step"], res["bytes_per_step"]
    value = round(byts / sec / 1e9, 4)
    cb = {"value": value, "unit": "GB/s", "cores": res["threads"], "kind": "oracle",
          "sample": f"one decode layer of the 128K workload per step (8 KV-head units of 131,072 tokens) over "
                    f"{res['threads']} processes on {res['nproc']} host cores; float64 numpy; {args.steps} timed "
                    f"steps after {args.warmup} warm-up"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "llama31_8b_decode_128k", "layers": LAYERS, "batch": 1, "context": CONTEXT,
                       "q_heads": HQ, "kv_heads": HKV, "head_dim": D, "page": P,
                       "step": "the oracle's decode of one layer (of the 32 in a step)"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _reference_steps(steps, warmup):
    """The reference arm's timed loop (in the CPU child)."""
    import multiprocessing as mp
    import workloads as W
    global _CPU_PROBLEM
    _CPU_PROBLEM = _oracle_decode_problem(W.LLAMA_128K)
    n = len(_CPU_PROBLEM["units"])
    ncpu = os.cpu_count() or 1
    with mp.get_context("fork").Pool(min(ncpu, n)) as pool:
        for _ in range(max(1, warmup)):
            pool.map(_oracle_decode_unit, range(n), chunksize=1)
        t0 = time.perf_counter()
        for _ in range(steps):
            pool.map(_oracle_decode_unit, range(n), chunksize=1)
        sec = (time.perf_counter() - t0) / max(1, steps)
    return {"seconds_per_step": sec, "bytes_per_step": _CPU_PROBLEM["bytes"], "threads": min(ncpu, n),
            "nproc": ncpu}


def ours_arm(args, rank, world, local_rank):
    import torch
    from fp8_kv_cache_reshape_gb300.sharding import kv_head_shard
    device = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(device))

    def barrier():
        if dist is not None:
            dist.barrier()

    # head-sharded across ranks: rank r holds KV heads [r * 8 / N, (r + 1) * 8 / N)
    # (and their query-head groups) of N sequences; no collective on the data path
    shard = kv_head_shard(HQ, HKV, world, rank)
    wl = build_workload(device, seed=7 + rank, batch=world, q_heads=shard.q_heads, kv_heads=shard.kv_heads)
    g_step = capture(lambda: run_step(wl))
    g_dec = capture(lambda: run_step(wl, decode_only=True))
    g_two = capture(lambda: run_step(wl, two_calls=True))
    for _ in range(max(3, args.warmup)):
        g_step.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        total_ms = time_graph(g_step, args.steps)
        # the dominant kernel pair alone: 32 decode calls per replay
        dec_reps = max(200, args.steps)
        dec_ms = time_graph(g_dec, dec_reps)
    barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(total_ms, dist, device)
    st = int(wl["status"].item())
    assert st == 0, f"device status {st:#x}"
    # the two-call form and the end-to-end step right after, in the same conditions
    with ClockSampler(local_rank) as clk2:
        two_reps = max(20, args.steps)
        two_ms = time_graph(g_two, two_reps) / two_reps  # the same step as two calls per layer
        e2e_fn, h2d, d2h = e2e_setup(wl)
        g_e2e = capture(e2e_fn)
        e2e_reps = max(3, args.steps)
        e2e_ms = time_graph(g_e2e, e2e_reps) / e2e_reps
        eager_ms = time_eager(e2e_fn, 3) / 3
    e2e_ms = max_over_ranks(e2e_ms, dist, device)

    call_bytes = decode_bytes(CONTEXT, batch=world, hq=shard.q_heads, hkv=shard.kv_heads)
    step_bytes = LAYERS * (call_bytes + cache_write_bytes(world, hkv=shard.kv_heads))
    ms_per_step = total_ms / args.steps
    value = job_value(world, step_bytes, args.steps, total_ms)
    hbm, src = _hbm_peak()
    call_ms = dec_ms / (dec_reps * LAYERS)
    achieved = call_bytes / (call_ms * 1e-3) / 1e9
    traffic = decode_traffic() if world == 1 else None
    legs = world == 1  # the characterisation legs run on single-GPU runs only
    sweep = clocked(local_rank, context_sweep, wl, g_dec) if legs and not args.no_sweep else None
    configs = None
    if legs and not args.no_configs:
        configs = {"tiny_decode_512": clocked(local_rank, tiny_leg, device),
                   "llama31_8b_decode_conc8_20k": clocked(local_rank, conc8_leg, device),
                   "gpt_oss_20b_hybrid_decode_32k": clocked(local_rank, hybrid_leg, device)}
    pf = None
    if legs and not args.no_prefill:
        if args.prefill_head_dim == 256:
            pf = clocked(local_rank, prefill_leg, device, head_dim=256)
        else:
            pf = clocked(local_rank, prefill_leg, device)
    if pf is not None and not args.no_e5m2:
        pf["e5m2_cache"] = clocked(local_rank, prefill_leg, device, cache_dtype="fp8_e5m2")
        pf["per_token_scales"] = clocked(local_rank, prefill_leg, device, per_token=True)
    no_cmp = not legs or args.no_sweep
    bf = None if (no_cmp or args.no_bf16) else clocked(local_rank, format_compare, sweep, device, "bf16")
    e5 = None if (no_cmp or args.no_e5m2) else clocked(local_rank, format_compare, sweep, device, "fp8_e5m2")
    pt = None if (no_cmp or args.no_per_token) else clocked(local_rank, format_compare, sweep, device, "fp8_e4m3",
                                                             per_token=True)
    abl = None
    if not (no_cmp or args.no_ablation):  # single- against two-level accumulation
        sl = clocked(local_rank, format_compare, sweep, device, "fp8_e4m3", accumulation="single_level")
        abl = {"decode_single_level": sl,
               "prefill_single_level": None if args.no_prefill else clocked(local_rank, prefill_leg, device,
                                                                            accumulation="single_level"),
               "prefill_head_dim_256": None if args.no_prefill else clocked(local_rank, prefill_leg, device,
                                                                            head_dim=256)}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 storage, f16/f32 MMA, f32 accumulate", "data": "synthetic",
        "config": {"workload": "llama31_8b_decode_128k", "layers": LAYERS, "batch": world, "context": CONTEXT,
                   "q_heads": HQ, "kv_heads": HKV, "head_dim": D, "page": P, "block_table": "permuted",
                   "cache_layout": "paired K|V pages" if PAIRED else "separate K and V caches",
                   "scales": "per-KV-head amax/448, 4 outlier channels x20",
                   "l2": "inputs larger than L2: 32 distinct 256 MiB layer caches per step and rank",
                   "parallelism": (f"KV heads sharded over {world} GPUs ({shard.kv_heads} KV / {shard.q_heads} "
                                   f"query heads each), batch {world}; no collective on the data path")
                   if world > 1 else "1 GPU",
                   "us_per_layer": round(ms_per_step * 1e3 / LAYERS, 3)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic,
                     "kernel": "paged decode attention call (split-KV partial + LSE combine), per layer",
                     "peak_source": f"{src} hbm_gbs",
                     "avg_call_us": round(call_ms * 1e3, 3), "bytes_per_call": call_bytes,
                     "timing": f"{dec_reps} replays of a CUDA graph of {LAYERS} decode calls"},
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "how": "public API calls: one host->device copy of the step's inputs (every layer's q and new "
                       "K/V, one pinned staging buffer), the 32 decode calls, one device->host copy of every "
                       "layer's output; captured once in a CUDA graph and replayed",
                "eager_python_ms_per_step": round(eager_ms, 4),
                "eager_python_value": round(world * step_bytes / (eager_ms * 1e-3) / 1e9, 1)},
        "gpu_launches": args.steps * LAYERS * 2,
        "timing": "CUDA graph of one step (32 x [decode partial with the new token's cache write + combine]) "
                  "replayed",
        "step_two_calls": {"ms_per_step": round(two_ms, 4),
                           "value": round(world * step_bytes / (two_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                           "how": "the same step as kvq_reshape_and_cache + kvq_paged_decode_attention per layer "
                                  "(3 kernels per layer)", "clocks": clk2.summary()},
        "clocks": clk.summary(),
        "sweep": sweep,
        "configs": configs,
        "prefill": pf,
        "bf16_compare": bf,
        "e5m2_compare": e5,
        "per_token_compare": pt,
        "accumulation_ablation": abl,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        head, per_config = cpu_baselines()
        line["cpu_baseline"] = head
        line["cpu_baseline_per_config"] = per_config
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    if len(sys.argv) == 3 and sys.argv[1] == "--_cpu-child":
        a = json.loads(sys.argv[2])
        if a["what"] == "configs":
            print(json.dumps(cpu_baselines_run(min_seconds=a.get("min_seconds", 1.0))), flush=True)
        else:
            print(json.dumps(_reference_steps(a["steps"], a["warmup"])), flush=True)
        return
    args = parse()
    global LAYERS, PAIRED
    LAYERS = args.layers
    PAIRED = not args.separate_caches
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    ours_arm(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
