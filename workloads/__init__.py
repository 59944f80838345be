"""Seeded synthetic inputs shaped like the workloads the FP8 KV-cache pages
measure.  Both the CUDA path's tests / bench and the oracle's tests draw from
here; the module holds no quantization or attention arithmetic.

Recipe (every tensor from a torch.Generator seeded per case):
* Q, K, V: float32 N(0, 1) rounded to bfloat16.
* Outlier channels (the Llama-3.1-8B-shaped case): 4 channels per KV head,
  picked by the generator, multiplied by 20 in both K and V.
* Per-KV-head static scales: the caller's calibration, amax / 448 over the
  tokens of each head ("FP8 and KV cache", dynamic vs static scale), or 1.0
  when uncalibrated (the vLLM blog's accuracy runs).
* Block tables: the pages of all sequences are a random permutation of a
  pool with 12.5% spare pages, so pages are shuffled across sequences.
* Context lengths: fixed, or uniform in a range (concurrency-8 case, about
  20k tokens +-20%).

Shapes follow the pages: Llama-3.1-8B (32 query / 8 KV heads, head_dim 128,
32 layers), 128K context, concurrency 8 at ~20k tokens, gpt-oss-20b
(64 query / 8 KV heads, head_dim 64, 24 layers alternating full and
sliding-window-128 attention).
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0
PAGE = 16


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    context: int                      # tokens per sequence (fixed lengths)
    context_range: Optional[tuple] = None  # (lo, hi) inclusive, ragged batches
    page: int = PAGE
    outliers: int = 0                 # outlier channels per KV head (x20)
    calibrated: bool = True           # amax/448 scales, else 1.0
    layers: int = 1
    window_layers: str = "none"       # "none" | "even" : even layers use SW
    window: int = -1


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    new_tokens: int
    cached_tokens: int
    q_heads: int
    kv_heads: int
    head_dim: int
    page: int = PAGE
    batch: int = 1


TINY = DecodeConfig("tiny_decode_512", batch=1, q_heads=4, kv_heads=1, head_dim=64,
                    context=512, calibrated=False)
LLAMA_128K = DecodeConfig("llama31_8b_decode_128k", batch=1, q_heads=32, kv_heads=8,
                          head_dim=128, context=131072, outliers=4, layers=32)
CONC8 = DecodeConfig("llama31_8b_decode_conc8_20k", batch=8, q_heads=32, kv_heads=8,
                     head_dim=128, context=24576, context_range=(16384, 24576))
PREFILL = PrefillConfig("llama31_8b_chunked_prefill_4k_on_28k", new_tokens=4096,
                        cached_tokens=28672, q_heads=32, kv_heads=8, head_dim=128)
HYBRID = DecodeConfig("gpt_oss_20b_hybrid_decode_32k", batch=8, q_heads=64, kv_heads=8,
                      head_dim=64, context=32768, layers=24, window_layers="even",
                      window=128)

CONFIGS = {c.name: c for c in (TINY, LLAMA_128K, CONC8, PREFILL, HYBRID)}


def config_seed(name: str) -> int:
    """1..5 for the named configurations, a stable hash for others."""
    names = list(CONFIGS)
    return 1 + names.index(name) if name in names else 100 + zlib.crc32(name.encode()) % 100000


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """float32 N(0,1) rounded to bfloat16."""
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def outlier_channels(kv_heads: int, head_dim: int, n: int, gen: torch.Generator) -> torch.Tensor:
    """[kv_heads][n] distinct channel indices per head (on the CPU)."""
    return torch.stack([torch.randperm(head_dim, generator=gen)[:n] for _ in range(kv_heads)])


def apply_outliers(x: torch.Tensor, channels: torch.Tensor, factor: float = 20.0) -> torch.Tensor:
    """Multiply the chosen channels of x [T][Hkv][D] by `factor` (exact in
    bfloat16 for a factor of 20 up to rounding; the result is re-rounded)."""
    if channels.numel() == 0:
        return x
    y = x.float()
    ch = channels.to(x.device)
    for h in range(ch.shape[0]):
        y[:, h, ch[h]] *= factor
    return y.to(torch.bfloat16)


def calibrate_amax(x: torch.Tensor, fmt_max: float = None) -> torch.Tensor:
    """Caller-side static calibration: per-head amax / (the format's largest
    value: 448 for E4M3, 57344 for E5M2), float32 [Hkv]."""
    a = x.float().abs().amax(dim=(0, 2))
    s = (a / (E4M3_MAX if fmt_max is None else fmt_max)).to(torch.float32)
    return torch.where(s > 0, s, torch.ones_like(s))


def context_lengths(cfg: DecodeConfig, gen: torch.Generator) -> list:
    if cfg.context_range is None:
        return [cfg.context] * cfg.batch
    lo, hi = cfg.context_range
    return [int(v) for v in torch.randint(lo, hi + 1, (cfg.batch,), generator=gen)]


def paged_layout(lengths, page: int, gen: torch.Generator, spare: float = 0.125):
    """Block table int32 [B][max_blocks] (unused entries = 0) for sequences of
    the given lengths, pages drawn from a shuffled pool with `spare` extra
    pages.  Returns (block_table, num_blocks)."""
    pages = [max(1, math.ceil(L / page)) for L in lengths]
    total = sum(pages)
    num_blocks = total + max(1, int(math.ceil(total * spare)))
    perm = torch.randperm(num_blocks, generator=gen)
    max_blocks = max(pages)
    bt = torch.zeros((len(lengths), max_blocks), dtype=torch.int32)
    at = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[at:at + n].to(torch.int32)
        at += n
    return bt, num_blocks


def slots_for(block_table: torch.Tensor, seq: int, positions: torch.Tensor, page: int) -> torch.Tensor:
    """int64 cache slots of the given token positions of one sequence."""
    blocks = block_table[seq].to(torch.int64)[positions // page]
    return blocks * page + positions % page


def case_generator(cfg: DecodeConfig, layer: int = 0, seed_base: int = 0) -> torch.Generator:
    """The generator of decode_case(cfg, layer, seed_base); its first draw is
    the context lengths."""
    return generator(seed_base + 1000 * config_seed(cfg.name) + layer)


def decode_lengths(cfg: DecodeConfig, layer: int = 0, seed_base: int = 0) -> list:
    """The context lengths decode_case(cfg, layer, seed_base) uses, without
    building the case (for byte counts and GPU-side workloads)."""
    return context_lengths(cfg, case_generator(cfg, layer, seed_base))


@dataclasses.dataclass
class DecodeCase:
    """One decode layer: the tokens to cache and the step's query."""
    cfg: DecodeConfig
    q: torch.Tensor            # bf16 [B][Hq][D]
    k: torch.Tensor            # bf16 [T][Hkv][D] every cached token, all sequences
    v: torch.Tensor
    slot_mapping: torch.Tensor  # int64 [T]
    block_table: torch.Tensor  # int32 [B][max_blocks]
    seq_lens: torch.Tensor     # int32 [B]
    num_blocks: int
    k_scale: torch.Tensor      # float32 [Hkv]
    v_scale: torch.Tensor
    sm_scale: float
    window: int
    cache_dtype: str           # "fp8_e4m3" | "fp8_e5m2" | "bf16"


def decode_case(cfg: DecodeConfig, layer: int = 0, seed_base: int = 0, lengths=None,
                window: Optional[int] = None, cache_dtype: str = "fp8_e4m3",
                only_window_tokens: bool = False) -> DecodeCase:
    """Seeded inputs for one decode layer of `cfg` (CPU tensors).

    Every position 0..L-1 of every sequence is a cached token (the last one
    being the step's own token).  With only_window_tokens, only the last
    `window` positions are produced (what a sliding-window layer reads)."""
    gen = case_generator(cfg, layer, seed_base)
    lens = list(lengths) if lengths is not None else context_lengths(cfg, gen)
    win = cfg.window if window is None else window
    bt, num_blocks = paged_layout(lens, cfg.page, gen)
    ks, ps = [], []
    for b, L in enumerate(lens):
        start = max(0, L - win) if (only_window_tokens and win >= 0) else 0
        pos = torch.arange(start, L, dtype=torch.int64)
        ps.append(pos)
        ks.append(slots_for(bt, b, pos, cfg.page))
    slot = torch.cat(ks) if ks else torch.zeros(0, dtype=torch.int64)
    T = int(slot.numel())
    k = randn_bf16((T, cfg.kv_heads, cfg.head_dim), gen)
    v = randn_bf16((T, cfg.kv_heads, cfg.head_dim), gen)
    if cfg.outliers:
        ch = outlier_channels(cfg.kv_heads, cfg.head_dim, cfg.outliers, gen)
        k = apply_outliers(k, ch)
        v = apply_outliers(v, ch)
    q = randn_bf16((cfg.batch if lengths is None else len(lens), cfg.q_heads, cfg.head_dim), gen)
    if cfg.calibrated and cache_dtype in ("fp8_e4m3", "fp8_e5m2") and T > 0:
        fmt_max = E5M2_MAX if cache_dtype == "fp8_e5m2" else E4M3_MAX
        k_scale, v_scale = calibrate_amax(k, fmt_max), calibrate_amax(v, fmt_max)
    else:
        k_scale = torch.ones(cfg.kv_heads, dtype=torch.float32)
        v_scale = torch.ones(cfg.kv_heads, dtype=torch.float32)
    return DecodeCase(cfg, q, k, v, slot, bt, torch.tensor(lens, dtype=torch.int32),
                      num_blocks, k_scale, v_scale, 1.0 / math.sqrt(cfg.head_dim),
                      win, cache_dtype)


@dataclasses.dataclass
class PrefillCase:
    cfg: PrefillConfig
    q: torch.Tensor            # bf16 [Tq][Hq][D]
    k: torch.Tensor            # bf16 [T][Hkv][D] every cached token incl. new
    v: torch.Tensor
    slot_mapping: torch.Tensor
    block_table: torch.Tensor
    cu_seqlens_q: torch.Tensor  # int32 [B+1]
    seq_lens: torch.Tensor     # int32 [B]
    num_blocks: int
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    q_scale: torch.Tensor      # float32 [1]
    sm_scale: float


def prefill_case(cfg: PrefillConfig, seed_base: int = 0, new_tokens=None, cached_tokens=None,
                 batch=None) -> PrefillCase:
    """Seeded chunked-prefill inputs: each sequence has `cached_tokens` old
    tokens plus `new_tokens` new ones, all in the cache."""
    gen = generator(seed_base + 4000)
    nq = cfg.new_tokens if new_tokens is None else new_tokens
    nc = cfg.cached_tokens if cached_tokens is None else cached_tokens
    B = cfg.batch if batch is None else batch
    lens = [nc + nq] * B
    bt, num_blocks = paged_layout(lens, cfg.page, gen)
    slot = torch.cat([slots_for(bt, b, torch.arange(L, dtype=torch.int64), cfg.page)
                      for b, L in enumerate(lens)])
    T = int(slot.numel())
    k = randn_bf16((T, cfg.kv_heads, cfg.head_dim), gen)
    v = randn_bf16((T, cfg.kv_heads, cfg.head_dim), gen)
    q = randn_bf16((B * nq, cfg.q_heads, cfg.head_dim), gen)
    cu = torch.arange(0, B + 1, dtype=torch.int32) * nq
    q_scale = (q.float().abs().amax() / E4M3_MAX).reshape(1).to(torch.float32)
    return PrefillCase(cfg, q, k, v, slot, bt, cu, torch.tensor(lens, dtype=torch.int32),
                       num_blocks, calibrate_amax(k), calibrate_amax(v), q_scale,
                       1.0 / math.sqrt(cfg.head_dim))
