"""Paged KV-cache write, query quantization and the KV byte formulas.

Test infrastructure: only the tests, the smoke check and the bench's CPU
baseline may import this module.

Cache layout (the library's documented format; the pages fix none)
------------------------------------------------------------------
* K cache: ``[num_blocks][Hkv][P][D]`` -- one (block, KV head) page holds P
  tokens, each a row of D values.
* V cache: ``[num_blocks][Hkv][D][P]`` -- the same page transposed, one row
  of P tokens per dimension.
* Element type: E4M3 or E5M2 bytes (uint8) or bfloat16 (stored as uint16
  bits).
* Token slot s lives in block s // P at offset s % P (PagedAttention as
  described in "FP8 quantization and long-context inference", section 6).

Sources
-------
* "The state of FP8 KV-cache and attention quantization in vLLM", section
  "Kernel and vLLM improvements", per-head scales: the cache-write kernel
  takes an array of scales, one per KV head, instead of one scalar.
* "FP8 and KV cache", section "How to enable it in the engine": scales may be
  per tensor (one each for Q, K, V) or per attention head; uncalibrated
  scales are 1.0; with FP8 attention the query is also quantized to FP8.
* "FP8 and KV cache", section "KV cache": K and V together hold
  2 x layers x kv_heads x head_dim values per token (65,536 for 32 x 8 x 128;
  128 KiB per token in BF16, 64 KiB in FP8; 16 GiB / 8 GiB for a 128K
  sequence), and the decode lower bound is bytes read / peak bandwidth.
* "kv-cache-quantization-fp8-scale-granularity" (inference-research note):
  327,680 bytes (320 KiB) per token for 80 x 8 x 128 in BF16, 40.0 GiB at 128K.
* "FP8 and KV cache", "How to enable it in the engine": the cache dtypes
  include fp8_e4m3 and fp8_e5m2 (codec in e5m2.py).
"""
from __future__ import annotations

import numpy as np

from . import e4m3, e5m2

FP8 = "fp8_e4m3"
FP8_E5M2 = "fp8_e5m2"
BF16 = "bf16"
FP8_TYPES = (FP8, FP8_E5M2)


def codec(cache_dtype):
    """The 8-bit codec module of an FP8 cache dtype."""
    if cache_dtype == FP8:
        return e4m3
    if cache_dtype == FP8_E5M2:
        return e5m2
    raise ValueError(f"not an FP8 cache dtype: {cache_dtype!r}")


# ---------------------------------------------------------------- bfloat16 ---
def bf16_bits_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> the float32 values they encode."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f32_to_bf16_bits_exact(x) -> np.ndarray:
    """float32 values that are exactly bfloat16 -> their uint16 bits.

    Raises if any value is not representable (the inputs here are bf16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value is not exactly representable in bfloat16")
    return (u >> 16).astype(np.uint16)


def _bf16_bits_or_none(x):
    """uint16 bit patterns if every value of x is a bfloat16, else None."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if np.any(u & 0xFFFF):
        return None
    return (u >> 16).astype(np.uint16)


# -------------------------------------------------------------- cache write ---
def reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                      cache_dtype=FP8):
    """Write new tokens into the paged cache in place.

    k, v: float32 arrays [T][Hkv][D] holding bfloat16 values.
    slot_mapping: int64 [T]; a negative slot means "skip this token".
    k_cache: [num_blocks][Hkv][P][D]; v_cache: [num_blocks][Hkv][D][P];
    uint8 for FP8 (E4M3 or E5M2), uint16 (bf16 bits) for BF16.
    k_scale, v_scale: float32 [Hkv] (ignored for BF16).

    For FP8 each element becomes encode(fl32(x / s[h])) in the cache's
    8-bit format.  A slot at or beyond
    num_blocks * P is an error: the token is skipped and the returned flag is
    True.  Returns (k_cache, v_cache, bad_slot_seen).
    """
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    T, Hkv, D = k.shape
    num_blocks, _, P, _ = k_cache.shape
    slots = np.asarray(slot_mapping, dtype=np.int64)
    if cache_dtype in FP8_TYPES:
        fmt = codec(cache_dtype)
        ks = np.asarray(k_scale, np.float32)
        vs = np.asarray(v_scale, np.float32)
        kb, vb = _bf16_bits_or_none(k), _bf16_bits_or_none(v)
        if kb is not None and vb is not None:
            kq = np.empty(k.shape, np.uint8)
            vq = np.empty(v.shape, np.uint8)
            for h in range(Hkv):  # one table per head: encode(fl32(x / s[h])) for every bf16 x
                kq[:, h] = fmt.quantize_bf16_bits(kb[:, h], ks[h])
                vq[:, h] = fmt.quantize_bf16_bits(vb[:, h], vs[h])
        else:
            kq = fmt.quantize(k, ks[None, :, None])
            vq = fmt.quantize(v, vs[None, :, None])
    else:
        kq = f32_to_bf16_bits_exact(k)
        vq = f32_to_bf16_bits_exact(v)
    bad = bool(np.any(slots >= num_blocks * P))
    keep = (slots >= 0) & (slots < num_blocks * P)
    blk, off = slots[keep] // P, slots[keep] % P
    k_cache[blk, :, off, :] = kq[keep]
    v_cache[blk, :, :, off] = vq[keep]
    return k_cache, v_cache, bad


# ------------------------------------------------- per-token dynamic scales ---
def fmt_max(cache_dtype):
    """Largest finite value of an FP8 cache format (448 or 57344)."""
    return codec(cache_dtype).E4M3_MAX if cache_dtype == FP8 else codec(cache_dtype).E5M2_MAX


def per_token_scales(x, cache_dtype=FP8):
    """Dynamic scale of every token and head: s[t][h] = fl32(amax_d |x[t][h][d]|
    / fmt_max), so each token's largest element maps onto the format's largest
    value ("FP8 and KV cache", "Dynamic or static scale": per-token scales
    3.2/448 and 180/448; "FP8 quantization and long-context inference",
    section 2.2: every new token gets its own scale).  A token whose values
    are all zero gets scale 1.0 (reading: the pages do not cover it)."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    s = (amax / np.float32(fmt_max(cache_dtype))).astype(np.float32)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def reshape_and_cache_per_token(k, v, slot_mapping, k_cache, v_cache, kv_scale_cache, cache_dtype=FP8):
    """Cache write with per-token dynamic scales, in place.

    As reshape_and_cache, but each (token, head) is quantized with its own
    scale from per_token_scales(); the K and V scales are stored at the
    token's slot of kv_scale_cache (float32 [num_blocks][Hkv][2][P]:
    [..][0][off] K, [..][1][off] V -- the library's interleaved layout).
    Returns (k_cache, v_cache, kv_scale_cache, bad_slot_seen)."""
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    fmt = codec(cache_dtype)
    num_blocks, _, P, _ = k_cache.shape
    slots = np.asarray(slot_mapping, dtype=np.int64)
    sk = per_token_scales(k, cache_dtype)  # [T][Hkv]
    sv = per_token_scales(v, cache_dtype)
    kq = fmt.quantize(k, sk[:, :, None])
    vq = fmt.quantize(v, sv[:, :, None])
    bad = bool(np.any(slots >= num_blocks * P))
    keep = (slots >= 0) & (slots < num_blocks * P)
    blk, off = slots[keep] // P, slots[keep] % P
    k_cache[blk, :, off, :] = kq[keep]
    v_cache[blk, :, :, off] = vq[keep]
    kv_scale_cache[blk, :, 0, off] = sk[keep]
    kv_scale_cache[blk, :, 1, off] = sv[keep]
    return k_cache, v_cache, kv_scale_cache, bad


def gather_scales(scale_cache, block_table_row, positions, kv_head):
    """Per-token scales ([n]) of the given positions of one sequence and head
    from one plane [num_blocks][Hkv][P] of the scale cache."""
    P = scale_cache.shape[2]
    pos = np.asarray(positions, dtype=np.int64)
    blocks = np.asarray(block_table_row, dtype=np.int64)[pos // P]
    return scale_cache[blocks, kv_head, pos % P]


def quantize_query(q, q_scale):
    """q8 = encode(fl32(q / s_q)) with one per-tensor scale s_q."""
    return e4m3.quantize(q, np.float32(q_scale))


def gather_tokens(cache_k, cache_v, block_table_row, positions, kv_head):
    """K rows and V rows ([n][D] each) of the given token positions of one
    sequence and one KV head, read through the block table."""
    P = cache_k.shape[2]
    pos = np.asarray(positions, dtype=np.int64)
    blocks = np.asarray(block_table_row, dtype=np.int64)[pos // P]
    off = pos % P
    kk = cache_k[blocks, kv_head, off, :]
    vv = cache_v[blocks, kv_head, :, off]
    return kk, vv


# ------------------------------------------------------------ byte formulas ---
def kv_values_per_token(layers, kv_heads, head_dim):
    """K plus V values per token: 2 * layers * kv_heads * head_dim."""
    return 2 * layers * kv_heads * head_dim


def kv_bytes(layers, kv_heads, head_dim, bytes_per_value, tokens=1, batch=1):
    """KV-cache bytes: 2 * layers * kv_heads * head_dim * tokens * batch * bytes."""
    return kv_values_per_token(layers, kv_heads, head_dim) * tokens * batch * bytes_per_value


def decode_time_lower_bound_s(weight_bytes, kv_bytes_per_seq, batch, bandwidth_bytes_per_s):
    """Bytes read per decode step (weights + batch x KV) / peak bandwidth."""
    return (weight_bytes + batch * kv_bytes_per_seq) / bandwidth_bytes_per_s
