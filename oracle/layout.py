"""The library's physical page format, restated from its documentation
(include/kvq.h, "Cache format"), for byte-exact comparisons.

Test infrastructure: only the tests, the smoke check and the bench's CPU
baseline may import this module.

The oracle computes caches in the logical layout K[block][h][t][d],
V[block][h][d][t]; these functions permute bytes between that and the
physical layout:
* K page: row t of D elements (row_bytes = D * esize); its 16-byte chunk j
  sits at chunk j ^ (t % 8) for 128-byte rows, j ^ ((t // 2) % 4) for 64-byte
  rows, and (j & 8) | ((j ^ t) & 7) for 256-byte rows (BF16 at D = 128).
* FP8 K page at D = 256: two 2 KiB half-pages, half h holding dims
  128h .. 128h + 127 of all 16 tokens as 128-byte rows; chunk j of token t
  at byte (j // 8) * 2048 + t * 128 + ((j % 8) ^ (t % 8)) * 16.
* V page (FP8): row d of 16 slots; token t in slot rho(t),
  rho = [0,1,4,5,8,9,12,13,2,3,6,7,10,11,14,15].
* V page (BF16): row d of 16 bf16; token t in slot t, and the two 16-byte
  halves of the row are swapped when (d // 4) is odd.
* Per-token V page (FP8): the V page above, then a scale tail of 16 K scales
  and 16 V scales (float32, slot t at tail[t] and tail[16 + t]).
No arithmetic of the method lives here.
"""
from __future__ import annotations

import numpy as np

P = 16
RHO = np.array([0, 1, 4, 5, 8, 9, 12, 13, 2, 3, 6, 7, 10, 11, 14, 15])


def k_chunk_position(t: int, j: int, row_bytes: int) -> int:
    if row_bytes == 128:
        return j ^ (t % 8)
    if row_bytes == 64:
        return j ^ ((t // 2) % 4)
    if row_bytes == 256:
        return (j & 8) | ((j ^ t) & 7)
    raise ValueError(row_bytes)


def _k_perm(D: int, esize: int) -> np.ndarray:
    """Physical byte index -> logical byte index within one K page."""
    rb = D * esize
    perm = np.empty(P * rb, dtype=np.int64)
    for t in range(P):
        for j in range(rb // 16):
            if esize == 1 and D == 256:
                phys = (j // 8) * 2048 + t * 128 + ((j % 8) ^ (t % 8)) * 16
            else:
                phys = t * rb + k_chunk_position(t, j, rb) * 16
            perm[phys: phys + 16] = t * rb + j * 16 + np.arange(16)
    return perm


def _v_perm(D: int, esize: int) -> np.ndarray:
    """Physical byte index -> logical byte index within one V page
    (logical: row d, token t, esize bytes per element)."""
    rb = P * esize
    perm = np.empty(D * rb, dtype=np.int64)
    for d in range(D):
        for t in range(P):
            if esize == 1:
                phys = d * rb + RHO[t]
                perm[phys] = d * rb + t
            else:
                half = (t // 8) ^ ((d // 4) % 2)
                phys = d * rb + half * 16 + (t % 8) * 2
                perm[phys: phys + 2] = d * rb + t * 2 + np.arange(2)
    return perm


def _as_bytes(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    return x.view(np.uint8).reshape(x.shape[0], x.shape[1], -1)


def to_device_format(k_cache, v_cache):
    """Logical caches (uint8 E4M3 or uint16 bf16 bits) -> physical byte arrays
    [num_blocks][Hkv][page_bytes]."""
    esize = k_cache.dtype.itemsize
    nb, H, _, D = k_cache.shape
    kb = _as_bytes(k_cache)
    vb = _as_bytes(v_cache)
    return kb[:, :, _k_perm(D, esize)].copy(), vb[:, :, _v_perm(D, esize)].copy()


def from_device_format(kd, vd, D: int, esize: int):
    """Physical byte arrays -> logical caches (uint8 or uint16)."""
    nb, H, _ = kd.shape
    kp, vp = _k_perm(D, esize), _v_perm(D, esize)
    kl = np.empty_like(kd)
    vl = np.empty_like(vd)
    kl[:, :, kp] = kd
    vl[:, :, vp] = vd
    dt = np.uint8 if esize == 1 else np.uint16
    return (kl.view(dt).reshape(nb, H, P, D), vl.view(dt).reshape(nb, H, D, P))


def to_device_format_per_token(k_cache, v_cache, kv_scale_cache):
    """Logical FP8 caches and the scale cache [nb][Hkv][2][P] (float32) ->
    (K pages, V pages with their scale tails)."""
    kd, vd = to_device_format(k_cache, v_cache)
    tail = np.ascontiguousarray(kv_scale_cache, dtype=np.float32).view(np.uint8).reshape(kd.shape[0], kd.shape[1], -1)
    return kd, np.concatenate([vd, tail], axis=2)


def from_device_format_per_token(kd, vd, D: int):
    """(K pages, V pages with tails) -> logical FP8 caches and the scale
    cache [nb][Hkv][2][P] (float32)."""
    nb, H, _ = vd.shape
    codes = np.ascontiguousarray(vd[:, :, :P * D])
    tail = np.ascontiguousarray(vd[:, :, P * D:]).view(np.float32).reshape(nb, H, 2, P)
    kl, vl = from_device_format(kd, codes, D, 1)
    return kl, vl, tail


def to_device_format_paired(k_cache, v_cache, kv_scale_cache=None):
    """The paired layout: [num_blocks][Hkv][K page | V page] bytes (with
    per-token scales, the V page carries its scale tail)."""
    if kv_scale_cache is None:
        kd, vd = to_device_format(k_cache, v_cache)
    else:
        kd, vd = to_device_format_per_token(k_cache, v_cache, kv_scale_cache)
    return np.concatenate([kd, vd], axis=2)
