"""Pins of the oracle's cache write, query quantization and byte formulas.

* brute force: every element placed by explicit per-element loops;
* sentinel bytes untouched; skipped (negative) slots; out-of-range slots
  reported;
* the byte formulas against the values the pages print (tests/golden).
"""
import json
import math
import os

import numpy as np
import torch

from oracle import e4m3, kv_cache
from oracle.kv_cache import FP8, BF16

GOLD = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes.json")


def _tiny(T=37, Hkv=3, D=8, P=4, nb=16, seed=0):
    rng = np.random.default_rng(seed)
    k = torch.from_numpy(rng.standard_normal((T, Hkv, D)).astype(np.float32)).bfloat16().float().numpy()
    v = torch.from_numpy(rng.standard_normal((T, Hkv, D)).astype(np.float32) * 3).bfloat16().float().numpy()
    slots = rng.permutation(nb * P)[:T].astype(np.int64)
    if T > 5:
        slots[5] = -1
    ks = (np.abs(k).max(axis=(0, 2)) / 448).astype(np.float32)
    vs = np.array([1.0, 0.5, 0.01], dtype=np.float32)[:Hkv]
    return k, v, slots, ks, vs


def test_cache_write_bruteforce_fp8():
    k, v, slots, ks, vs = _tiny()
    T, Hkv, D = k.shape
    P, nb = 4, 16
    kc = np.full((nb, Hkv, P, D), 0xA5, np.uint8)
    vc = np.full((nb, Hkv, D, P), 0xA5, np.uint8)
    kc, vc, bad = kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs, FP8)
    assert not bad
    ek = np.full_like(kc, 0xA5)
    ev = np.full_like(vc, 0xA5)
    for t in range(T):
        if slots[t] < 0:
            continue
        blk, off = int(slots[t]) // P, int(slots[t]) % P
        for h in range(Hkv):
            for d in range(D):
                ek[blk, h, off, d] = e4m3.encode_bruteforce(np.float32(k[t, h, d]) / np.float32(ks[h]))
                ev[blk, h, d, off] = e4m3.encode_bruteforce(np.float32(v[t, h, d]) / np.float32(vs[h]))
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
    # sentinel bytes: exactly the unwritten slots keep 0xA5 everywhere
    written = set(int(s) for s in slots if s >= 0)
    for s in range(nb * P):
        if s not in written:
            assert np.all(kc[s // P, :, s % P, :] == 0xA5) and np.all(vc[s // P, :, :, s % P] == 0xA5)


def test_cache_write_bf16_is_bit_copy():
    k, v, slots, ks, vs = _tiny(seed=1)
    P, nb = 4, 16
    T, Hkv, D = k.shape
    kc = np.full((nb, Hkv, P, D), 0xA5A5, np.uint16)
    vc = np.full((nb, Hkv, D, P), 0xA5A5, np.uint16)
    kc, vc, bad = kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs, BF16)
    for t in range(T):
        if slots[t] < 0:
            continue
        blk, off = divmod(int(slots[t]), P)
        assert np.array_equal(kv_cache.bf16_bits_to_f32(kc[blk, :, off, :]), k[t])
        assert np.array_equal(kv_cache.bf16_bits_to_f32(vc[blk, :, :, off]), v[t])


def test_cache_write_bad_slot_flagged_and_skipped():
    k, v, slots, ks, vs = _tiny(T=4)
    slots = np.array([0, 64, 3, 1000], dtype=np.int64)  # 64 = nb*P is out of range
    kc = np.full((16, 3, 4, 8), 0xA5, np.uint8)
    vc = np.full((16, 3, 8, 4), 0xA5, np.uint8)
    kc, vc, bad = kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs, FP8)
    assert bad
    # tokens 0 and 2 written (slots 0 and 3); token 1 (slot 64) and 3 skipped
    assert np.array_equal(kc[0, :, 0, :], e4m3.quantize(k[0], ks[:, None]))
    assert np.array_equal(kc[0, :, 3, :], e4m3.quantize(k[2], ks[:, None]))
    assert np.sum(kc != 0xA5) == np.sum(kc[0, :, [0, 3], :] != 0xA5)


def test_gather_identity_vs_permuted_pages():
    k, v, _, ks, vs = _tiny(T=20, seed=2)
    P, nb = 4, 16
    for perm in (np.arange(nb), np.random.default_rng(5).permutation(nb)):
        bt = perm[:5]
        slots = (bt[np.arange(20) // P] * P + np.arange(20) % P).astype(np.int64)
        kc = np.zeros((nb, 3, P, 8), np.uint8)
        vc = np.zeros((nb, 3, 8, P), np.uint8)
        kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs, FP8)
        kk, vv = kv_cache.gather_tokens(kc, vc, bt, np.arange(20), 1)
        assert np.array_equal(kk, e4m3.quantize(k[:, 1], ks[1]))
        assert np.array_equal(vv, e4m3.quantize(v[:, 1], vs[1]))


def test_quantize_query_matches_torch_cast():
    rng = np.random.default_rng(9)
    q = torch.from_numpy(rng.standard_normal((33, 4, 64)).astype(np.float32) * 5).bfloat16().float().numpy()
    s = np.float32(0.037)
    ours = kv_cache.quantize_query(q, s)
    t = (torch.from_numpy(q) / torch.tensor(s)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, t)


def test_byte_formulas_against_pages():
    g = json.load(open(GOLD))
    for r in g["values_per_token"]:
        assert kv_cache.kv_values_per_token(r["layers"], r["kv_heads"], r["head_dim"]) == r["values"]
    for r in g["bytes_per_token"]:
        b = kv_cache.kv_bytes(r["layers"], r["kv_heads"], r["head_dim"], r["bytes"])
        assert b == r["per_token"]
        assert kv_cache.kv_bytes(r["layers"], r["kv_heads"], r["head_dim"], r["bytes"], tokens=131072) / 2 ** 30 == r["per_128k_gib"]
    for r in g["approx_total_gb"]:
        b = kv_cache.kv_bytes(r["layers"], r["kv_heads"], r["head_dim"], r["bytes"], r["tokens"], r["batch"])
        assert math.floor(b / 1e9) == r["about_gb"]
    lb = g["decode_lower_bound"]
    per_seq = {kb: kv_cache.kv_bytes(lb["layers"], lb["kv_heads"], lb["head_dim"], kb, lb["tokens"]) for kb in (1, 2)}
    for r in lb["rows"]:
        kvb = per_seq[r["kv_bytes"]]
        total_gb = (r["weights_gb"] * 1e9 + lb["batch"] * kvb) / 1e9
        assert round(total_gb, 1) == r["step_gb"]
        t = kv_cache.decode_time_lower_bound_s(r["weights_gb"] * 1e9, kvb, lb["batch"], lb["bandwidth_gbs"] * 1e9)
        # the page rounds twice in one row (20.149 ms -> 20.15 -> 20.2)
        assert abs(t * 1e3 - r["ms"]) < 0.06
        assert round(100 * lb["batch"] * kvb / (total_gb * 1e9)) == r["kv_share_pct"]
    bf = 16e9 + 3 * per_seq[2]
    f8 = 16e9 + 3 * per_seq[1]
    assert round(100 * (1 - f8 / bf)) == lb["fewer_bytes_pct_fp8_kv"]
    cap = g["capacity"]
    for r in cap["rows"]:
        per = kv_cache.kv_values_per_token(cap["layers"], cap["kv_heads"], cap["head_dim"]) * cap["tokens"] * r["kv_bits"] / 8
        assert int((cap["hbm_gb"] - cap["reserve_gb"] - r["weights_gb"]) * 1e9 // per) == r["seqs"]


def test_device_format_is_a_bijection_with_documented_positions():
    from oracle import layout
    rng = np.random.default_rng(0)
    for D, dt in ((128, np.uint8), (64, np.uint8), (64, np.uint16), (128, np.uint16)):
        info = np.iinfo(dt)
        kc = rng.integers(0, info.max + 1, (3, 2, 16, D), dtype=dt)
        vc = rng.integers(0, info.max + 1, (3, 2, D, 16), dtype=dt)
        kd, vd = layout.to_device_format(kc, vc)
        k2, v2 = layout.from_device_format(kd, vd, D, np.dtype(dt).itemsize)
        assert np.array_equal(k2, kc) and np.array_equal(v2, vc)
        es = np.dtype(dt).itemsize
        rb = D * es
        # spot positions by the documented rule, element by element
        kb = kc.view(np.uint8).reshape(3, 2, 16, rb)
        for t in (0, 3, 9, 15):
            for j in range(rb // 16):
                pj = {128: j ^ (t % 8), 64: j ^ ((t // 2) % 4), 256: (j & 8) | ((j ^ t) & 7)}[rb]
                assert np.array_equal(kd[1, 1, t * rb + pj * 16: t * rb + pj * 16 + 16], kb[1, 1, t, j * 16: j * 16 + 16])
        for d in (0, 5, D - 1):
            for t in range(16):
                if es == 1:
                    slot = [0, 1, 4, 5, 8, 9, 12, 13, 2, 3, 6, 7, 10, 11, 14, 15][t]
                    assert vd[2, 0, d * 16 + slot] == vc[2, 0, d, t]
                else:
                    half = (t // 8) ^ ((d // 4) % 2)
                    off = d * 32 + half * 16 + (t % 8) * 2
                    assert vd[2, 0, off: off + 2].view(np.uint16)[0] == vc[2, 0, d, t]
