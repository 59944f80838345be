"""Pins of the oracle's per-token dynamic scales (cache write and decode).

* the worked example of "FP8 and KV cache", "Dynamic or static scale"
  (tests/golden): the scales of tokens A = [0.01, -0.8, 3.2] and
  B = [2.0, -45, 180] come out as 3.2/448 and 180/448 from the tokens
  themselves, each token's maximum lands on 448, and 0.01 reads back 0.0098;
* a special case that reduces to the per-head path: when every token of a
  head has the same maximum, per-token scales equal the per-head amax / 448
  scale, and cache bytes and decode results are identical;
* decode against the plain softmax definition by brute force;
* the all-zero token (scale 1.0, zero codes).
"""
import json
import math
import os

import numpy as np
import torch

from oracle import attention, e4m3, e5m2, kv_cache

GOLD = os.path.join(os.path.dirname(__file__), "golden", "e4m3_worked_examples.json")


def _gold():
    g = json.load(open(GOLD))
    approx = {(s["num"], s["den"]): s for s in g["scale_values"]}
    return g, approx


def _write_tokens(tokens, cache_dtype=kv_cache.FP8):
    x = np.array(tokens, dtype=np.float32)[:, None, :]  # [T][1][D]
    T, _, D = x.shape
    kc = np.zeros((1, 1, 16, D), np.uint8)
    vc = np.zeros((1, 1, D, 16), np.uint8)
    sc = np.zeros((1, 1, 2, 16), np.float32)
    kv_cache.reshape_and_cache_per_token(x, x, np.arange(T), kc, vc, sc, cache_dtype)
    return kc, vc, sc[:, :, 0], sc[:, :, 1]


def test_worked_example_per_token_scales():
    g, approx = _gold()
    A = [0.01, -0.8, 3.2]
    B = [2.0, -45.0, 180.0]
    kc, vc, ksc, vsc = _write_tokens([A, B])
    sA, sB = float(ksc[0, 0, 0]), float(ksc[0, 0, 1])
    # the scales are found from the tokens' own maxima and match the page's figures
    assert sA == float(np.float32(np.float32(3.2) / np.float32(448.0)))
    assert abs(sA - approx[(3.2, 448.0)]["approx"]) <= approx[(3.2, 448.0)]["tol"]
    assert abs(sB - approx[(180.0, 448.0)]["approx"]) <= approx[(180.0, 448.0)]["tol"]
    assert np.array_equal(ksc, vsc)
    # each token's largest value lands on 448 (code 0x7E)
    assert kc[0, 0, 0, 2] == 0x7E and kc[0, 0, 1, 2] == 0x7E
    # read-backs the page prints for the dynamic scale
    for ex in g["readback"]:
        if ex["scale_num"] != 3.2:
            continue
        d = A.index(ex["x"])
        back = float(e4m3.decode(kc[0, 0, 0, d])) * sA
        assert abs(back - ex["readback"]) <= ex["tol"], ex
    back_b = e4m3.decode(kc[0, 0, 1]) * sB
    assert np.allclose(back_b, B, rtol=2.0 ** -4)


def _case(g, lens, Hkv=2, D=64, same_amax=False, cache_dtype=kv_cache.FP8):
    P = 16
    T = sum(lens)
    x = lambda: torch.from_numpy(g.standard_normal((T, Hkv, D)).astype(np.float32) * 2).to(
        torch.bfloat16).float().numpy()
    k, v = x(), x()
    if same_amax:  # every token of a head reaches the same maximum, in channel 0
        for arr in (k, v):
            m = np.abs(arr).max(axis=(0, 2)) * 1.01
            arr[:, :, 0] = torch.from_numpy(m[None, :].repeat(T, 0)).to(torch.bfloat16).float().numpy()
            arr[:, :, 1:] = np.clip(arr[:, :, 1:], -arr[:, :, :1], arr[:, :, :1])
    pages = [(L + P - 1) // P for L in lens]
    nb = sum(pages) + 3
    perm = g.permutation(nb)
    bt = np.zeros((len(lens), max(pages)), np.int32)
    slots, at = [], 0
    for b, L in enumerate(lens):
        bt[b, :pages[b]] = perm[at:at + pages[b]]
        at += pages[b]
        slots += [bt[b, t // P] * P + t % P for t in range(L)]
    kc = np.full((nb, Hkv, P, D), 0xA5, np.uint8)
    vc = np.full((nb, Hkv, D, P), 0xA5, np.uint8)
    sc = np.full((nb, Hkv, 2, P), np.nan, np.float32)
    kv_cache.reshape_and_cache_per_token(k, v, np.array(slots), kc, vc, sc, cache_dtype)
    return k, v, np.array(slots), kc, vc, sc, bt


def test_equal_maxima_reduce_to_per_head_scales():
    g = np.random.default_rng(21)
    lens = [40, 17]
    k, v, slots, kc, vc, sc, bt = _case(g, lens, same_amax=True)
    kh = (np.abs(k).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
    vh = (np.abs(v).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
    kc2 = np.full_like(kc, 0xA5)
    vc2 = np.full_like(vc, 0xA5)
    kv_cache.reshape_and_cache(k, v, slots, kc2, vc2, kh, vh, kv_cache.FP8)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)
    q = torch.from_numpy(g.standard_normal((2, 8, 64)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    sl = np.array(lens)
    for mode in ("pure", "mirror"):
        a, la = attention.paged_decode_per_token(q, kc, vc, sc, bt, sl, 0.125, mode=mode)
        b, lb = attention.paged_decode(q, kc2, vc2, kh, vh, bt, sl, 0.125, mode=mode)
        assert np.allclose(a, b, rtol=0, atol=1e-12) and np.allclose(la, lb, rtol=0, atol=1e-12)


def test_decode_per_token_against_definition():
    g = np.random.default_rng(22)
    for cache_dtype in (kv_cache.FP8, kv_cache.FP8_E5M2):
        fmt = e4m3 if cache_dtype == kv_cache.FP8 else e5m2
        lens = [29]
        k, v, slots, kc, vc, sc, bt = _case(g, lens, Hkv=1, D=32, cache_dtype=cache_dtype)
        ksc, vsc = sc[:, :, 0], sc[:, :, 1]
        q = torch.from_numpy(g.standard_normal((1, 2, 32)).astype(np.float32)).to(torch.bfloat16).float().numpy()
        out, lse = attention.paged_decode_per_token(q, kc, vc, sc, bt, np.array(lens), 0.2, mode="pure",
                                                    cache_dtype=cache_dtype)
        mir, _ = attention.paged_decode_per_token(q, kc, vc, sc, bt, np.array(lens), 0.2, mode="mirror",
                                                  cache_dtype=cache_dtype)
        for h in range(2):
            rows = []
            for t in range(lens[0]):
                blk, off = slots[t] // 16, slots[t] % 16
                kh = [fmt.decode_code(kc[blk, 0, off, d]) * float(ksc[blk, 0, off]) for d in range(32)]
                vh = [fmt.decode_code(vc[blk, 0, d, off]) * float(vsc[blk, 0, off]) for d in range(32)]
                sm = float(np.float32(0.2))  # the softmax scale is a float32 input
                rows.append((sm * sum(float(q[0, h, d]) * kh[d] for d in range(32)), vh))
            m = max(s for s, _ in rows)
            w = [math.exp(s - m) for s, _ in rows]
            ref = [sum(w[t] * rows[t][1][d] for t in range(len(rows))) / sum(w) for d in range(32)]
            assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-12)
            assert abs(lse[0, h] - (m + math.log(sum(w)))) < 1e-12
        assert np.max(np.abs(mir - out)) < 2e-3


def test_zero_token_gets_unit_scale():
    kc, vc, ksc, vsc = _write_tokens([[0.0, 0.0, -0.0], [1.0, 2.0, 4.0]])
    assert ksc[0, 0, 0] == 1.0 and np.all(kc[0, 0, 0] & 0x7F == 0)
    assert ksc[0, 0, 1] == np.float32(np.float32(4.0) / np.float32(448.0))
    kc5, _, ksc5, _ = _write_tokens([[1.0, 2.0, 4.0]], kv_cache.FP8_E5M2)
    assert ksc5[0, 0, 0] == np.float32(np.float32(4.0) / np.float32(57344.0)) and kc5[0, 0, 0, 2] == 0x7B


def test_per_token_device_layout_round_trip_and_tail_position():
    """The per-token V page is the V codes followed by the scale tail:
    K scale of slot t at byte P*D + 4t, V scale at P*D + 64 + 4t."""
    from oracle import layout
    rng = np.random.default_rng(3)
    nb, H, D = 3, 2, 64
    kc = rng.integers(0, 256, (nb, H, 16, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, H, D, 16), dtype=np.uint8)
    sc = rng.random((nb, H, 2, 16)).astype(np.float32)
    kd, vd = layout.to_device_format_per_token(kc, vc, sc)
    assert kd.shape == (nb, H, 16 * D) and vd.shape == (nb, H, 16 * D + 128)
    for t in (0, 7, 15):
        assert vd[1, 1, 16 * D + 4 * t: 16 * D + 4 * t + 4].view(np.float32)[0] == sc[1, 1, 0, t]
        assert vd[2, 0, 16 * D + 64 + 4 * t: 16 * D + 68 + 4 * t].view(np.float32)[0] == sc[2, 0, 1, t]
    k2, v2, s2 = layout.from_device_format_per_token(kd, vd, D)
    assert np.array_equal(k2, kc) and np.array_equal(v2, vc) and np.array_equal(s2, sc)
