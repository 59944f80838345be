"""Pins of the oracle's E5M2 codec and of the E5M2 cache path.

* the format's range from "FP8 quantization and long-context inference"
  (section 1 table: about +-57344) and its closed forms;
* E5M2 is the top byte of an IEEE binary16: the decode table against
  numpy's float16 for all 256 codes;
* encode against an integer round-half-even of float16 bit patterns (every
  float16 input), against torch's float8_e5m2 cast (inputs clamped to the
  range, since that cast does not saturate), and against brute force;
* the cache write and decode attention with an E5M2 cache against
  per-element brute force and the plain softmax definition.
"""
import math

import numpy as np
import torch

from oracle import attention, e4m3, e5m2, kv_cache


def test_closed_forms_and_page_range():
    t = e5m2.DECODE_TABLE
    fin = t[np.isfinite(t)]
    # gtnt section 1: E5M2 reaches about +-57344, E4M3 about +-448
    assert e5m2.E5M2_MAX == 57344.0 and np.max(fin) == 57344.0 and np.min(fin) == -57344.0
    assert e4m3.E4M3_MAX == 448.0
    assert t[0x7B] == 1.75 * 2 ** 15
    assert np.min(fin[fin > 0]) == 2.0 ** -16 == e5m2.E5M2_MIN_SUBNORMAL
    assert t[0x04] == 2.0 ** -14 and t[0x03] == 0.75 * 2.0 ** -14  # smallest normal, largest subnormal
    assert t[0x7C] == math.inf and t[0xFC] == -math.inf
    assert np.sum(np.isnan(t)) == 6
    assert fin.size == 248
    for c in range(0x7C):
        assert t[c | 0x80] == -t[c]


def test_decode_table_is_the_top_byte_of_float16():
    ref = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    t = e5m2.DECODE_TABLE
    assert np.array_equal(np.isnan(ref), np.isnan(t))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], t[ok])


def test_encode_every_float16_against_integer_rounding():
    h = np.arange(65536, dtype=np.uint32)
    mag = h & 0x7FFF
    finite = mag < 0x7C00
    # round half to even on the low 8 bits of the magnitude, then saturate at 0x7B
    r = (mag + 0x7F + ((mag >> 8) & 1)) >> 8
    r = np.minimum(r, 0x7B)
    want = (r | ((h >> 15) << 7)).astype(np.uint8)
    x = h.astype(np.uint16).view(np.float16).astype(np.float32)
    got = e5m2.encode(x)
    assert np.array_equal(got[finite], want[finite])
    # infinities saturate, NaN maps to 0x7F
    assert e5m2.encode(np.float32(np.inf)) == 0x7B and e5m2.encode(np.float32(-np.inf)) == 0xFB
    assert e5m2.encode(np.float32(np.nan)) == 0x7F


def test_encode_against_torch_cast():
    g = np.random.default_rng(5)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.uniform(-6, 5, 20000),
                        (e5m2.DECODE_TABLE[:0x7B] + e5m2.DECODE_TABLE[1:0x7C]) / 2]).astype(np.float32)
    x = np.concatenate([x, -x])
    clamped = np.clip(x, -57344.0, 57344.0).astype(np.float32)
    ref = torch.from_numpy(clamped).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(e5m2.encode(x), ref)


def test_encode_against_bruteforce_and_round_trip():
    g = np.random.default_rng(6)
    x = (g.standard_normal(600) * 10.0 ** g.uniform(-6, 5, 600)).astype(np.float32)
    x = np.concatenate([x, [0.0, -0.0, 57344.0, 61439.0, 61440.0, 1e9, 2.0 ** -17, 2.0 ** -18, -3.0 * 2 ** -18]])
    fast = e5m2.encode(x)
    for xi, c in zip(x, fast):
        assert c == e5m2.encode_bruteforce(xi), xi
    codes = np.array([c for c in range(256) if np.isfinite(e5m2.DECODE_TABLE[c])], dtype=np.uint8)
    assert np.array_equal(e5m2.encode(e5m2.decode(codes).astype(np.float32)), codes)


def test_quantize_is_one_division_then_one_rounding():
    x = np.float32(180.0)
    s = np.float32(np.float32(0.3))
    q = (x / s).astype(np.float32)
    assert e5m2.quantize(x, s) == e5m2.encode_bruteforce(q)
    # values beyond the range saturate: 1e6 / 1 -> 57344
    assert e5m2.dequantize(e5m2.quantize(np.float32(1e6), np.float32(1.0)), 1.0) == 57344.0


def _tiny_cache(g, T=37, Hkv=2, D=64, P=16):
    nb = (T + P - 1) // P + 2
    k = (g.standard_normal((T, Hkv, D)) * 3).astype(np.float32)
    v = (g.standard_normal((T, Hkv, D)) * 3).astype(np.float32)
    k = torch.from_numpy(k).to(torch.bfloat16).float().numpy()
    v = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    perm = g.permutation(nb)
    slots = np.array([perm[t // P] * P + t % P for t in range(T)], dtype=np.int64)
    ks = (np.abs(k).max(axis=(0, 2)) / 57344.0 * 300).astype(np.float32)
    vs = (np.abs(v).max(axis=(0, 2)) / 57344.0 * 300).astype(np.float32)
    kc = np.full((nb, Hkv, P, D), 0xA5, np.uint8)
    vc = np.full((nb, Hkv, D, P), 0xA5, np.uint8)
    kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs, kv_cache.FP8_E5M2)
    bt = np.array([perm[: (T + P - 1) // P]], dtype=np.int32)
    return k, v, slots, kc, vc, ks, vs, bt


def test_cache_write_e5m2_bruteforce():
    g = np.random.default_rng(7)
    k, v, slots, kc, vc, ks, vs, bt = _tiny_cache(g)
    T, Hkv, D = k.shape
    for t in range(T):
        blk, off = slots[t] // 16, slots[t] % 16
        for h in range(Hkv):
            for d in range(0, D, 7):
                qk = np.float32(np.float32(k[t, h, d]) / ks[h])
                qv = np.float32(np.float32(v[t, h, d]) / vs[h])
                assert kc[blk, h, off, d] == e5m2.encode_bruteforce(qk)
                assert vc[blk, h, d, off] == e5m2.encode_bruteforce(qv)


def test_decode_e5m2_against_definition():
    g = np.random.default_rng(8)
    k, v, slots, kc, vc, ks, vs, bt = _tiny_cache(g)
    T, Hkv, D = k.shape
    Hq = 4
    q = torch.from_numpy(g.standard_normal((1, Hq, D)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    sm = 1.0 / math.sqrt(D)
    out, lse = attention.paged_decode(q, kc, vc, ks, vs, bt, np.array([T]), sm, cache_dtype=kv_cache.FP8_E5M2,
                                      mode="pure")
    mir, _ = attention.paged_decode(q, kc, vc, ks, vs, bt, np.array([T]), sm, cache_dtype=kv_cache.FP8_E5M2,
                                    mode="mirror")
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        kh = np.array([[e5m2.decode_code(kc[slots[t] // 16, kv, slots[t] % 16, d]) * float(ks[kv])
                        for d in range(D)] for t in range(T)])
        vh = np.array([[e5m2.decode_code(vc[slots[t] // 16, kv, d, slots[t] % 16]) * float(vs[kv])
                        for d in range(D)] for t in range(T)])
        s = [sm * sum(float(q[0, h, d]) * kh[t, d] for d in range(D)) for t in range(T)]
        m = max(s)
        p = [math.exp(x - m) for x in s]
        ref = sum(p[t] * vh[t] for t in range(T)) / sum(p)
        assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-12)
        assert abs(lse[0, h] - (m + math.log(sum(p)))) < 1e-12
    # the mirrored query rounding moves the result by far less than the test tolerance
    assert np.max(np.abs(mir - out)) < 2e-3


def test_prefill_over_an_e5m2_cache_non_causal_rows_equal_decode():
    """Prefill over an E5M2 cache: a non-causal row is decode attention of
    the dequantized E4M3 query over the same E5M2 codes (pure mode)."""
    from oracle import attention
    rng = np.random.default_rng(31)
    L, Hkv, Hq, D, nq = 90, 2, 4, 16, 6
    k = torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).bfloat16().float().numpy()
    v = torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).bfloat16().float().numpy()
    nb = -(-L // 16) + 2
    bt = rng.permutation(nb)[: -(-L // 16)].astype(np.int32)[None, :]
    slots = bt[0][np.arange(L) // 16].astype(np.int64) * 16 + np.arange(L) % 16
    ks = np.full(Hkv, np.abs(k).max() / 57344, np.float32)
    vs = np.full(Hkv, np.abs(v).max() / 57344, np.float32)
    kc = np.zeros((nb, Hkv, 16, D), np.uint8)
    vc = np.zeros((nb, Hkv, D, 16), np.uint8)
    kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs, kv_cache.FP8_E5M2)
    qs = np.float32(0.01)
    q8 = kv_cache.quantize_query(rng.standard_normal((nq, Hq, D)).astype(np.float32), qs)
    out = attention.prefill(q8, qs, kc, vc, ks, vs, bt, np.array([0, nq]), np.array([L]), 0.3, causal=False,
                            mode="pure", cache_dtype=kv_cache.FP8_E5M2)
    qdq = (e4m3.decode(q8) * float(qs)).astype(np.float32)
    for i in range(nq):
        dec, _ = attention.paged_decode(qdq[i:i + 1], kc, vc, ks, vs, bt, np.array([L]), 0.3, mode="pure",
                                        cache_dtype=kv_cache.FP8_E5M2)
        assert np.allclose(out[i], dec[0], rtol=1e-6, atol=1e-7)
    # and it is not the E4M3 reading of the same bytes
    wrong = attention.prefill(q8, qs, kc, vc, ks, vs, bt, np.array([0, nq]), np.array([L]), 0.3, causal=False,
                              mode="pure")
    assert not np.allclose(out, wrong, rtol=1e-2)
