"""Pins of the oracle's E4M3 codec against what the pages and the format fix.

* worked examples printed in "FP8 and KV cache" (tests/golden);
* closed forms of the format: max 448, min subnormal 2^-9, two NaN codes;
* a library special case: torch's float8_e4m3fn cast (round-to-nearest-even,
  not saturating) agrees with the oracle on inputs clamped to +-448;
* brute force over all codes on random and tie inputs;
* invariants: decode(encode(decode(c))) == decode(c) for every finite code.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLD = os.path.join(os.path.dirname(__file__), "golden", "e4m3_worked_examples.json")


def test_closed_forms():
    t = e4m3.DECODE_TABLE
    fin = t[np.isfinite(t)]
    assert np.max(fin) == 448.0 and np.min(fin) == -448.0
    assert np.min(fin[fin > 0]) == 2.0 ** -9
    assert np.sum(np.isnan(t)) == 2 and np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert fin.size == 254
    # largest normal 1.75 * 2^8, smallest normal 2^-6, largest subnormal 7/8 * 2^-6
    assert t[0x7E] == 1.75 * 2 ** 8 and t[0x08] == 2.0 ** -6 and t[0x07] == 0.875 * 2 ** -6
    # sign symmetry
    for c in range(0x7F):
        assert t[c | 0x80] == -t[c]


def test_worked_examples_from_pages():
    g = json.load(open(GOLD))
    assert e4m3.E4M3_MAX == g["e4m3_max"]["value"]
    assert e4m3.E4M3_MIN_SUBNORMAL == g["min_subnormal"]["value"]
    assert abs(g["min_subnormal"]["value"] - g["min_subnormal"]["approx_page"]) < 5e-6
    for s in g["scale_values"]:
        assert abs(np.float32(s["num"]) / np.float32(s["den"]) - s["approx"]) <= s["tol"]
    for ex in g["readback"]:
        s = np.float32(np.float32(ex["scale_num"]) / np.float32(ex["scale_den"]))
        code = e4m3.quantize(np.float32(ex["x"]), s)
        back = float(e4m3.dequantize(code, s))
        assert abs(back - ex["readback"]) <= ex["tol"], ex
        if "rel_err_pct" in ex:
            assert round(abs(back - ex["x"]) / ex["x"] * 100, 1) == ex["rel_err_pct"]
        if "quotient" in ex:
            assert np.float32(ex["x"]) / s == pytest.approx(ex["quotient"], rel=1e-6)
            assert int(code) == 0x7E


def test_specific_codes():
    s = np.float32(3.2) / np.float32(448.0)
    assert int(e4m3.quantize(np.float32(0.01), s)) == 0x3B       # 1.375
    assert int(e4m3.quantize(np.float32(-0.8), s)) == 0xEE       # -112
    assert int(e4m3.quantize(np.float32(3.2), s)) == 0x7E        # 448
    s2 = np.float32(120.0) / np.float32(448.0)
    assert int(e4m3.quantize(np.float32(0.01), s2)) == 0x12      # 0.0390625
    assert int(e4m3.encode(np.float32(-1e-5))) == 0x80           # signed zero kept
    assert int(e4m3.encode(np.float32(-0.0))) == 0x80
    assert int(e4m3.encode(np.float32(0.0))) == 0x00
    assert int(e4m3.encode(np.float32(np.nan))) == 0x7F
    assert int(e4m3.encode(np.float32(np.inf))) == 0x7E
    assert int(e4m3.encode(np.float32(-np.inf))) == 0xFE
    assert int(e4m3.encode(np.float32(1e30))) == 0x7E
    # ties: 2^-10 is halfway between 0 and 2^-9 -> even (0); 3*2^-10 -> 2^-8 (even code 2)
    assert int(e4m3.encode(np.float32(2.0 ** -10))) == 0x00
    assert int(e4m3.encode(np.float32(3 * 2.0 ** -10))) == 0x02
    # 432 is halfway between 416 (0x7D, odd) and 448 (0x7E, even)
    assert int(e4m3.encode(np.float32(432.0))) == 0x7E
    assert int(e4m3.encode(np.float32(431.99))) == 0x7D


def _torch_reference(x):
    """torch's e4m3fn cast (RNE, NaN on overflow) after clamping to +-448."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    t = torch.where(torch.isnan(t), t, t.clamp(-448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_against_torch_dense_bit_sample():
    # every 257th float32 bit pattern (~16.7M values), all exponents and signs
    bits = np.arange(0, 2 ** 32, 257, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    ours = e4m3.encode(x)
    ref = _torch_reference(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(ours[nan] == 0x7F)


def test_against_torch_ties_and_neighbours():
    vals = e4m3.DECODE_TABLE[:0x7F]
    mids = 0.5 * (vals[:-1] + vals[1:])
    pts = np.concatenate([vals, mids]).astype(np.float32)
    around = [pts]
    for k in (1, 2):
        around.append(np.nextafter(pts, np.float32(np.inf), dtype=np.float32))
        around.append(np.nextafter(pts, np.float32(-np.inf), dtype=np.float32))
        pts_k = around[-1]
    x = np.concatenate(around)
    x = np.concatenate([x, -x])
    assert np.array_equal(e4m3.encode(x), _torch_reference(x))


def test_against_bruteforce():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(2000) * 10.0 ** rng.uniform(-4, 3, 2000),
        0.5 * (e4m3.DECODE_TABLE[1:0x7F] + e4m3.DECODE_TABLE[:0x7E]),
        [0.0, -0.0, 448.0, 447.99, 500.0, -500.0, 2 ** -10, 2 ** -11, 1e-9],
    ]).astype(np.float32)
    fast = e4m3.encode(x)
    slow = np.array([e4m3.encode_bruteforce(v) for v in x], dtype=np.uint8)
    assert np.array_equal(fast, slow)


def test_roundtrip_invariant():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes)
    again = e4m3.encode(vals.astype(np.float32))
    assert np.array_equal(e4m3.decode(again), vals)
    # every finite code except -0 maps back to itself
    nz = codes != 0x80
    assert np.array_equal(again[nz], codes[nz])


def test_quantize_divides_in_float32():
    # x / s rounded to float32 first, then to E4M3: pick x, s where the float64
    # quotient and the float32 quotient land on different sides of a midpoint
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200000).astype(np.float32)
    s = np.float32(0.0123)
    q = e4m3.quantize(x, s)
    ref = _torch_reference((x / s).astype(np.float32))
    assert np.array_equal(q, ref)


def test_bf16_table_equals_quantize():
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    for s in (1.0, 0.0123, 3.2 / 448, 120 / 448, 1e-3):
        t = e4m3.quantize_bf16_table(s)
        fin = ~np.isnan(x)
        assert np.array_equal(t[fin], e4m3.quantize(x[fin], np.float32(s)))
