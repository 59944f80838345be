"""E4M3 (OCP FP8 "FN") codec, written from the format's definition.

Test infrastructure: only the tests, the smoke check and the bench's CPU
baseline may import this module.

Sources
-------
* "FP8 and KV cache" (cooking-agi tutorial), section "Dynamic or static
  scale": E4M3's largest value is 448; a value whose quotient by the scale
  exceeds 448 is clipped to 448 in saturating mode; OCP's conversion also
  defines an overflow-to-NaN mode (not used here).
* Same page, section "How to enable it in the engine": the smallest
  subnormal is 2^-9 (about 0.00195) and 0.001 rounds up to it.
* "FP8 quantization and long-context inference" (gtnt.cn), section 1: the
  format has 4 exponent bits and 3 mantissa bits and a range of about +-448;
  section 1.1: quantizing is round(x / scale), dequantizing is q * scale.

Readings where the pages are silent
-----------------------------------
* Rounding is round-to-nearest, ties to the code with an even mantissa
  (the pages only say "round").
* NaN inputs encode to 0x7F; negative values that round to zero keep their
  sign (0x80).
* Exponent bias 7; exponent field 0 is subnormal; 0x7F / 0xFF are NaN; there
  is no infinity (the OCP E4M3 encoding the tutorial points to).

Everything is evaluated in float64, where every E4M3 value, every float32
value and every midpoint between neighbouring E4M3 values is exact.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_SUBNORMAL = 2.0 ** -9
NAN_CODE = 0x7F
SAT_CODE = 0x7E  # +448


def decode_code(code: int) -> float:
    """Value of one E4M3 byte from its sign / exponent / mantissa fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# Table of all 256 code values (float64), built field by field.
DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)

# Non-negative finite codes 0x00..0x7E in increasing order of value.
_POS_CODES = np.arange(0, 0x7F, dtype=np.int64)
_POS_VALUES = DECODE_TABLE[:0x7F].copy()
assert np.all(np.diff(_POS_VALUES) > 0)


def decode(codes) -> np.ndarray:
    """Decode an array of E4M3 bytes to float64."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(values) -> np.ndarray:
    """Saturating round-to-nearest-even encoding of float32 values.

    For each value: NaN -> 0x7F; |v| >= 448 -> sign | 0x7E; otherwise the
    finite code nearest to |v| (ties to the even code, i.e. even mantissa
    LSB), with the sign bit of v kept.  The nearest code is found by locating
    |v| between two neighbouring code values and comparing it exactly against
    their midpoint.
    """
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    nan = np.isnan(flat)
    neg = np.signbit(flat)
    a = np.abs(np.where(nan, 0.0, flat))
    sat = a >= E4M3_MAX
    a_in = np.where(sat, 0.0, a)
    lo = np.searchsorted(_POS_VALUES, a_in, side="right") - 1  # value[lo] <= a
    lo = np.clip(lo, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    mid = 0.5 * (_POS_VALUES[lo] + _POS_VALUES[hi])
    pick_hi = (a_in > mid) | ((a_in == mid) & (hi != lo) & (lo % 2 == 1))
    code = np.where(pick_hi, hi, lo)
    code = np.where(sat, SAT_CODE, code)
    code = code | np.where(neg, 0x80, 0)
    code = np.where(nan, NAN_CODE, code)
    out[:] = code.astype(np.uint8)
    return out.reshape(v.shape)


def encode_bruteforce(x: float) -> int:
    """Encode one float by scanning all 127 non-negative finite codes.

    Slow and independent of `encode`: the reference the fast path is checked
    against on small inputs.
    """
    x = float(np.float32(x))
    if np.isnan(x):
        return NAN_CODE
    s = 0x80 if np.signbit(x) else 0
    a = abs(x)
    if a >= E4M3_MAX:
        return s | SAT_CODE
    best, best_d = 0, None
    for c in range(0x7F):
        d = abs(decode_code(c) - a)
        if best_d is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    return s | best


def quantize(x, scale) -> np.ndarray:
    """q = encode(fl32(x / scale)): one correctly rounded float32 division,
    then one saturating RNE rounding to E4M3 ("FP8 quantization and
    long-context inference", section 1.1: round(w / scale); "FP8 and KV
    cache", "Dynamic or static scale": 180 divided by s is 672, saturated).
    `x` and `scale` broadcast; both are taken as float32."""
    xf = np.asarray(x, dtype=np.float32)
    sf = np.asarray(scale, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        v = (xf / sf).astype(np.float32)
    return encode(v)


def dequantize(codes, scale) -> np.ndarray:
    """x_hat = decode(q) * scale, in float64."""
    return decode(codes) * np.asarray(scale, dtype=np.float32).astype(np.float64)


_ALL_BF16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)


def quantize_bf16_table(scale) -> np.ndarray:
    """quantize() evaluated once for every bfloat16 input: uint8 [65536],
    indexed by the bf16 bit pattern.  The same function as quantize() on a
    finite domain, used to keep large test cases fast."""
    return quantize(_ALL_BF16, np.float32(scale))


def quantize_bf16_bits(bits, scale) -> np.ndarray:
    """quantize() of bfloat16 inputs given as uint16 bit patterns."""
    return quantize_bf16_table(scale)[np.asarray(bits, dtype=np.uint16)]
