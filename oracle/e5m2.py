"""E5M2 (OCP FP8) codec, written from the format's definition.

Test infrastructure: only the tests, the smoke check and the bench's CPU
baseline may import this module.

Sources
-------
* "FP8 quantization and long-context inference" (gtnt.cn), section 1, the
  format table: E5M2 has 5 exponent bits and 2 mantissa bits and a range of
  about +-57344 (against +-448 for E4M3); section 1.1: quantizing is
  round(x / scale), dequantizing is q * scale.
* "FP8 and KV cache" (cooking-agi tutorial), section "How to enable it in
  the engine": fp8_e5m2 is one of the KV-cache dtypes the engine accepts;
  section "Dynamic or static scale": out-of-range quotients saturate in the
  saturating conversion mode.

Readings where the pages are silent
-----------------------------------
* The OCP E5M2 encoding, which keeps IEEE conventions: exponent bias 15,
  exponent field 0 is subnormal (m/4 * 2^-14), exponent field 31 holds
  infinity (mantissa 0) and NaN (mantissa != 0).  Largest finite value
  1.75 * 2^15 = 57344 (code 0x7B), smallest subnormal 2^-16 (code 0x01).
* Conversion as for E4M3 in this library: round to nearest, ties to the
  even mantissa, saturating to +-57344 (infinity is never produced); NaN
  encodes to 0x7F; negative values that round to zero keep their sign.

Everything is evaluated in float64, where every E5M2 value, every float32
value and every midpoint between neighbouring E5M2 values is exact.
"""
from __future__ import annotations

import numpy as np

E5M2_MAX = 57344.0
E5M2_MIN_SUBNORMAL = 2.0 ** -16
NAN_CODE = 0x7F
SAT_CODE = 0x7B  # +57344


def decode_code(code: int) -> float:
    """Value of one E5M2 byte from its sign / exponent / mantissa fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 2) & 0x1F
    m = code & 0x3
    if e == 0x1F:
        return sign * float("inf") if m == 0 else float("nan")
    if e == 0:
        return sign * (m / 4.0) * 2.0 ** -14
    return sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)


# Table of all 256 code values (float64), built field by field.
DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)

# Non-negative finite codes 0x00..0x7B in increasing order of value.
_POS_VALUES = DECODE_TABLE[:SAT_CODE + 1].copy()
assert np.all(np.diff(_POS_VALUES) > 0)


def decode(codes) -> np.ndarray:
    """Decode an array of E5M2 bytes to float64."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(values) -> np.ndarray:
    """Saturating round-to-nearest-even encoding of float32 values.

    NaN -> 0x7F; |v| >= 57344 -> sign | 0x7B; otherwise the finite code
    nearest to |v| (ties to the even mantissa), found by locating |v| between
    two neighbouring code values and comparing it exactly with their
    midpoint, with the sign bit of v kept."""
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    flat = v.reshape(-1)
    nan = np.isnan(flat)
    neg = np.signbit(flat)
    a = np.abs(np.where(nan, 0.0, flat))
    sat = a >= E5M2_MAX
    a_in = np.where(sat, 0.0, a)
    lo = np.searchsorted(_POS_VALUES, a_in, side="right") - 1  # value[lo] <= a
    lo = np.clip(lo, 0, SAT_CODE)
    hi = np.minimum(lo + 1, SAT_CODE)
    mid = 0.5 * (_POS_VALUES[lo] + _POS_VALUES[hi])
    pick_hi = (a_in > mid) | ((a_in == mid) & (hi != lo) & (lo % 2 == 1))
    code = np.where(pick_hi, hi, lo)
    code = np.where(sat, SAT_CODE, code)
    code = code | np.where(neg, 0x80, 0)
    code = np.where(nan, NAN_CODE, code)
    return code.astype(np.uint8).reshape(v.shape)


def encode_bruteforce(x: float) -> int:
    """Encode one float by scanning all 124 non-negative finite codes (slow,
    independent of `encode`)."""
    x = float(np.float32(x))
    if np.isnan(x):
        return NAN_CODE
    s = 0x80 if np.signbit(x) else 0
    a = abs(x)
    if a >= E5M2_MAX:
        return s | SAT_CODE
    best, best_d = 0, None
    for c in range(SAT_CODE + 1):
        d = abs(decode_code(c) - a)
        if best_d is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    return s | best


def quantize(x, scale) -> np.ndarray:
    """q = encode(fl32(x / scale)): one correctly rounded float32 division,
    then one saturating RNE rounding to E5M2 ("FP8 quantization and
    long-context inference", section 1.1: round(w / scale))."""
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
    """quantize() for every bfloat16 input: uint8 [65536] indexed by the bf16
    bit pattern (the same function on a finite domain, for speed)."""
    return quantize(_ALL_BF16, np.float32(scale))


def quantize_bf16_bits(bits, scale) -> np.ndarray:
    """quantize() of bfloat16 inputs given as uint16 bit patterns."""
    return quantize_bf16_table(scale)[np.asarray(bits, dtype=np.uint16)]
