"""FP8 (E4M3) K/V pages -- quantisation and dequantisation, plain definitions.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The KV-cache tutorial ("KV Cache complete guide", §6.2 KVQuant and
per-channel quantisation) quantises every channel d of head h with its own
scale s_{h,d} (and zero point z_{h,d}) so that a few outlier channels do not
set the range of all the others, and names FP8 as what serving engines use in
practice; §6.3 dequantises as code times scale and writes the attention score
over the dequantised keys.  The reading this oracle takes (the library
documents the same one):

  * symmetric: zero point 0;
  * one scale per (layer, KV head, dimension), one set for K and one for V;
  * code = E4M3(x * r) with r = fp32(1 / s), the product x * r in fp32,
    rounded to the nearest E4M3 value (ties to an even mantissa) and
    saturated at +-448 (no infinities are produced);
  * the stored value is decode(code) * s.

E4M3 (the OCP 8-bit floating-point format): a sign bit, four exponent bits
with bias 7, three mantissa bits.  Exponent field 0 holds the subnormals
m * 2^-9; fields 1..15 hold (1 + m/8) * 2^(e-7); the format has no
infinities, and S.1111.111 is NaN, so the largest finite magnitude is
1.75 * 2^8 = 448.

Pins (tests/test_fp8_oracle.py): decoded values of hand-picked codes, every
code against torch's float8_e4m3fn, the round trip of all finite codes, ties,
saturation, subnormals and the half-ulp error bound.
"""
from __future__ import annotations

import numpy as np

MAX = 448.0


def decode(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8 array), float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


# the 127 non-negative finite values, in code order (which is value order)
_POS = decode(np.arange(127, dtype=np.uint8))


def encode(x) -> np.ndarray:
    """Nearest E4M3 code of each value (float64 array): ties go to the even
    code (mantissa bit 0 clear), magnitudes at or above 448 and infinities
    saturate to +-448, NaN maps to 0x7F; the sign is kept (a negative value
    that rounds to zero gives 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    finite = np.isfinite(a)
    a_f = np.where(finite, a, MAX)
    # lower neighbour: the last value <= a
    lo = np.clip(np.searchsorted(_POS, a_f, side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    d_lo = a_f - _POS[lo]
    d_hi = _POS[hi] - a_f
    up = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1))
    code = np.where(up, hi, lo)
    code = np.where(a_f >= MAX, 126, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


def quantize(x, scale) -> np.ndarray:
    """Codes of values x [..., d] with per-channel scales scale [d]: the
    product x * fp32(1 / scale) is taken in fp32, then rounded to E4M3."""
    r = (np.float32(1.0) / f32(scale)).astype(np.float32)
    prod = (f32(x) * r).astype(np.float32)
    return encode(prod.astype(np.float64))


def dequantize(codes, scale) -> np.ndarray:
    """Stored values: decode(code) * scale, float64."""
    return decode(codes) * np.asarray(scale, dtype=np.float64)
