"""E5M2 (FP8, 1 sign / 5 exponent / 2 mantissa bits, bias 15) decoding in float64.

Test infrastructure only (see the package docstring).

The KV cache of the page "[Kernel][SM70] Pipeline batched E5M2 XQA decode"
(section "Purpose": FP8 E5M2 KV) stores one E5M2 code per element. The decode
is exact: every E5M2 value is an fp16 value, namely the fp16 whose high byte is
the code and whose low byte is zero. Two independent routes are given here and
tests check them against each other, against exact rational arithmetic and
against torch's float8_e5m2 cast on all 256 codes.
"""
from __future__ import annotations

import numpy as np


def decode_closed_form(codes) -> np.ndarray:
    """Value of each code by the format's closed form.

    For code x: s = x >> 7, e = (x >> 2) & 31, m = x & 3.
      e == 0       -> (-1)^s * 2^-14 * m/4      (zero and subnormals)
      1 <= e <= 30 -> (-1)^s * 2^(e-15) * (1 + m/4)
      e == 31      -> +-inf if m == 0 else NaN
    """
    x = np.asarray(codes, dtype=np.int64)
    s = (x >> 7) & 1
    e = (x >> 2) & 31
    m = (x & 3).astype(np.float64)
    sign = np.where(s == 1, -1.0, 1.0)
    sub = sign * np.ldexp(m / 4.0, -14)
    norm = sign * np.ldexp(1.0 + m / 4.0, (e - 15).astype(np.int64))
    special = np.where(m == 0, sign * np.inf, np.nan)
    out = np.where(e == 0, sub, np.where(e == 31, special, norm))
    return out.astype(np.float64)


def decode_fp16_view(codes) -> np.ndarray:
    """Value of each code via the fp16 bit pattern ``code << 8``, widened to float64."""
    x = np.asarray(codes, dtype=np.uint8).astype(np.uint16) << np.uint16(8)
    with np.errstate(invalid="ignore"):
        return x.view(np.float16).astype(np.float64)


def fp16_bits(codes) -> np.ndarray:
    """The fp16 bit pattern an exact dequantisation must produce: ``code << 8``."""
    return np.asarray(codes, dtype=np.uint8).astype(np.uint16) << np.uint16(8)


def lut() -> np.ndarray:
    """float64 value of all 256 codes (index = code), via the fp16-view route."""
    return decode_fp16_view(np.arange(256, dtype=np.uint8))


def dequantize(codes, scale: float) -> np.ndarray:
    """Scaled value ``scale * decode(code)`` in float64 (scale taken as given)."""
    with np.errstate(invalid="ignore"):
        return lut()[np.asarray(codes, dtype=np.uint8)] * float(scale)
