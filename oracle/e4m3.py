"""E4M3 (FP8, 1 sign / 4 exponent / 3 mantissa bits, bias 7) decoding in float64.

Test infrastructure only (see the package docstring).

E4M3 is the other FP8 KV-cache format; the page "[Kernel][WIP] Follow up
FlashNext batch HC fusion and QSA route audit" (section "Test Result") names
E4M3 quality as not yet admitted beside the E5M2 path. Unlike E5M2, an E4M3
code is not the high byte of its fp16 value, so decoding is a real conversion.
The format (OCP 8-bit floating point, E4M3 "fn" variant): no infinities, the
two codes S.1111.111 are NaN, everything else is finite.
"""
from __future__ import annotations

import numpy as np


def decode_closed_form(codes) -> np.ndarray:
    """Value of each code by the format's closed form.

    For code x: s = x >> 7, e = (x >> 3) & 15, m = x & 7.
      e == 0            -> (-1)^s * 2^-6 * m/8            (zero and subnormals)
      e == 15 and m == 7 -> NaN
      otherwise         -> (-1)^s * 2^(e-7) * (1 + m/8)
    """
    x = np.asarray(codes, dtype=np.int64)
    s = (x >> 7) & 1
    e = (x >> 3) & 15
    m = (x & 7).astype(np.float64)
    sign = np.where(s == 1, -1.0, 1.0)
    sub = sign * np.ldexp(m / 8.0, -6)
    norm = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    out = np.where(e == 0, sub, norm)
    out = np.where((e == 15) & (m == 7), np.nan, out)
    return out.astype(np.float64)


def decode_by_fields(codes) -> np.ndarray:
    """A second route: rebuild an fp32 bit pattern from the fields and widen.

    A normal code moves its exponent from bias 7 to fp32's bias 127 and its 3
    mantissa bits to the top of fp32's 23; a subnormal is m * 2^-9 exactly.
    """
    x = np.asarray(codes, dtype=np.uint8).astype(np.uint32)
    s = (x >> 7) & 1
    e = (x >> 3) & 15
    m = x & 7
    bits = (s << 31) | ((e + 120) << 23) | (m << 20)
    normal = bits.view(np.float32).astype(np.float64)
    sub = np.where(s == 1, -1.0, 1.0) * m.astype(np.float64) * 2.0**-9
    out = np.where(e == 0, sub, normal)
    with np.errstate(invalid="ignore"):
        out = np.where((e == 15) & (m == 7), np.nan, out)
    return out


def lut() -> np.ndarray:
    """float64 value of all 256 codes (index = code), via the closed form."""
    return decode_closed_form(np.arange(256, dtype=np.uint8))
