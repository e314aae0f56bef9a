"""Pins of the oracle's E5M2 decode (CPU only).

The decode must be bit-exact on all 256 codes. It is pinned three independent
ways: the closed-form route against the fp16-view route, both against torch's
float8_e5m2 cast (a library routine), and both against the landmark values of
the E5M2 encoding in ``tests/golden/e5m2_landmarks.txt``. The exhaustive
all-codes check follows the exhaustive bit-pattern proof pattern on the page
"[Kernel][SM70] Fold DeepSeek V4 MXFP4 decode exponents" (section "Test Result").
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import e5m2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e5m2_landmarks.txt")
ALL = np.arange(256, dtype=np.uint8)


def _same(a, b):
    """Bitwise float64 equality, NaN == NaN, and signed zeros distinguished."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.all(both_nan | (a.view(np.uint64) == b.view(np.uint64)))


def test_closed_form_equals_fp16_view_all_codes():
    assert _same(e5m2.decode_closed_form(ALL), e5m2.decode_fp16_view(ALL))


def test_matches_torch_float8_e5m2_all_codes():
    ref = torch.from_numpy(ALL.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    assert _same(e5m2.decode_fp16_view(ALL), ref)
    assert _same(e5m2.decode_closed_form(ALL), ref)


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            rows.append((int(code, 16), val))
    return rows


@pytest.mark.parametrize("route", [e5m2.decode_closed_form, e5m2.decode_fp16_view])
def test_landmark_values(route):
    rows = _golden()
    assert len(rows) >= 20
    for code, val in rows:
        got = float(route(np.array([code], np.uint8))[0])
        if val == "nan":
            assert math.isnan(got), hex(code)
        elif val in ("inf", "-inf"):
            assert got == float(val), hex(code)
        else:
            assert Fraction(got) == Fraction(val), hex(code)
            if val.startswith("-"):
                assert math.copysign(1.0, got) < 0, hex(code)


def test_finite_codes_are_strictly_increasing_and_symmetric():
    v = e5m2.decode_fp16_view(ALL)
    pos = v[:0x7C]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(v[0x80:0xFC], -pos)
    assert pos.max() == 57344.0
    assert np.count_nonzero(np.isfinite(v)) == 248
    assert np.count_nonzero(np.isnan(v)) == 6


def test_fp16_bits_are_the_code_shifted_into_the_high_byte():
    bits = e5m2.fp16_bits(ALL)
    assert bits.dtype == np.uint16
    assert np.array_equal(bits >> 8, ALL.astype(np.uint16))
    assert np.all((bits & 0xFF) == 0)


def test_dequantize_scales_exactly_for_power_of_two_scales():
    for scale in (1.0, 0.5, 2.0**-12):
        got = e5m2.dequantize(ALL, scale)
        fin = np.isfinite(got)
        exact = [Fraction(float(x)) * Fraction(scale) for x in e5m2.decode_closed_form(ALL)[fin]]
        assert all(Fraction(float(g)) == x for g, x in zip(got[fin], exact))
