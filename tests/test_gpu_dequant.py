"""Bit-exact GPU E5M2 dequantisation against the oracle (all 256 codes, both routes).

The exhaustive code proof pattern follows the page "[Kernel][SM70] Fold DeepSeek
V4 MXFP4 decode exponents" (section "Test Result"): every code, every route.
"""
import numpy as np
import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from oracle import e5m2

pytestmark = pytest.mark.gpu


def _codes_both_parities():
    a = np.arange(256, dtype=np.uint8)
    # 8-byte groups alternate between the two conversion routes; rolling by 8
    # swaps the parity of every group, so each code meets both routes
    return np.concatenate([a, np.roll(a, 8)])


@pytest.mark.parametrize("n_extra", [0, 3])
def test_fp16_bits_exact_all_codes(n_extra):
    codes = np.concatenate([_codes_both_parities(), np.arange(n_extra, dtype=np.uint8)])
    bits, _ = xqa.xqa_dequant_e5m2(torch.from_numpy(codes).cuda(), 1.0, with_f32=False)
    torch.cuda.synchronize()
    got = bits.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, e5m2.fp16_bits(codes))


@pytest.mark.parametrize("scale", [1.0, 0.5, 2.0**-12])
def test_scaled_values_exact(scale):
    codes = _codes_both_parities()
    _, f32 = xqa.xqa_dequant_e5m2(torch.from_numpy(codes).cuda(), scale)
    torch.cuda.synchronize()
    got = f32.cpu().numpy().astype(np.float64)
    ref = e5m2.dequantize(codes, scale)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_large_random_buffer():
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 256, size=1_000_003, dtype=np.uint8)
    bits, _ = xqa.xqa_dequant_e5m2(torch.from_numpy(codes).cuda(), 1.0, with_f32=False)
    torch.cuda.synchronize()
    assert np.array_equal(bits.cpu().numpy().view(np.uint16), e5m2.fp16_bits(codes))
