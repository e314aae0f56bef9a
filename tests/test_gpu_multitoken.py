"""GPU parity of multi-token decode (T new tokens per sequence, causal among
them) against the float64 oracle, through the C ABI.

The pages name multi-token (MTP) decode only as a variant their target
excluded ("no MTP", page "[Kernel][SM70] Pipeline batched E5M2 XQA decode",
section "Purpose"). Same tolerance as the single-token tests.
"""
import numpy as np
import pytest

from gpu_helpers import assert_close, oracle_of, run
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EDGE = [1, 2, 3, 15, 16, 17, 31, 33, 1024, 2049, 0]


@pytest.mark.parametrize("kv_dtype", ["e5m2", "e4m3"])
@pytest.mark.parametrize("hq,hkv,t", [(8, 1, 2), (32, 4, 2), (16, 4, 3), (16, 4, 4), (4, 2, 8),
                                      (8, 8, 1)])
def test_multi_token_matches_oracle(hq, hkv, t, kv_dtype):
    w = wl.make_custom(EDGE, hq, hkv, seed=hq * 10 + t, q_len=t, kv_dtype=kv_dtype)
    out = run(w)
    assert out.shape == w.q.shape
    assert_close(out, oracle_of(w), f"G={hq // hkv} T={t} {kv_dtype}")


@pytest.mark.parametrize("merge_mode", [0, 1])
@pytest.mark.parametrize("max_ctas", [0, 7, 1])
def test_multi_token_split_counts(merge_mode, max_ctas):
    w = wl.make_custom([5, 300, 4097, 2], 32, 4, seed=7, q_len=2)
    assert_close(run(w, max_ctas=max_ctas, merge_mode=merge_mode), oracle_of(w), "split")


def test_b16_ragged_two_new_tokens():
    w = wl.make_workload("b16_ragged_ctx16384_19200", q_len=2)
    assert_close(run(w), oracle_of(w), "b16 T=2")


def test_one_new_token_in_4d_equals_single_token_bitwise():
    w = wl.make_custom([40, 1000, 7], 32, 4, seed=8)
    single = run(w)
    w4 = w.copy()
    w4.q = w.q[:, None]
    multi = run(w4)
    assert np.array_equal(single.view(np.uint16), multi[:, 0].view(np.uint16))


def test_last_new_token_equals_single_token_decode():
    w = wl.make_custom([40, 1000, 7, 300], 16, 4, seed=9, q_len=3)
    multi = run(w)
    w1 = w.copy()
    w1.q = np.ascontiguousarray(w.q[:, 2])
    assert_close(multi[:, 2], oracle_of(w1), "last token")


def test_multi_token_nhd():
    w = wl.make_custom([17, 600, 3], 16, 4, seed=10, q_len=4)
    a = run(w)
    b = run(wl.to_nhd(w))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
