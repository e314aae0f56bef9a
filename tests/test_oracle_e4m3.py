"""Pins of the oracle's E4M3 decode and of the E4M3 / NHD options of the
attention oracle (CPU only).

E4M3 decoding is pinned three ways on all 256 codes: the closed form against
an independent field-rebuilding route, both against torch's float8_e4m3fn
cast (a library routine), and both against the landmark values of the format
in tests/golden/e4m3_landmarks.txt. The NHD cache layout is pinned by
bitwise equality with the HND result of the same logical cache.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import attention, e4m3
from paged_fp8_kv_gqa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_landmarks.txt")
ALL = np.arange(256, dtype=np.uint8)


def _same(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.all((np.isnan(a) & np.isnan(b)) | (a.view(np.uint64) == b.view(np.uint64)))


def _torch_e4m3(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8).copy()).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_two_routes_and_torch_agree_on_all_codes():
    c, f, t = e4m3.decode_closed_form(ALL), e4m3.decode_by_fields(ALL), _torch_e4m3(ALL)
    assert _same(c, f) and _same(c, t)


@pytest.mark.parametrize("route", [e4m3.decode_closed_form, e4m3.decode_by_fields])
def test_landmarks(route):
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        got = float(route(np.array([int(code, 16)], np.uint8))[0])
        n += 1
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert Fraction(got) == Fraction(val), code
            if val.startswith("-"):
                assert math.copysign(1.0, got) < 0
    assert n >= 20


def test_format_structure():
    v = e4m3.decode_closed_form(ALL)
    assert np.count_nonzero(np.isnan(v)) == 2 and not np.any(np.isinf(v))
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0) and pos.max() == 448.0
    assert np.array_equal(v[0x80:0xFF], -pos)


def test_planted_bias_mistake_is_caught():
    import inspect

    src = inspect.getsource(e4m3.decode_closed_form).replace("(e - 7)", "(e - 8)")
    ns = {"np": np}
    exec(src, ns)
    bad = ns["decode_closed_form"](ALL)
    fin = np.isfinite(_torch_e4m3(ALL))
    assert not np.array_equal(bad[fin], _torch_e4m3(ALL)[fin])


def test_encoder_matches_torch_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16)
    ok = np.isfinite(x) & (np.abs(x.astype(np.float64)) <= 448.0)
    mine = wl.float_to_e4m3_rne(x[ok].astype(np.float32))
    ref = torch.from_numpy(x[ok].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)
    assert list(wl.float_to_e4m3_rne(np.array([500.0, -1e4], np.float32))) == [0x7E, 0xFE]


def _sdpa_e4m3(w):
    table = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64)
    out = np.zeros(w.q.shape)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        n = int(w.context_lens[b])
        if n == 0:
            continue
        idx = [(int(w.block_tables[b, t // 16]), t % 16) for t in range(n)]
        K = torch.stack([table[torch.from_numpy(w.k_cache[p, :, s].astype(np.int64))] for p, s in idx], 1)
        V = torch.stack([table[torch.from_numpy(w.v_cache[p, :, s].astype(np.int64))] for p, s in idx], 1)
        K = (K * w.k_scale).repeat_interleave(G, 0)
        V = (V * w.v_scale).repeat_interleave(G, 0)
        Q = torch.from_numpy(w.q[b].astype(np.float64))[:, None, :]
        out[b] = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], V[None])[0, :, 0].numpy()
    return out


def test_e4m3_attention_against_sdpa():
    w = wl.make_custom([5, 40, 17, 1], 8, 2, seed=4, kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    got = attention.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                           w.context_lens, w.k_scale, w.v_scale, kv_dtype="e4m3")
    assert np.allclose(got, _sdpa_e4m3(w), rtol=1e-12, atol=1e-12)


def test_e4m3_single_token_is_the_v_row():
    w = wl.make_custom([1, 1], 8, 2, seed=5, kv_dtype="e4m3", v_scale=0.25)
    got = attention.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                           w.context_lens, 1.0, 0.25, kv_dtype="e4m3")
    for b in range(2):
        for h in range(8):
            assert np.array_equal(got[b, h], 0.25 * e4m3.decode_closed_form(
                w.v_cache[w.block_tables[b, 0], h // 4, 0]))


@pytest.mark.parametrize("kv_dtype", ["e5m2", "e4m3"])
def test_nhd_layout_gives_the_hnd_result_bitwise(kv_dtype):
    w = wl.make_custom([3, 33, 64, 0, 100], 16, 4, seed=6, kv_dtype=kv_dtype)
    n = wl.to_nhd(w)
    assert n.k_cache.shape == (w.num_blocks, 16, 4, 128) and n.num_kv_heads == 4
    a = attention.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                         w.context_lens, 1.0, 1.0, kv_dtype=kv_dtype)
    b = attention.paged_decode_attention(n.q, n.k_cache, n.v_cache, n.block_tables,
                                         n.context_lens, 1.0, 1.0, kv_dtype=kv_dtype,
                                         kv_layout="nhd")
    assert np.all(np.isfinite(a)) and np.array_equal(a, b)


def test_e4m3_workloads_hold_no_nan_inside_contexts():
    w = wl.make_workload("b12_boundary", kv_dtype="e4m3")
    assert w.kv_dtype == "e4m3" and w.k_scale == 2.0**-6
    for b in range(w.batch):
        n = int(w.context_lens[b])
        pages = w.block_tables[b, : (n + 15) // 16]
        codes = w.k_cache[pages].transpose(0, 2, 1, 3).reshape(-1, 4, 128)[:n]
        assert np.all((codes & 0x7F) != 0x7F)
