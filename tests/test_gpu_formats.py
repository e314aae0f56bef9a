"""GPU parity of the E4M3 KV format, the NHD cache layout and device-pointer
scales (through the C ABI).

E4M3 is the FP8 format the page "[Kernel][WIP] Follow up FlashNext batch HC
fusion and QSA route audit" (section "Test Result") lists as not yet admitted
beside E5M2. Same tolerance as the E5M2 tests: |gpu - ref| <= 2e-3 + 1e-2*|ref|.
"""
import functools

import numpy as np
import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from gpu_helpers import Dev, assert_close, oracle_of, run, to_dev
from oracle import e4m3
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def e4m3_workload(name):
    return wl.make_workload(name, kv_dtype="e4m3")


def _codes_both_parities():
    a = np.arange(256, dtype=np.uint8)
    return np.concatenate([a, np.roll(a, 8)])  # each code meets both conversion routes


def test_e4m3_fp16_bits_exact_all_codes():
    codes = _codes_both_parities()
    bits, f32 = xqa.xqa_dequant_e4m3(torch.from_numpy(codes).cuda(), 0.25)
    torch.cuda.synchronize()
    got = bits.cpu().numpy().view(np.float16).astype(np.float64)
    ref = e4m3.decode_closed_form(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))
    assert np.all(np.isnan(got[~fin]))
    f = f32.cpu().numpy().astype(np.float64)
    assert np.array_equal(f[fin], 0.25 * ref[fin])


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_e4m3_workload_matches_oracle(name):
    w = e4m3_workload(name)
    assert_close(run(w), oracle_of(w), f"{name} e4m3")


def test_e4m3_single_token_is_the_v_row_exactly():
    # exact value equality (a -0 code comes out as +0: the accumulator starts at +0)
    w = wl.make_custom([1, 1], 16, 2, seed=41, kv_dtype="e4m3", v_scale=0.5)
    out = run(w)
    for b in range(2):
        for h in range(16):
            want = (e4m3.decode_closed_form(w.v_cache[w.block_tables[b, 0], h // 8, 0]) * 0.5)
            assert np.array_equal(out[b, h].astype(np.float64), want.astype(np.float16).astype(np.float64))


@pytest.mark.parametrize("kv_dtype", ["e5m2", "e4m3"])
@pytest.mark.parametrize("name", ["b16_ragged_ctx16384_19200", "b12_boundary"])
def test_nhd_layout_equals_hnd_bitwise(name, kv_dtype):
    w = wl.make_workload(name, kv_dtype=kv_dtype) if kv_dtype == "e4m3" else wl.make_workload(name)
    a = run(w)
    b = run(wl.to_nhd(w))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    if name == "b12_boundary":
        assert_close(b, oracle_of(wl.to_nhd(w)), "nhd")


def test_nhd_poisoned_neighbours_are_never_read():
    # in NHD a page interleaves all kv heads: poison the other heads' rows and
    # the tail slots; the output must not change
    w = wl.to_nhd(wl.make_custom([7, 40, 33], 8, 2, seed=42))
    clean = run(w)
    p = w.copy()
    for b in range(3):
        ctx = int(p.context_lens[b])
        last = p.block_tables[b, (ctx + 15) // 16 - 1]
        if ctx % 16:
            p.k_cache[last, ctx % 16:] = 0x7B
            p.v_cache[last, ctx % 16:] = 0x7B
    assert np.array_equal(clean.view(np.uint16), run(p).view(np.uint16))


@pytest.mark.parametrize("kv_dtype", ["e5m2", "e4m3"])
def test_device_scales_equal_host_scales_bitwise(kv_dtype):
    w = wl.make_custom([100, 3000, 17], 32, 4, seed=43, kv_dtype=kv_dtype, k_scale=0.75,
                       v_scale=1.5)
    d = Dev(w)
    d.run()
    host = d.result().copy()
    ks = torch.tensor([0.75], dtype=torch.float32, device="cuda")
    vs = torch.tensor([1.5], dtype=torch.float32, device="cuda")
    d.out.fill_(float("nan"))
    xqa.xqa_decode(d.q, d.k, d.v, d.bt, d.lens, ks, vs, out=d.out, workspace=d.ws, shape=d.shape)
    dev = d.result()
    assert np.array_equal(host.view(np.uint16), dev.view(np.uint16))
    assert_close(dev, oracle_of(w), "device scales")


def test_graph_replay_reads_new_device_scales():
    w = wl.make_custom([64, 500, 2049], 32, 4, seed=44)
    d = Dev(w)
    ks = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    vs = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        xqa.xqa_decode(d.q, d.k, d.v, d.bt, d.lens, ks, vs, out=d.out, workspace=d.ws,
                       shape=d.shape, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            xqa.xqa_decode(d.q, d.k, d.v, d.bt, d.lens, ks, vs, out=d.out, workspace=d.ws,
                           shape=d.shape, stream=s)
    torch.cuda.synchronize()
    ks.fill_(0.5)
    vs.fill_(2.0)
    d.out.fill_(float("nan"))
    g.replay()
    got = d.result()
    w2 = w.copy()
    w2.k_scale, w2.v_scale = 0.5, 2.0
    assert_close(got, oracle_of(w2), "replayed with new scales")


def test_e4m3_split_and_merge_modes_agree_bitwise():
    w = e4m3_workload("b12_boundary")
    a = run(w, merge_mode=0)
    b = run(w, merge_mode=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
