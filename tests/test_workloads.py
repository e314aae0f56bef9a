"""Checks of the seeded input generators (CPU only)."""
import numpy as np
import pytest
import torch

from paged_fp8_kv_gqa_gb300 import workloads as wl


def test_encoder_matches_torch_on_every_in_range_fp16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16)
    ok = np.isfinite(x) & (np.abs(x.astype(np.float64)) <= 57344.0)
    mine = wl.fp16_to_e5m2_rne(x[ok])
    ref = torch.from_numpy(x[ok].copy()).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_encoder_saturates():
    x = np.array([60000.0, -65504.0, 61439.0], np.float16)
    assert list(wl.fp16_to_e5m2_rne(x)) == [0x7B, 0xFB, 0x7B]


def test_finite_codes():
    f = wl.finite_e5m2_codes()
    assert f.shape == (248,)
    assert 0x7B in f and 0x7C not in f and 0xFB in f and 0xFF not in f


@pytest.mark.parametrize("name", wl.WORKLOADS[:2] + (wl.WORKLOADS[4],))
def test_workload_structure(name):
    w = wl.make_workload(name)
    B, hq, D = w.q.shape
    assert D == 128 and w.block_size == 16 and hq % w.num_kv_heads == 0
    npages = (w.context_lens.astype(np.int64) + 15) // 16
    used = []
    for b in range(B):
        row = w.block_tables[b]
        assert np.all(row[: npages[b]] >= 0) and np.all(row[: npages[b]] < w.num_blocks)
        assert np.all(row[npages[b]:] == -1)
        used.extend(row[: npages[b]].tolist())
        n = int(w.context_lens[b])
        if n % 16:
            last = row[npages[b] - 1]
            assert np.all(w.k_cache[last, :, n % 16:] == wl.POISON_CODE)
            assert np.all(w.v_cache[last, :, n % 16:] == wl.POISON_CODE)
    assert len(used) == len(set(used))
    unused = np.setdiff1d(np.arange(w.num_blocks), used)
    if unused.size:
        assert np.all(w.k_cache[unused] == wl.POISON_CODE)
    # no inf/NaN codes inside any context
    for b in range(B):
        n = int(w.context_lens[b])
        pages = w.block_tables[b, : npages[b]]
        for cache in (w.k_cache, w.v_cache):
            codes = cache[pages].transpose(0, 2, 1, 3).reshape(-1, w.num_kv_heads, D)[:n]
            assert np.all(((codes >> 2) & 0x1F) != 0x1F)


def test_named_shapes():
    w = wl.make_workload("tiny_b1_ctx256")
    assert w.q.shape == (1, 8, 128) and w.num_blocks == 16
    assert np.array_equal(w.block_tables[0], np.arange(16))
    w = wl.make_workload("b4_uniform_ctx1024")
    assert w.num_blocks == 4096 and w.k_scale == 0.5 and list(w.context_lens) == [1024] * 4
    w = wl.make_workload("b12_boundary")
    assert tuple(w.context_lens) == wl.BOUNDARY_CONTEXTS and w.k_scale == 2.0**-12
    assert w.kv_bytes == 76849 * 4 * 128 * 2
    # the 32768-token sequence carries every finite code in its first 248 tokens
    b = wl.BOUNDARY_CONTEXTS.index(32768)
    first = w.k_cache[w.block_tables[b, :16]].transpose(0, 2, 1, 3).reshape(256, 4, 128)[:248]
    assert set(np.unique(first).tolist()) == set(wl.finite_e5m2_codes().tolist())


def test_ragged_lengths_and_determinism():
    a = wl.make_workload("b16_ragged_ctx16384_19200")
    assert a.q.shape == (16, 32, 128)
    assert np.all((a.context_lens >= 16384) & (a.context_lens <= 19200))
    b = wl.make_workload("b16_ragged_ctx16384_19200")
    assert np.array_equal(a.context_lens, b.context_lens)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.block_tables, b.block_tables)


def test_relocation_keeps_logical_kv():
    w = wl.make_custom([5, 40, 17], 8, 2, seed=1)
    r = wl.relocate_pages(w, seed=2)
    assert not np.array_equal(r.block_tables, w.block_tables)
    for b in range(3):
        n = int(w.context_lens[b])
        np_ = (n + 15) // 16
        a = w.k_cache[w.block_tables[b, :np_]]
        c = r.k_cache[r.block_tables[b, :np_]]
        assert np.array_equal(a, c)
