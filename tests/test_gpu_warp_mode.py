"""GPU parity of the partial kernel's warp mode (through the C ABI).

Batches of many short sequences (at least four segments per CTA, none longer
than 32 pages) are worked with whole segment pieces per warp instead of every
eighth page per warp. Same tolerance as the other parity tests; the fused and
the separate merge stay bitwise equal.
"""
import numpy as np
import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from gpu_helpers import Dev, assert_close, oracle_of, run, to_dev
from oracle import plan as oplan
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MIN_PIECES, MAX_PIECE_PAGES = 4, 32  # the kernel's warp-mode rule


def _warp_mode_share(w):
    """Share of the non-empty CTA ranges that meet the warp-mode rule (0 when
    the host does not pick the warp-mode kernel): at least MIN_PIECES pieces,
    none longer than MAX_PIECE_PAGES pages. Computed from the oracle's plan, to
    show that a test batch really exercises the mode."""
    n_max = torch.cuda.get_device_properties(0).multi_processor_count
    hkv = w.num_kv_heads
    if w.batch * hkv < MIN_PIECES * n_max:
        return 0.0
    pl = oplan.plan(w.context_lens, hkv, w.block_tables.shape[1], n_max, 16)
    st, cc, n = pl["seg_start"], pl["seg_cc"], pl["num_ctas"]
    hits = ranges = 0
    for i in range(n):
        a, e = oplan.cta_range(i, st, cc, n)
        if a == e:
            continue
        ranges += 1
        s = int(np.searchsorted(st, a, side="right") - 1)
        lens = []
        while s < len(st) - 1 and st[s] < e:
            lens.append(int(min(st[s + 1], e) - max(st[s], a)))
            s += 1
        if sum(x > 0 for x in lens) >= MIN_PIECES and max(lens) <= MAX_PIECE_PAGES:
            hits += 1
    return hits / ranges


def _short_batch(seed, hq=32, hkv=4, q_len=1, kv_dtype="e5m2", batch=160):
    # 160 x 4 = 640 segments >= 4 per CTA on a 152-SM GPU; up to 25 pages each,
    # some a single token, some exactly a page or two
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, 400, size=batch)
    ctx[::17] = 16
    ctx[5::23] = 1
    ctx[7::29] = 32
    ctx = np.maximum(ctx, q_len)
    return wl.make_custom(ctx, hq, hkv, seed=seed, q_len=q_len, kv_dtype=kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["e5m2", "e4m3"])
@pytest.mark.parametrize("hq,hkv,q_len", [(32, 4, 1), (16, 4, 2), (8, 8, 1)])
def test_warp_mode_matches_oracle(kv_dtype, hq, hkv, q_len):
    w = _short_batch(101 + hq + q_len, hq, hkv, q_len, kv_dtype, batch=160 if hkv == 4 else 80)
    assert _warp_mode_share(w) > 0.5  # most ranges in warp mode, the rest in CTA mode
    a = run(w, merge_mode=0)
    b = run(w, merge_mode=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert_close(a, oracle_of(w), f"warp mode {kv_dtype} G={hq // hkv} T={q_len}")


def test_warp_mode_nhd_equals_hnd_bitwise():
    w = _short_batch(111)
    assert np.array_equal(run(w).view(np.uint16), run(wl.to_nhd(w)).view(np.uint16))


def test_warp_mode_relocation_and_determinism():
    w = _short_batch(112)
    a = run(w)
    assert np.array_equal(a.view(np.uint16), run(w).view(np.uint16))
    assert np.array_equal(a.view(np.uint16), run(wl.relocate_pages(w, seed=5)).view(np.uint16))


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_warp_mode_bad_block_id_is_contained(merge_mode):
    w = _short_batch(113)
    ref = oracle_of(w)
    bad = 37
    w.block_tables[bad, 0] = w.num_blocks + 3
    d = Dev(w, merge_mode=merge_mode)
    d.run()
    out = d.result()
    assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
    assert np.all(np.isnan(out[bad].astype(np.float32)))
    good = [b for b in range(w.batch) if b != bad]
    assert_close(out[good], ref[good], "rows beside a bad block id (warp mode)")


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_warp_mode_leaves_the_tickets_at_zero(merge_mode):
    # split pieces in warp mode take the same self-clearing merge tickets as in
    # CTA mode; after good and bad calls the ticket words must be zero again
    w = _short_batch(114)
    assert _warp_mode_share(w) > 0.5
    ref = oracle_of(w)
    d = Dev(w, merge_mode=merge_mode)
    for bad in (False, True, False):
        if bad:
            d.bt[11, 0] = w.num_blocks + 5
        else:
            d.bt.copy_(to_dev(w.block_tables))
        d.run()
        out = d.result()
        torch.cuda.synchronize()
        tickets = d.ws[64:64 + 8 * 1024].cpu().numpy().view(np.int32)
        assert np.all(tickets == 0)
        if bad:
            assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
            assert np.all(np.isnan(out[11].astype(np.float32)))
        else:
            assert d.status() == xqa.XQA_OK
            assert_close(out, ref, "warp mode")
