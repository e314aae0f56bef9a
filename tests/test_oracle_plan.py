"""Pins of the oracle's work-partition definition (CPU only).

The partition is integer work, so its pins are brute force: every flattened
page is owned by exactly one CTA, shares differ by at most one page, the closed
form for "which CTA owns page p" agrees with the ranges, pieces tile every
segment exactly, and piece slots are unique and below ``n + nseg``.
"""
import numpy as np
import pytest

from oracle import plan


@pytest.mark.parametrize("seed", range(12))
def test_partition_brute_force(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 20))
    hkv = int(rng.integers(1, 5))
    mbs = int(rng.integers(1, 40))
    ctx = rng.integers(0, mbs * 16 + 1, size=B)
    ctx[rng.random(B) < 0.2] = 0
    max_ctas = int(rng.integers(1, 160))
    minp = int(rng.integers(1, 12))
    p = plan.plan(ctx, hkv, mbs, max_ctas, minp)
    starts, total, n = p["seg_start"], p["total_pages"], p["num_ctas"]
    pages = np.diff(starts)
    assert np.array_equal(pages, np.repeat((ctx + 15) // 16, hkv))
    if total == 0:
        assert n == 0
        return
    assert 1 <= n <= max_ctas
    assert n == min(max_ctas, -(-total // minp))
    owner = np.full(total, -1)
    sizes = []
    for i in range(n):
        a, e = plan.cta_range(i, total, n)
        sizes.append(e - a)
        assert np.all(owner[a:e] == -1)
        owner[a:e] = i
    assert np.all(owner >= 0)
    assert max(sizes) - min(sizes) <= 1
    for pg in range(total):
        assert plan.cta_of_page(pg, total, n) == owner[pg]
    pcs = plan.pieces(starts, n)
    slots = [x[4] for x in pcs]
    assert len(set(slots)) == len(slots)
    assert max(slots) < n + len(pages)
    covered = np.zeros(total, int)
    for i, s, a, e, slot in pcs:
        assert starts[s] <= a < e <= starts[s + 1]
        assert owner[a] == i and owner[e - 1] == i
        assert slot == i + s
        covered[a:e] += 1
    assert np.all(covered == 1)


def test_invalid_context_marks_segment_bad_with_no_pages():
    p = plan.plan([16, -1, 33, 10_000], 2, 4, 8, 1)
    assert list(p["seg_bad"]) == [False, False, True, True, False, False, True, True]
    assert list(np.diff(p["seg_start"])) == [1, 1, 0, 0, 3, 3, 0, 0]


def test_num_ctas_edges():
    assert plan.num_ctas(0, 152, 8) == 0
    assert plan.num_ctas(1, 152, 8) == 1
    assert plan.num_ctas(16, 152, 8) == 2
    assert plan.num_ctas(17, 152, 8) == 3
    assert plan.num_ctas(10**6, 152, 8) == 152
