"""Pins of the oracle's work-partition definition (CPU only).

The partition is integer work, so its pins are brute force: the cost line is
built item by item (each segment's switch cost, then its pages), cut into n
runs of positions whose lengths differ by at most one; every flattened page is
owned by exactly one CTA, the closed forms for a CTA's page range and for
"which CTA owns page p" agree with that walk, pieces tile every segment
exactly, and piece slots are unique and below ``n + nseg``.
"""
import numpy as np
import pytest

from oracle import plan


def _walk(starts, n):
    """Brute force: the line as a list of items (-1 cost unit, else a page),
    each position given to CTA floor-division owner."""
    items = []
    for s in range(len(starts) - 1):
        pages = int(starts[s + 1] - starts[s])
        items += [-1] * int(plan.seg_cost([pages])[0])
        items += list(range(int(starts[s]), int(starts[s + 1])))
    V = len(items)
    bounds = [(i * V) // n for i in range(n + 1)]
    owner = np.full(int(starts[-1]), -1)
    for i in range(n):
        for pos in range(bounds[i], bounds[i + 1]):
            if items[pos] >= 0:
                owner[items[pos]] = i
    return owner, bounds, V


@pytest.mark.parametrize("seed", range(16))
def test_partition_brute_force(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 20))
    hkv = int(rng.integers(1, 5))
    mbs = int(rng.integers(1, 40))
    ctx = rng.integers(0, mbs * 16 + 1, size=B)
    ctx[rng.random(B) < 0.2] = 0
    small = rng.random(B) < 0.3  # many short segments: the switch cost dominates
    ctx[small] = np.minimum(rng.integers(1, 8 * 16, size=int(small.sum())), mbs * 16)
    max_ctas = int(rng.integers(1, 160))
    minp = int(rng.integers(1, 12))
    p = plan.plan(ctx, hkv, mbs, max_ctas, minp)
    starts, total, n, cc = p["seg_start"], p["total_pages"], p["num_ctas"], p["seg_cc"]
    pages = np.diff(starts)
    assert np.array_equal(pages, np.repeat((ctx + 15) // 16, hkv))
    costs = np.where(pages == 0, 0, 32)
    assert np.array_equal(cc, np.cumsum(costs))
    if total == 0:
        assert n == 0
        return
    assert 1 <= n <= max_ctas
    assert n == min(max_ctas, -(-total // minp))
    owner, bounds, V = _walk(starts, n)
    assert V == plan.line_length(starts, cc)
    assert max(np.diff(bounds)) - min(np.diff(bounds)) <= 1
    assert np.all(owner >= 0)
    for i in range(n):
        a, e = plan.cta_range(i, starts, cc, n)
        assert np.all(owner[a:e] == i)
        assert np.sum(owner == i) == e - a
    for pg in range(total):
        assert plan.cta_of_page(pg, starts, cc, n) == owner[pg]
        assert plan.page_at(plan.page_position(pg, starts, cc), starts, cc) == pg
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


def test_tiny_segments_are_spread_over_ctas():
    # sixteen one-page segments ahead of one long sequence: with page counts
    # alone CTA 0 would hold all sixteen; on the cost line it holds a few
    ctx = [16] * 16 + [16 * 2000]
    p = plan.plan(ctx, 1, 2000, 64, 8)
    starts, cc, n = p["seg_start"], p["seg_cc"], p["num_ctas"]
    owners = [plan.cta_of_page(int(starts[s]), starts, cc, n) for s in range(16)]
    per_cta = np.bincount(owners)
    assert per_cta.max() <= 5
    assert len(set(owners)) >= 4


def test_every_segment_costs_a_fixed_amount():
    # two equal long segments over two CTAs: the cut lands mid-line, i.e. in
    # the middle of the pages once both switch costs are counted
    p = plan.plan([16 * 100, 16 * 100], 1, 100, 2, 1)
    starts, cc, n = p["seg_start"], p["seg_cc"], p["num_ctas"]
    assert list(cc) == [32, 64]
    assert plan.cta_range(0, starts, cc, 2) == (0, 100)
    assert plan.cta_range(1, starts, cc, 2) == (100, 200)


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
