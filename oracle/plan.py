"""Integer definition of the split-KV work partition.

Test infrastructure only (see the package docstring).

The page "[Kernel][WIP] Follow up FlashNext batch HC fusion and QSA route audit"
(section "Test Result") structures split-KV attention as planner -> forward ->
merge, and records that a capacity-sized grid leaves CTAs empty on short
contexts while fixed grids or contiguous grouping regress long contexts, and
that too few CTAs is catastrophic. The pages give no partition rule; the one
adopted here (a reading) sizes every split from the total work:

* a *segment* is one (sequence b, kv head g) pair, index ``s = b*Hkv + g``; it
  holds ``ceil(ctx_b / BS)`` pages (0 if ``ctx_b`` is 0 or invalid);
* segments are laid end to end, ``seg_start`` is the exclusive prefix sum of
  their page counts and ``P = seg_start[-1]`` is the total;
* the number of CTAs is ``n = 0`` if ``P == 0`` else
  ``min(max_ctas, max(1, ceil(P / min_pages_per_cta)))``;
* the work is cut on a *cost line*: the segments are laid end to end, each
  preceded by its switch cost ``seg_cost(pages)`` (32 page units for a
  non-empty segment, 0 for an empty one: a value tuned on the GPU kernel,
  which the pages do not state; with it a CTA holding many tiny segments no
  longer takes several times longer than the rest); page ``p`` of segment ``s`` sits
  at position ``p + cc[s]`` with ``cc[s]`` the sum of the costs of segments
  ``0..s``, and the line is ``V = P + cc[-1]`` long;
* CTA ``i`` owns the positions ``[floor(i*V/n), floor((i+1)*V/n))`` and so
  the pages there, a contiguous run (possibly empty): every CTA gets the same
  cost whatever the length mix, long sequences are split across CTAs, short
  ones share a CTA and many tiny ones are spread over several;
* the intersection of CTA ``i`` with segment ``s`` is a *piece*; its partial
  result slot is ``i + s`` (unique, since walking the flattened order every
  piece boundary advances ``i`` or ``s``).

A context length outside ``[0, MBS*BS]`` marks the segment bad (0 pages).
"""
from __future__ import annotations

import numpy as np


def segment_pages(context_lens, num_kv_heads: int, max_blocks_per_seq: int, block_size: int = 16):
    """Pages per segment and the bad-segment flags: (int64 [B*Hkv], bool [B*Hkv])."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    bad_seq = (ctx < 0) | (ctx > int(max_blocks_per_seq) * block_size)
    pages_seq = np.where(bad_seq, 0, (ctx + block_size - 1) // block_size)
    pages = np.repeat(pages_seq, num_kv_heads)
    bad = np.repeat(bad_seq, num_kv_heads)
    return pages.astype(np.int64), bad


def segment_starts(pages) -> np.ndarray:
    """Exclusive prefix sum with the total appended: int64 [nseg + 1]."""
    pages = np.asarray(pages, dtype=np.int64)
    out = np.zeros(pages.shape[0] + 1, dtype=np.int64)
    out[1:] = np.cumsum(pages)
    return out


SEG_COST = 32


def seg_cost(pages) -> np.ndarray:
    """Switch cost of each segment on the cost line, in page units."""
    pages = np.asarray(pages, dtype=np.int64)
    return np.where(pages <= 0, 0, SEG_COST)


def cost_prefix(seg_start) -> np.ndarray:
    """cc[s] = cost of segments 0..s (inclusive): int64 [nseg]."""
    return np.cumsum(seg_cost(np.diff(np.asarray(seg_start, dtype=np.int64)))).astype(np.int64)


def line_length(seg_start, cc) -> int:
    return int(seg_start[-1]) + (int(cc[-1]) if len(cc) else 0)


def page_position(p: int, seg_start, cc) -> int:
    """Position of flattened page p on the cost line."""
    s = int(np.searchsorted(seg_start, p, side="right") - 1)
    return int(p) + int(cc[s])


def page_at(a: int, seg_start, cc) -> int:
    """The first page at a position >= a (P if there is none)."""
    seg_start = np.asarray(seg_start, dtype=np.int64)
    for s in range(len(cc)):
        first, end = int(seg_start[s]) + int(cc[s]), int(seg_start[s + 1]) + int(cc[s])
        if end > a:
            return int(seg_start[s]) if a <= first else int(seg_start[s]) + (a - first)
    return int(seg_start[-1])


def num_ctas(total_pages: int, max_ctas: int, min_pages_per_cta: int) -> int:
    if total_pages <= 0:
        return 0
    want = -(-int(total_pages) // int(min_pages_per_cta))
    return int(min(int(max_ctas), max(1, want)))


def cta_range(i: int, seg_start, cc, n: int):
    """Flattened page range [begin, end) of CTA ``i``: its positions on the line."""
    line = line_length(seg_start, cc)
    return page_at((i * line) // n, seg_start, cc), page_at(((i + 1) * line) // n, seg_start, cc)


def cta_of_page(p: int, seg_start, cc, n: int) -> int:
    """The CTA whose range holds flattened page ``p`` (closed form on its position)."""
    return ((page_position(p, seg_start, cc) + 1) * n - 1) // line_length(seg_start, cc)


def pieces(seg_start, n: int):
    """All (cta, segment, page_begin, page_end, slot) pieces, in flattened order."""
    seg_start = np.asarray(seg_start, dtype=np.int64)
    cc = cost_prefix(seg_start)
    out = []
    for i in range(n):
        a, e = cta_range(i, seg_start, cc, n)
        if a == e:
            continue
        s = int(np.searchsorted(seg_start, a, side="right") - 1)
        while a < e:
            seg_end = int(seg_start[s + 1])
            if seg_end <= a:
                s += 1
                continue
            b_end = min(seg_end, e)
            out.append((i, s, a, b_end, i + s))
            a = b_end
            s += 1
    return out


def plan(context_lens, num_kv_heads: int, max_blocks_per_seq: int, max_ctas: int,
         min_pages_per_cta: int, block_size: int = 16) -> dict:
    """Everything the device planner publishes, as numpy/int values."""
    pages, bad = segment_pages(context_lens, num_kv_heads, max_blocks_per_seq, block_size)
    starts = segment_starts(pages)
    total = int(starts[-1])
    n = num_ctas(total, max_ctas, min_pages_per_cta)
    return {
        "seg_start": starts,
        "seg_cc": cost_prefix(starts),
        "seg_bad": bad,
        "total_pages": total,
        "num_ctas": n,
        "num_segments": int(pages.shape[0]),
    }
