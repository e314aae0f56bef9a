"""CPU oracle for paged E5M2-KV grouped-query decode attention.

TEST INFRASTRUCTURE ONLY. This package is the slow, plain, obviously-correct
statement of what the decode path computes, in float64 numpy. Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path (the CUDA library and its Python binding) never
does, and shares no code, table or constant with it.

Modules:

* :mod:`oracle.e5m2` — E5M2 code -> value, by the closed form of the format and
  by the fp16 bit-view route (the two are checked against each other).
* :mod:`oracle.attention` — masked softmax attention over the paged cache.
* :mod:`oracle.plan` — the integer work partition the device planner must
  reproduce bit-exactly (pages per (sequence, kv head), equal page shares per
  CTA, piece slots).

Every function here is pinned by ``-m "not gpu"`` tests against closed forms,
a library routine, brute force and invariants; none is "parity unpinned".
"""
