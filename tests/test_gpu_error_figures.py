"""Error figures of every workload in both FP8 formats (through the C ABI).

The stated bound is max abs error 2e-3 and max rel error 1e-2 on the fp16
outputs against the float64 oracle. The parity tests apply it element by
element as |gpu - ref| <= 2e-3 + 1e-2*|ref|; here the two figures are also
measured separately: max abs over all elements, max rel over the elements
with |ref| > 2e-3. The outputs of all five workloads stay below 4 in
magnitude, where one fp16 rounding step is at most 9.8e-4, so the abs bound
is asserted outright for every workload and format. Max rel is reported, not
asserted: next to |ref| = 2e-3 the rounding of the softmax weights to fp16
alone can reach 1e-2 of the output.

Run with ``-s`` to see the table; with XQA_ERROR_TABLE=<path> it is also
written to that file.
"""
import functools
import os

import numpy as np
import pytest

from gpu_helpers import ATOL, assert_close, oracle_of, run
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

_ROWS = []


@functools.lru_cache(maxsize=None)
def _workload(name, kv_dtype):
    return wl.make_workload(name, kv_dtype=kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["e5m2", "e4m3"])
@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_error_figures(name, kv_dtype):
    w = _workload(name, kv_dtype)
    ref = oracle_of(w)
    got = run(w)
    stats = assert_close(got, ref, f"{name} {kv_dtype}")  # the combined bound, every element
    assert stats["max_abs"] <= ATOL, (name, kv_dtype, stats)
    _ROWS.append((name, kv_dtype, stats["max_abs"], stats["max_rel"],
                  float(np.abs(ref).max())))


def test_zz_print_error_table():
    if not _ROWS:
        pytest.skip("no figures collected in this run")
    lines = ["| workload | format | max abs | max rel (abs(ref) > 2e-3) | max abs(ref) |",
             "|---|---|---|---|---|"]
    for name, fmt, a, r, m in _ROWS:
        lines.append(f"| {name} | {fmt} | {a:.3e} | {r:.3e} | {m:.3g} |")
    table = "\n".join(lines)
    print("\n" + table)
    path = os.environ.get("XQA_ERROR_TABLE")
    if path:
        with open(path, "w") as f:
            f.write(table + "\n")
