"""Host-side helpers of bench.py (no GPU): the clock summary, quantiles, the
code hash that decides whether the committed ncu traffic still applies, and
the committed profile summary's machine-read lines."""
import os
import re

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1;  // note\n/* block\n   comment */ const char* s = "// kept";\n'
           "char q = '\"'; asm(\"mov.b32 %0, %1; // in a string\");\n")
    out = bench._code_only(src)
    assert "note" not in out and "block" not in out
    assert '"// kept"' in out and "'\"'" in out and "// in a string" in out
    assert out == bench._code_only(src.replace("  // note", "  // another note"))
    assert out != bench._code_only(src.replace("a = 1", "a = 2"))


def test_kernel_hash_ignores_comment_edits_only():
    path = os.path.join(ROOT, bench.KERNEL_SOURCES[0])
    text = open(path, encoding="utf-8").read()
    base = bench._code_only(text)
    assert bench._code_only(text.replace("// ", "//  edited ", 5)) == base
    assert "__launch_bounds__(kThreads, 1)" in text
    changed = text.replace("__launch_bounds__(kThreads, 1)", "__launch_bounds__(kThreads, 2)", 1)
    assert bench._code_only(changed) != base


def test_profile_summary_lines_parse_and_match_the_kv_bytes():
    text = open(bench.PROFILE_SUMMARY).read()
    src = re.search(r"^kernel_source_sha256: ([0-9a-f]{16})$", text, re.M)
    traffic = re.search(r"^dram_bytes_per_launch: (\d+)$", text, re.M)
    assert src and traffic
    kv_bytes = 286_227_456  # sum of B16 ragged contexts x 4 kv heads x 256 B
    # DRAM traffic of one launch: every KV byte once, plus q, tables and outputs
    assert kv_bytes <= int(traffic.group(1)) <= 1.02 * kv_bytes


def test_summarize_clocks_median_max_and_reasons():
    rows = [
        ["0", "2070", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["0", "1980", "2070", "1100", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["0", "2070", "2070", "1000", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["0", "[N/A]", "2070", "1000", "0x0", "", "", "", ""],
    ]
    c = bench.summarize_clocks(rows)
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    assert bench.summarize_clocks([]) is None


def test_quantile_matches_numpy_linear():
    rng = np.random.default_rng(3)
    for n in (1, 2, 5, 17):
        v = sorted(rng.normal(size=n).tolist())
        for q in (0.0, 0.1, 0.5, 0.9, 1.0):
            assert abs(bench._quantile(v, q) - np.quantile(v, q)) < 1e-12


def test_stamp_breakdown_on_synthetic_stamps():
    # three CTAs past the wait at t = 1000 ns; CTA 2 holds no pages
    st = np.zeros((3, 10), np.int64)
    st[0, :8] = [500, 1000, 1500, 3000, 43000, 44000, 45000, 46000]
    st[1, :8] = [600, 1100, 1600, 3500, 45000, 45500, 47000, 48000]
    st[2, :8] = [700, 1200, 0, 0, 0, 0, 0, 1300]
    st[0, 8:] = [100, 1]
    st[1, 8:] = [120, 2]
    b = bench.stamp_breakdown(st, 4096)
    assert b["ctas_with_work"] == 2
    assert b["first_pages_us"] == 2.25 and b["first_pages_last_cta_us"] == 2.5
    assert b["pages_done_last_us"] == 44.0 and b["exit_last_us"] == 47.0
    rate = 100 * 4096 / 40000 + 120 * 4096 / 41500  # bytes per ns = GB/s
    assert abs(b["steady_gbs"] - rate) < 1e-9
    assert b["pages_per_cta_min_max"] == [100, 120]


def test_stamp_columns_per_cta():
    st = np.zeros((2, 12), np.int64)
    st[0, :8] = [500, 1000, 1500, 3000, 43000, 44000, 45000, 46000]
    st[0, 8:] = [100, 1, 1200, 2000]
    st[1, :8] = [600, 1100, 0, 0, 0, 0, 0, 1300]
    c = bench.stamp_columns(st)
    assert c["pages"].tolist() == [100, 0] and c["segments"].tolist() == [1, 0]
    assert c["exit"].tolist() == [45.0, 0.3]
    assert c["lengths_loaded"][0] == 0.2 and np.isnan(c["lengths_loaded"][1])
    assert c["block_ids_loaded"][0] == 1.0
    assert np.isnan(c["range_known"][1])
