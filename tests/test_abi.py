"""C ABI checks that need no GPU: the library builds, loads, exports every
function include/xqa.h declares, and rejects bad host arguments before touching
a device."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_fp8_kv_gqa_gb300 as xqa
from paged_fp8_kv_gqa_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xqa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return xqa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(xqa_[a-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(xqa.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", xqa.LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\bT\s+(xqa_\w+)", nm.stdout))
        assert set(declared_functions()) <= exported


def test_status_strings(lib):
    for code in (0, 1, 2, 3, 4, 5, 6, 16, 17, 18, 19):
        s = xqa.xqa_status_string(code)
        assert s and s != "unknown status"
    assert xqa.xqa_status_string(12345) == "unknown status"


def test_host_validation_without_device(lib):
    shape = xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0)
    n = ctypes.c_size_t(0)
    assert lib.xqa_workspace_size(ctypes.byref(shape), ctypes.byref(n)) == xqa.XQA_OK
    nseg = 64
    # header, merge tickets (two words per CTA), status words and first-page
    # hints (16 per CTA) (fixed size: 1024 CTAs at most), then segment starts,
    # bad-context flags and the cost-line prefix
    head = 64 + 8 * 1024 + 4 * 1024 + 4 * 16 * 1024 + 4 * (nseg + 1) + 4 * nseg + 4 * nseg
    head = (head + 255) // 256 * 256
    assert n.value == head + (152 + nseg) * (16 * 128 + 32) * 4
    for bad in (
        xqa.XqaShape(16, 32, 4, 64, 16, 1200, 22240, 0.0, 152, 0),   # head_dim
        xqa.XqaShape(16, 32, 4, 128, 32, 1200, 22240, 0.0, 152, 0),  # block size
        xqa.XqaShape(16, 30, 4, 128, 16, 1200, 22240, 0.0, 152, 0),  # Hq % Hkv
        xqa.XqaShape(16, 128, 4, 128, 16, 1200, 22240, 0.0, 152, 0),  # G = 32
        xqa.XqaShape(0, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0),   # batch
        xqa.XqaShape(16, 32, 4, 128, 16, 1200, 2**28, 0.0, 152, 0),  # pool too large for int32 rows
        xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0, 2),  # merge mode
        xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0, 0, 2),  # kv dtype
        xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0, 0, 0, 2),  # kv layout
        xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0, 0, 0, 0, 3),  # G * T > 16
    ):
        assert lib.xqa_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == xqa.XQA_ERR_SHAPE
    g16 = xqa.XqaShape(16, 64, 4, 128, 16, 1200, 22240, 0.0, 152, 0)  # G = 16, one token
    assert lib.xqa_workspace_size(ctypes.byref(g16), ctypes.byref(n)) == xqa.XQA_OK
    g16t2 = xqa.XqaShape(16, 64, 4, 128, 16, 1200, 22240, 0.0, 152, 0, 0, 0, 0, 2)
    assert lib.xqa_workspace_size(ctypes.byref(g16t2), ctypes.byref(n)) == xqa.XQA_ERR_SHAPE
    assert lib.xqa_workspace_size(None, ctypes.byref(n)) == xqa.XQA_ERR_NULL
    assert lib.xqa_decode(None, None, None, None, None, 1.0, 1.0, None, ctypes.byref(shape), None,
                          0, None) == xqa.XQA_ERR_NULL
    assert lib.xqa_dequant_e5m2(None, 0, 1.0, None, None, None) == xqa.XQA_OK
    assert lib.xqa_dequant_e5m2(None, 5, 1.0, None, None, None) == xqa.XQA_ERR_NULL


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(xqa, "_lib", None)
    monkeypatch.setattr(xqa, "LIB_PATH", "/nonexistent/libxqa.so")
    with pytest.raises(RuntimeError, match="missing"):
        xqa.load_library()


def test_argument_checks_come_before_any_device_call(lib):
    # Addresses below are never dereferenced: each call is rejected by a host
    # check that runs before the first CUDA call (max_ctas is explicit, so no
    # SM-count query either). Pointer order: q, K, V, tables, lengths, out.
    shape = xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, 152, 0)
    n = ctypes.c_size_t(0)
    assert lib.xqa_workspace_size(ctypes.byref(shape), ctypes.byref(n)) == xqa.XQA_OK
    q, k, v, bt, lens, out, ws = (0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000,
                                  0x100000)
    sh = ctypes.byref(shape)

    def decode(q, k, v, bt, lens, out, ws=ws, nbytes=n.value):
        return lib.xqa_decode(q, k, v, bt, lens, 1.0, 1.0, out, sh, ws, nbytes, None)

    assert decode(q, k, v, bt, lens, out, ws=ws + 128) == xqa.XQA_ERR_ALIGN  # 256-B workspace
    assert decode(q, k, v, bt, lens, out, ws=0) == xqa.XQA_ERR_NULL
    assert decode(q, k, v, bt, lens, out, nbytes=n.value - 1) == xqa.XQA_ERR_WORKSPACE
    for i in (0, 1, 2, 5):  # q, K, V and out must be 16-byte aligned
        ptrs = [q, k, v, bt, lens, out]
        ptrs[i] += 8
        assert decode(*ptrs) == xqa.XQA_ERR_ALIGN, i
    assert lib.xqa_attend_partial(q + 2, k, v, bt, lens, 1.0, 1.0, out, sh, ws, n.value,
                                  None) == xqa.XQA_ERR_ALIGN
    assert lib.xqa_plan(None, sh, ws, n.value, None) == xqa.XQA_ERR_NULL
    assert lib.xqa_plan(lens, sh, ws + 16, n.value, None) == xqa.XQA_ERR_ALIGN
    assert lib.xqa_plan(lens, sh, ws, 64, None) == xqa.XQA_ERR_WORKSPACE
    assert lib.xqa_combine(lens, 1.0, out + 2, sh, ws, n.value, None) == xqa.XQA_ERR_ALIGN
    negative = xqa.XqaShape(16, 32, 4, 128, 16, 1200, 22240, 0.0, -1, 0)
    assert lib.xqa_decode(q, k, v, bt, lens, 1.0, 1.0, out, ctypes.byref(negative), ws, n.value,
                          None) == xqa.XQA_ERR_SHAPE
    # the static-workspace entry point rejects a shape its array cannot hold
    m = re.search(r"#define XQA_STATIC_WORKSPACE_BYTES \(\(size_t\)(\d+) << (\d+)\)",
                  open(HEADER).read())
    static_bytes = int(m.group(1)) << int(m.group(2))
    big = xqa.XqaShape(8192, 32, 4, 128, 16, 16, 16, 0.0, 152, 0)
    assert xqa.xqa_workspace_size(big) > static_bytes
    assert lib.xqa_decode_static_workspace(q, k, v, bt, lens, 1.0, 1.0, out, ctypes.byref(big),
                                           None) == xqa.XQA_ERR_WORKSPACE


def test_kernels_per_call(lib):
    # the partial kernel derives the plan itself while the segment table fits
    # in shared memory (B*Hkv + 1 <= 2048 entries); larger batches add the
    # planner kernel, merge_mode 1 the combine kernel
    def count(batch, merge_mode=0):
        sh = xqa.XqaShape(batch, 32, 4, 128, 16, 64, 4096, 0.0, 152, 0, merge_mode)
        k = ctypes.c_int32(0)
        assert lib.xqa_kernels_per_call(ctypes.byref(sh), ctypes.byref(k)) == xqa.XQA_OK
        return k.value
    assert count(16) == 1
    assert count(511) == 1          # 2044 segments + 1 entries fit
    assert count(512) == 2          # 2048 segments + 1 do not
    assert count(16, merge_mode=1) == 2
    assert count(512, merge_mode=1) == 3
    assert lib.xqa_kernels_per_call(None, ctypes.byref(ctypes.c_int32())) == xqa.XQA_ERR_NULL


def test_max_ctas_is_clamped_to_the_ticket_region():
    a = xqa.xqa_workspace_size(xqa.XqaShape(16, 32, 4, 128, 16, 64, 4096, 0.0, 1024, 0))
    b = xqa.xqa_workspace_size(xqa.XqaShape(16, 32, 4, 128, 16, 64, 4096, 0.0, 5000, 0))
    assert a == b
