"""xqa_decode_static_workspace: decode for callers that may not allocate device memory.

Some callers cannot call cudaMalloc or hand the library a workspace: a plugin
in a runtime that owns all device memory, a path where an allocation (which
may synchronise the device) is not allowed, an operator interface that passes
only inputs and outputs. For them this entry point takes its scratch from a
fixed array in the library. It runs the same kernels on the same plan as
xqa_decode, so its output must equal xqa_decode's bit for bit, call after call
(the second call with a different shape, so that leftovers of the first cannot
leak into it). The array's status word is not exposed, so rows hit by a bad
block id or a bad context length must still come back as NaN. Kept in a file
that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from gpu_helpers import Dev, assert_close, oracle_of, to_dev, workload
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _static_call(lib, d: Dev, out: torch.Tensor) -> int:
    return lib.xqa_decode_static_workspace(
        d.q.data_ptr(), d.k.data_ptr(), d.v.data_ptr(), d.bt.data_ptr(), d.lens.data_ptr(),
        d.w.k_scale, d.w.v_scale, out.data_ptr(), ctypes.byref(d.shape),
        torch.cuda.current_stream().cuda_stream)


def _bits(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint16)


def test_static_workspace_equals_allocating_entry_point_bitwise():
    lib = xqa.load_library()
    for name in ("b12_boundary", "b4_uniform_ctx1024", "b12_boundary"):
        d = Dev(workload(name))
        d.run()
        ref = _bits(d.out)
        got = torch.full_like(d.q, float("nan"))
        assert _static_call(lib, d, got) == xqa.XQA_OK
        assert np.array_equal(_bits(got), ref), name


@pytest.mark.parametrize("kv_dtype,kv_layout,q_len,merge_mode",
                         [("e4m3", "hnd", 1, 0), ("e5m2", "nhd", 1, 1), ("e5m2", "hnd", 2, 0)])
def test_static_workspace_python_wrapper_formats(kv_dtype, kv_layout, q_len, merge_mode):
    w = wl.make_custom([900, 17, 1, 4100], 16, 2, seed=81, kv_dtype=kv_dtype, q_len=q_len)
    if kv_layout == "nhd":
        w = wl.to_nhd(w)
    d = Dev(w, merge_mode=merge_mode)
    d.run()
    ref = _bits(d.out)
    got = xqa.xqa_decode_static_workspace(d.q, d.k, d.v, d.bt, d.lens, w.k_scale, w.v_scale,
                                          merge_mode=merge_mode, kv_dtype=kv_dtype,
                                          kv_layout=kv_layout)
    assert np.array_equal(_bits(got), ref)


def test_static_workspace_bad_rows_are_nan():
    # a bad block id in sequence 1 and a context length past the table in
    # sequence 3: exactly their rows are NaN, every other row matches
    w = wl.make_custom([40, 3000, 5000, 70, 16], 8, 2, seed=82)
    ref = oracle_of(w)
    d = Dev(w)
    d.bt[1, 9] = w.num_blocks + 2
    d.lens[3] = w.max_blocks_per_seq * 16 + 1
    lib = xqa.load_library()
    for _ in range(2):  # and the array is left ready for the next call
        got = torch.zeros_like(d.q)
        assert _static_call(lib, d, got) == xqa.XQA_OK
        out = got.cpu().numpy()
        for b in range(w.batch):
            nan = np.isnan(out[b].astype(np.float32))
            assert nan.all() if b in (1, 3) else not nan.any(), b
        good = [0, 2, 4]
        assert_close(out[good], ref[good], "rows beside the bad ones")
    d.bt.copy_(to_dev(w.block_tables))
    d.lens.copy_(to_dev(w.context_lens))
    got = torch.zeros_like(d.q)
    assert _static_call(lib, d, got) == xqa.XQA_OK
    assert_close(got.cpu().numpy(), ref, "a good call after the bad ones")


def test_static_workspace_rejects_shapes_beyond_its_size():
    lib = xqa.load_library()
    d = Dev(workload("tiny_b1_ctx256"))
    big = xqa.XqaShape(8192, 32, 4, 128, 16, 16, 16, 0.0, 0, 0)
    assert xqa.xqa_workspace_size(big) > 8 << 20
    rc = lib.xqa_decode_static_workspace(
        d.q.data_ptr(), d.k.data_ptr(), d.v.data_ptr(), d.bt.data_ptr(), d.lens.data_ptr(),
        1.0, 1.0, d.out.data_ptr(), ctypes.byref(big), torch.cuda.current_stream().cuda_stream)
    assert rc == xqa.XQA_ERR_WORKSPACE
