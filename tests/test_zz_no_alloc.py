"""xqa_decode_static_workspace: decode for callers that may not allocate device memory.

Runs through the C ABI with the same inputs and outputs as xqa_decode but no
workspace argument (the scratch is the library's fixed per-device array), and
must give the same result as the allocating entry point on two calls in a row,
the second with a different shape so that leftovers of the first cannot leak
into it. Kept in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from gpu_helpers import ATOL, RTOL, Dev, workload

pytestmark = pytest.mark.gpu


def _static_call(lib, d: Dev, out: torch.Tensor) -> int:
    return lib.xqa_decode_static_workspace(
        d.q.data_ptr(), d.k.data_ptr(), d.v.data_ptr(), d.bt.data_ptr(), d.lens.data_ptr(),
        d.w.k_scale, d.w.v_scale, out.data_ptr(), ctypes.byref(d.shape),
        torch.cuda.current_stream().cuda_stream)


def test_static_workspace_matches_allocating_entry_point_twice():
    lib = xqa.load_library()
    for name in ("b12_boundary", "b4_uniform_ctx1024"):
        d = Dev(workload(name))
        d.run()
        ref = d.result().astype(np.float64)
        got_t = torch.full_like(d.q, float("nan"))
        assert _static_call(lib, d, got_t) == xqa.XQA_OK
        torch.cuda.synchronize()
        got = got_t.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), name
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)), name


def test_static_workspace_rejects_shapes_beyond_its_size():
    lib = xqa.load_library()
    d = Dev(workload("tiny_b1_ctx256"))
    big = xqa.XqaShape(8192, 32, 4, 128, 16, 16, 16, 0.0, 0, 0)
    assert xqa.xqa_workspace_size(big) > 8 << 20
    rc = lib.xqa_decode_static_workspace(
        d.q.data_ptr(), d.k.data_ptr(), d.v.data_ptr(), d.bt.data_ptr(), d.lens.data_ptr(),
        1.0, 1.0, d.out.data_ptr(), ctypes.byref(big), torch.cuda.current_stream().cuda_stream)
    assert rc == xqa.XQA_ERR_WORKSPACE
