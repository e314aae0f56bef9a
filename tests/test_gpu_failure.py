"""Device-side failure detection without faulting the GPU.

Every pipeline wait in the kernels is bounded; a wait that runs out records
XQA_ERR_DEVICE_TIMEOUT and the kernel returns. This follows the fail-closed
stance of the page "[Kernel][SM70] Fold DeepSeek V4 MXFP4 decode exponents"
(its source-audit comment): an error is reported as a status, never as a
kernel that quietly did nothing. The test makes a wait run out on a barrier
nothing arrives at and checks that the status comes back and that the context
still runs a correct decode afterwards.
"""
import time

import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from gpu_helpers import assert_close, oracle_of, run
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    t0 = time.perf_counter()
    status = xqa.xqa_selftest_wait_timeout(20_000_000)  # 20 ms
    elapsed = time.perf_counter() - t0
    assert status == xqa.XQA_ERR_DEVICE_TIMEOUT
    assert 0.02 <= elapsed < 5.0
    # the context is still usable: a decode right after succeeds and is correct
    w = wl.make_custom([33, 500], 8, 2, seed=51)
    assert_close(run(w), oracle_of(w), "after timeout")


def test_selftest_rejects_bad_budget():
    lib = xqa.load_library()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.xqa_selftest_wait_timeout(status.data_ptr(), 0, None) == xqa.XQA_ERR_SHAPE
    assert lib.xqa_selftest_wait_timeout(None, 1000, None) == xqa.XQA_ERR_NULL
