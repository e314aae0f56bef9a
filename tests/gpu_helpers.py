"""Helpers shared by the GPU parity tests (upload, run, compare)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from oracle import attention
from paged_fp8_kv_gqa_gb300 import workloads as wl

ATOL = 2e-3
RTOL = 1e-2


@functools.lru_cache(maxsize=None)
def workload(name: str) -> wl.Workload:
    return wl.make_workload(name)


@functools.lru_cache(maxsize=None)
def oracle_out(name: str) -> np.ndarray:
    w = workload(name)
    return attention.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                            w.context_lens, w.k_scale, w.v_scale)


def oracle_of(w: wl.Workload, sm_scale=None) -> np.ndarray:
    fn = attention.paged_decode_attention_multi if w.q.ndim == 4 else attention.paged_decode_attention
    return fn(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.k_scale, w.v_scale,
              sm_scale, kv_dtype=w.kv_dtype, kv_layout=w.kv_layout)


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Dev:
    """A workload's arrays on the GPU plus an output and a workspace."""

    def __init__(self, w: wl.Workload, max_ctas: int = 0, min_pages: int = 0, sm_scale=0.0,
                 merge_mode: int = 0):
        self.w = w
        self.q = to_dev(w.q)
        self.k = to_dev(w.k_cache)
        self.v = to_dev(w.v_cache)
        self.bt = to_dev(w.block_tables)
        self.lens = to_dev(w.context_lens)
        self.shape = xqa.make_shape(self.q, self.k, self.bt, sm_scale, max_ctas, min_pages,
                                    merge_mode, kv_dtype=w.kv_dtype, kv_layout=w.kv_layout)
        self.out = torch.full_like(self.q, float("nan"))
        self.ws = xqa.alloc_workspace(self.shape)

    def run(self, stream=None) -> torch.Tensor:
        xqa.xqa_decode(self.q, self.k, self.v, self.bt, self.lens, self.w.k_scale, self.w.v_scale,
                       out=self.out, workspace=self.ws, shape=self.shape, stream=stream)
        return self.out

    def result(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.out.cpu().numpy()

    def status(self) -> int:
        return xqa.xqa_read_status(self.ws)


def run(w: wl.Workload, **kw) -> np.ndarray:
    d = Dev(w, **kw)
    d.run()
    out = d.result()
    st = d.status()
    assert st == xqa.XQA_OK, xqa.xqa_status_string(st)
    return out


def assert_close(got16: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    """Elementwise |gpu - ref| <= ATOL + RTOL*|ref|; returns max abs / rel errors."""
    got = got16.astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    big = np.abs(ref) > ATOL
    stats = {
        "max_abs": float(err.max()),
        "max_rel": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
    }
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements out of tolerance; first {tuple(idx)} "
            f"gpu={got[tuple(idx)]!r} ref={ref[tuple(idx)]!r}; {stats}")
    return stats
