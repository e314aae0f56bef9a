"""Python binding of libxqa: paged E5M2-KV grouped-query decode attention on sm_103a.

Argument marshalling only. Every step of the decode runs in the CUDA kernels of
``libxqa.so``; PyTorch supplies device memory and streams. There is no CPU
fallback: if the library is not built, or a tensor is not on a CUDA device,
these functions raise.

The names mirror the C ABI declared in ``include/xqa.h``:
``xqa_workspace_size``, ``xqa_decode``, ``xqa_plan``, ``xqa_attend_partial``,
``xqa_combine``, ``xqa_decode_device_scales``, ``xqa_dequant_e5m2``,
``xqa_dequant_e4m3``, ``xqa_read_status``, ``xqa_read_plan``, ``xqa_status_string``,
``xqa_decode_static_workspace``, ``xqa_kernels_per_call``.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libxqa.so")

XQA_OK = 0
XQA_ERR_NULL = 1
XQA_ERR_SHAPE = 2
XQA_ERR_ALIGN = 3
XQA_ERR_WORKSPACE = 4
XQA_ERR_LAUNCH = 5
XQA_ERR_DEVICE = 6
XQA_ERR_BAD_BLOCK_ID = 16
XQA_ERR_CTX_TOO_LONG = 17
XQA_ERR_DEVICE_TIMEOUT = 18
XQA_ERR_DRAIN_TIMEOUT = 19

#: C symbols the library exports (kept in step with include/xqa.h).
EXPORTED = (
    "xqa_workspace_size",
    "xqa_decode",
    "xqa_plan",
    "xqa_attend_partial",
    "xqa_combine",
    "xqa_dequant_e5m2",
    "xqa_read_status",
    "xqa_read_plan",
    "xqa_status_string",
    "xqa_decode_static_workspace",
    "xqa_decode_device_scales",
    "xqa_dequant_e4m3",
    "xqa_selftest_wait_timeout",
    "xqa_kernels_per_call",
)

KV_DTYPES = {"e5m2": 0, "e4m3": 1}
KV_LAYOUTS = {"hnd": 0, "nhd": 1}


class XqaShape(ctypes.Structure):
    """Mirror of ``xqa_shape_t``."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
        ("max_ctas", ctypes.c_int32),
        ("min_pages_per_cta", ctypes.c_int32),
        ("merge_mode", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("kv_layout", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
    ]


class XqaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {xqa_status_string(code)} (status {code})")


_lib = None

_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_SHAPE = ctypes.POINTER(XqaShape)
_SIGS = {
    "xqa_workspace_size": [_SHAPE, ctypes.POINTER(_SZ)],
    "xqa_decode": [_P, _P, _P, _P, _P, _F, _F, _P, _SHAPE, _P, _SZ, _P],
    "xqa_plan": [_P, _SHAPE, _P, _SZ, _P],
    "xqa_attend_partial": [_P, _P, _P, _P, _P, _F, _F, _P, _SHAPE, _P, _SZ, _P],
    "xqa_combine": [_P, _F, _P, _SHAPE, _P, _SZ, _P],
    "xqa_dequant_e5m2": [_P, _SZ, _F, _P, _P, _P],
    "xqa_read_status": [_P, ctypes.POINTER(ctypes.c_int32), _P],
    "xqa_read_plan": [_P, _SHAPE, _P, _P, _P, _P, _P],
    "xqa_status_string": [ctypes.c_int],
    "xqa_decode_static_workspace": [_P, _P, _P, _P, _P, _F, _F, _P, _SHAPE, _P],
    "xqa_decode_device_scales": [_P, _P, _P, _P, _P, _P, _P, _P, _SHAPE, _P, _SZ, _P],
    "xqa_dequant_e4m3": [_P, _SZ, _F, _P, _P, _P],
    "xqa_selftest_wait_timeout": [_P, ctypes.c_uint64, _P],
    "xqa_kernels_per_call": [_SHAPE, ctypes.POINTER(ctypes.c_int32)],
}


def load_library() -> ctypes.CDLL:
    """Load libxqa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()' or "
                "python paged_fp8_kv_gqa_gb300/build.py)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, argtypes in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = ctypes.c_char_p if name == "xqa_status_string" else ctypes.c_int
        _lib = lib
    return _lib


def xqa_status_string(code: int) -> str:
    return load_library().xqa_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != XQA_OK:
        raise XqaError(code, where)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _cuda(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def make_shape(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
               sm_scale: float = 0.0, max_ctas: int = 0, min_pages_per_cta: int = 0,
               merge_mode: int = 0, kv_dtype: str = "e5m2", kv_layout: str = "hnd") -> XqaShape:
    """Shape descriptor from q [B, Hq, D] (or [B, T, Hq, D] for T new tokens per
    sequence), block_tables [B, MBS] and k_cache [NB, Hkv, BS, D] (kv_layout
    "hnd") or [NB, BS, Hkv, D] ("nhd")."""
    if q.dim() == 4:
        b, t_new, hq, d = q.shape
    else:
        (b, hq, d), t_new = q.shape, 1
    if kv_layout == "hnd":
        nb, hkv, bs, d2 = k_cache.shape
    else:
        nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or block_tables.shape[0] != b:
        raise ValueError("inconsistent q / k_cache / block_tables shapes")
    return XqaShape(int(b), int(hq), int(hkv), int(d), int(bs), int(block_tables.shape[1]),
                    int(nb), float(sm_scale), int(max_ctas), int(min_pages_per_cta),
                    int(merge_mode), KV_DTYPES[kv_dtype], KV_LAYOUTS[kv_layout], int(t_new))


def xqa_workspace_size(shape: XqaShape) -> int:
    n = _SZ(0)
    _check(load_library().xqa_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
           "xqa_workspace_size")
    return int(n.value)


def xqa_kernels_per_call(shape: XqaShape) -> int:
    """Kernels one xqa_decode call enqueues for this shape."""
    n = ctypes.c_int32(0)
    _check(load_library().xqa_kernels_per_call(ctypes.byref(shape), ctypes.byref(n)),
           "xqa_kernels_per_call")
    return int(n.value)


def alloc_workspace(shape: XqaShape, device=None) -> torch.Tensor:
    """A zero-filled uint8 device buffer of xqa_workspace_size bytes (256-byte
    aligned by torch). The library needs it zeroed once, before its first use;
    every call leaves it ready for the next."""
    return torch.zeros(xqa_workspace_size(shape), dtype=torch.uint8, device=device or "cuda")


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, workspace, shape):
    return (
        _cuda(q, torch.float16, "q"),
        _cuda(k_cache, torch.uint8, "k_cache"),
        _cuda(v_cache, torch.uint8, "v_cache"),
        _cuda(block_tables, torch.int32, "block_tables"),
        _cuda(context_lens, torch.int32, "context_lens"),
        _cuda(out, torch.float16, "out"),
        _cuda(workspace, torch.uint8, "workspace"),
    )


def xqa_decode(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale,
               out=None, workspace=None, shape: XqaShape | None = None, stream=None,
               sm_scale: float = 0.0, max_ctas: int = 0, min_pages_per_cta: int = 0,
               kv_dtype: str = "e5m2", kv_layout: str = "hnd"):
    """One decode step. Tensors: q fp16 [B,Hq,D]; k/v_cache uint8 FP8 codes
    [NB,Hkv,16,D] (or [NB,16,Hkv,D] for kv_layout "nhd"); block_tables int32
    [B,MBS]; context_lens int32 [B]. k_scale / v_scale are floats, or float32
    CUDA tensors of one element (read on the device: xqa_decode_device_scales).
    Returns ``out`` fp16 [B,Hq,D]."""
    if shape is None:
        shape = make_shape(q, k_cache, block_tables, sm_scale, max_ctas, min_pages_per_cta,
                           kv_dtype=kv_dtype, kv_layout=kv_layout)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(shape, q.device)
    a = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, workspace, shape)
    lib = load_library()
    if isinstance(k_scale, torch.Tensor) or isinstance(v_scale, torch.Tensor):
        ks = _cuda(k_scale, torch.float32, "k_scale")
        vs = _cuda(v_scale, torch.float32, "v_scale")
        _check(lib.xqa_decode_device_scales(a[0], a[1], a[2], a[3], a[4], ks, vs, a[5],
                                            ctypes.byref(shape), a[6], workspace.numel(),
                                            _stream_handle(stream)), "xqa_decode_device_scales")
        return out
    _check(lib.xqa_decode(a[0], a[1], a[2], a[3], a[4], float(k_scale), float(v_scale), a[5],
                          ctypes.byref(shape), a[6], workspace.numel(), _stream_handle(stream)),
           "xqa_decode")
    return out


def xqa_plan(context_lens, workspace, shape: XqaShape, stream=None) -> None:
    _check(load_library().xqa_plan(_cuda(context_lens, torch.int32, "context_lens"),
                                   ctypes.byref(shape), _cuda(workspace, torch.uint8, "workspace"),
                                   workspace.numel(), _stream_handle(stream)), "xqa_plan")


def xqa_attend_partial(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale, out,
                       workspace, shape: XqaShape, stream=None) -> None:
    a = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, workspace, shape)
    _check(load_library().xqa_attend_partial(a[0], a[1], a[2], a[3], a[4], float(k_scale),
                                             float(v_scale), a[5], ctypes.byref(shape), a[6],
                                             workspace.numel(), _stream_handle(stream)),
           "xqa_attend_partial")


def xqa_combine(context_lens, v_scale, out, workspace, shape: XqaShape, stream=None) -> None:
    _check(load_library().xqa_combine(_cuda(context_lens, torch.int32, "context_lens"),
                                      float(v_scale), _cuda(out, torch.float16, "out"),
                                      ctypes.byref(shape),
                                      _cuda(workspace, torch.uint8, "workspace"),
                                      workspace.numel(), _stream_handle(stream)), "xqa_combine")


def _dequant(fn_name, codes, scale, with_f32, stream):
    n = codes.numel()
    out16 = torch.empty(n, dtype=torch.int16, device=codes.device)
    out32 = torch.empty(n, dtype=torch.float32, device=codes.device) if with_f32 else None
    _check(getattr(load_library(), fn_name)(
        _cuda(codes, torch.uint8, "codes"), n, float(scale), out16.data_ptr(),
        out32.data_ptr() if out32 is not None else None, _stream_handle(stream)), fn_name)
    return out16, out32


def xqa_dequant_e5m2(codes: torch.Tensor, scale: float = 1.0, with_f32: bool = True, stream=None):
    """Exact dequantisation: returns (fp16 bit patterns as int16 tensor, fp32 scaled or None)."""
    return _dequant("xqa_dequant_e5m2", codes, scale, with_f32, stream)


def xqa_dequant_e4m3(codes: torch.Tensor, scale: float = 1.0, with_f32: bool = True, stream=None):
    """Exact E4M3 dequantisation: (fp16 bit patterns as int16 tensor, fp32 scaled or None)."""
    return _dequant("xqa_dequant_e4m3", codes, scale, with_f32, stream)


def xqa_read_status(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(-1)
    _check(load_library().xqa_read_status(_cuda(workspace, torch.uint8, "workspace"),
                                          ctypes.byref(v), _stream_handle(stream)),
           "xqa_read_status")
    return int(v.value)


def xqa_read_plan(workspace: torch.Tensor, shape: XqaShape, stream=None) -> dict:
    import numpy as np

    nseg = shape.batch * shape.num_kv_heads
    header = np.zeros(4, np.int32)
    seg_start = np.zeros(nseg + 1, np.int32)
    seg_bad = np.zeros(nseg, np.int32)
    seg_cost = np.zeros(nseg, np.int32)
    _check(load_library().xqa_read_plan(_cuda(workspace, torch.uint8, "workspace"),
                                        ctypes.byref(shape), header.ctypes.data,
                                        seg_start.ctypes.data, seg_bad.ctypes.data,
                                        seg_cost.ctypes.data, _stream_handle(stream)),
           "xqa_read_plan")
    return {"ctas_launched": int(header[0]), "num_ctas": int(header[1]), "total_pages": int(header[2]),
            "num_segments": int(header[3]), "seg_start": seg_start, "seg_bad": seg_bad,
            "seg_cc": seg_cost}


def xqa_decode_static_workspace(q, k_cache, v_cache, block_tables, context_lens, k_scale: float,
                                v_scale: float, out=None, shape: XqaShape | None = None,
                                stream=None, sm_scale: float = 0.0, max_ctas: int = 0,
                                min_pages_per_cta: int = 0, merge_mode: int = 0,
                                kv_dtype: str = "e5m2", kv_layout: str = "hnd"):
    """xqa_decode without a workspace argument, for callers that may not allocate
    device memory: the scratch is the library's fixed per-device array (see
    include/xqa.h). q may be [B, Hq, D] or [B, T, Hq, D] (T new tokens per
    sequence). Calls that may overlap on one device must be ordered."""
    if shape is None:
        shape = make_shape(q, k_cache, block_tables, sm_scale, max_ctas, min_pages_per_cta,
                           merge_mode, kv_dtype=kv_dtype, kv_layout=kv_layout)
    if out is None:
        out = torch.empty_like(q)
    ptrs = (
        _cuda(q, torch.float16, "q"),
        _cuda(k_cache, torch.uint8, "k_cache"),
        _cuda(v_cache, torch.uint8, "v_cache"),
        _cuda(block_tables, torch.int32, "block_tables"),
        _cuda(context_lens, torch.int32, "context_lens"),
        _cuda(out, torch.float16, "out"),
    )
    _check(load_library().xqa_decode_static_workspace(
        ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[4], float(k_scale), float(v_scale), ptrs[5],
        ctypes.byref(shape), _stream_handle(stream)), "xqa_decode_static_workspace")
    return out


def xqa_selftest_wait_timeout(budget_ns: int, stream=None) -> int:
    """Run the bounded-wait self-check (a wait nothing completes); returns the
    status the kernel wrote (XQA_ERR_DEVICE_TIMEOUT when the wait gave up)."""
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check(load_library().xqa_selftest_wait_timeout(status.data_ptr(), int(budget_ns),
                                                    _stream_handle(stream)),
           "xqa_selftest_wait_timeout")
    torch.cuda.synchronize()
    return int(status.item())
