// static_workspace.cu — a decode entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc: a plugin inside a host runtime that owns
// every byte of device memory through its own pool and forbids side
// allocations, a latency-critical path where an allocation (which may
// synchronise the device) is not allowed, or an operator interface that hands
// the kernel only its inputs and outputs and offers no workspace hook. For them
// xqa_decode_static_workspace runs the same kernels as xqa_decode, with
// the split-KV scratch taken from a fixed array that lives in the library's
// device image instead of a caller-provided buffer.
//
// The array is XQA_STATIC_WORKSPACE_BYTES per device, held for as long as the
// library stays loaded on that device. It starts zero-filled, as the decode
// kernels need a workspace to start (each call leaves it ready for the next).
// Its device address is looked up with cudaGetSymbolAddress on every call,
// with the caller's device current: a host-side lookup that allocates
// nothing, and stays right if the device's context is reset and the module
// reloaded at another address. Host code must never hand the symbol itself to
// a kernel, since in host code it names a host-side shadow, not device memory.
#include <cuda_runtime.h>

#include "xqa.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = XQA_STATIC_WORKSPACE_BYTES;

// Shared by every call on a device (zero-initialised when the module loads).
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

}  // namespace

extern "C" xqa_status_t xqa_decode_static_workspace(
    const void* q, const uint8_t* k_cache, const uint8_t* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, float k_scale, float v_scale, void* out,
    const xqa_shape_t* shape, void* stream) {
  if (!shape) return XQA_ERR_NULL;
  size_t need = 0;
  xqa_status_t st = xqa_workspace_size(shape, &need);
  if (st != XQA_OK) return st;
  if (need > kStaticWorkspaceBytes) return XQA_ERR_WORKSPACE;  // shape too large for the array
  void* ws = nullptr;
  if (cudaGetSymbolAddress(&ws, g_static_workspace) != cudaSuccess || ws == nullptr)
    return XQA_ERR_DEVICE;
  return xqa_decode(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale, out, shape,
                    ws, kStaticWorkspaceBytes, stream);
}
