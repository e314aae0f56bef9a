// static_workspace.cu — a decode entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc: a plugin inside a host runtime that owns
// every byte of device memory through its own pool and forbids side
// allocations, a latency-critical path where an allocation (which may
// synchronise the device) is not allowed, or an operator interface that hands
// the kernel only its inputs and outputs and offers no workspace hook. For them
// xqa_decode_static_workspace runs the same three kernels as xqa_decode, with
// the split-KV scratch taken from a fixed array that lives in the library's
// device image instead of a caller-provided buffer.
//
// The array is XQA_STATIC_WORKSPACE_BYTES per device, held for as long as the
// library stays loaded on that device. Its device address is looked up with
// cudaGetSymbolAddress the first time the entry point runs on a device (with
// that device current) and cached; host code must never hand the symbol itself
// to a kernel, since in host code it names a host-side shadow, not device
// memory.
#include <cuda_runtime.h>

#include <atomic>

#include "xqa.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = XQA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; the planner kernel of each call rewrites
// every word the later kernels of that call read, so nothing in it has to
// start at zero.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::atomic<void*> g_static_workspace_ptr[kMaxDevices];

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
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return XQA_ERR_DEVICE;
  void* ws = g_static_workspace_ptr[dev].load(std::memory_order_acquire);
  if (ws == nullptr) {
    if (cudaGetSymbolAddress(&ws, g_static_workspace) != cudaSuccess || ws == nullptr)
      return XQA_ERR_DEVICE;
    g_static_workspace_ptr[dev].store(ws, std::memory_order_release);
  }
  return xqa_decode(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale, out, shape,
                    ws, kStaticWorkspaceBytes, stream);
}
