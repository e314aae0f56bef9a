// dequant.cu — the exact E5M2 -> fp16 conversion on its own, for testing.
//
// Each thread converts one 8-byte group with the same byte-permutation helpers
// the attention kernel uses: even groups take the "adjacent codes of one word"
// route used for K, odd groups the "same byte of two words" route used for V,
// so a test over all 256 codes at both parities checks both routes bit for bit.
// This is the "E5M2 conversion" phase named on the page "[Kernel][SM70]
// Pipeline batched E5M2 XQA decode" (section "Pending work and gates"), and
// its E4M3 counterpart.
#include "xqa_device.cuh"
#include "xqa_launch.h"

namespace xqa {

template <int kFmt>
__global__ void dequant_kernel(const uint8_t* __restrict__ in, size_t n, float scale,
                               uint16_t* __restrict__ out16, float* __restrict__ out32) {
  const size_t ngroups = (n + 7) / 8;
  for (size_t grp = (size_t)blockIdx.x * blockDim.x + threadIdx.x; grp < ngroups;
       grp += (size_t)gridDim.x * blockDim.x) {
    const size_t base = grp * 8;
    uint32_t x = 0, y = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (base + k < n) x |= (uint32_t)in[base + k] << (8 * k);
      if (base + 4 + k < n) y |= (uint32_t)in[base + 4 + k] << (8 * k);
    }
    uint16_t h[8];
    if ((grp & 1) == 0) {
      const uint32_t r[4] = {KvConv<kFmt>::k_lo(x), KvConv<kFmt>::k_hi(x), KvConv<kFmt>::k_lo(y),
                             KvConv<kFmt>::k_hi(y)};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[2 * k] = (uint16_t)(r[k] & 0xffffu);
        h[2 * k + 1] = (uint16_t)(r[k] >> 16);
      }
    } else {
      uint32_t r[4];
      KvConv<kFmt>::v_pairs(x, y, r);
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // r[k] = {x_k, y_k}
        h[k] = (uint16_t)(r[k] & 0xffffu);
        h[4 + k] = (uint16_t)(r[k] >> 16);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (base + k < n) {
        out16[base + k] = h[k];
        if (out32) out32[base + k] = __half2float(__ushort_as_half(h[k])) * scale;
      }
    }
  }
}

// Self-check of the bounded pipeline wait: every thread waits on an mbarrier
// that nothing arrives at, with the given budget; the wait must give up and
// the kernel must record XQA_ERR_DEVICE_TIMEOUT and return. No copy is in
// flight, so leaving the barrier incomplete is harmless.
__global__ void wait_timeout_kernel(int32_t* status, unsigned long long budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int never;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    never = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool done = mbar_wait_bounded(&bar, 0, &never, budget_ns);
  if (!done && threadIdx.x == 0) atomicExch(status, XQA_ERR_DEVICE_TIMEOUT);
  if (done && threadIdx.x == 0) atomicExch(status, XQA_OK);
}

cudaError_t launch_wait_timeout(int32_t* status, unsigned long long budget_ns,
                                cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(status, budget_ns);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int kv_dtype, const uint8_t* in, size_t n, float scale,
                           uint16_t* out16, float* out32, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const size_t ngroups = (n + 7) / 8;
  size_t blocks = (ngroups + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (kv_dtype == XQA_KV_E4M3)
    dequant_kernel<XQA_KV_E4M3><<<(unsigned)blocks, 256, 0, stream>>>(in, n, scale, out16, out32);
  else
    dequant_kernel<XQA_KV_E5M2><<<(unsigned)blocks, 256, 0, stream>>>(in, n, scale, out16, out32);
  return cudaGetLastError();
}

}  // namespace xqa
