// combine.cu — log-sum-exp merge of the split-KV partial results.
//
// One CTA per (sequence, kv head) segment; a thread handles one column (new
// token x head) and 4 dims at a time. Segments processed whole by one
// partial CTA, and empty segments, were already written by the partial
// kernel. For a segment split over CTAs i_lo..i_hi this kernel reads the
// segment's merge ticket (how many of its pieces met a bad block id), clears
// it for the next call, and writes NaN rows if any did; otherwise it merges
// the pieces (slot i + s):
//   M = max_i m_i,  w_i = 2^(m_i - M),  L = sum_i w_i l_i,
//   out = fp16(sum_i w_i o_i * (v_scale / L))    (round to nearest even).
// This is the "merge" phase of the planner -> forward -> merge split-KV
// structure on the page "[Kernel][WIP] Follow up FlashNext batch HC fusion and
// QSA route audit" (section "Test Result").
#include <math.h>

#include "xqa_device.cuh"
#include "xqa_launch.h"

namespace xqa {

__device__ __forceinline__ void store_half4(__half* dst, float a, float b, float c, float d) {
  uint2 v;
  v.x = pack_half2(a, b);
  v.y = pack_half2(c, d);
  *reinterpret_cast<uint2*>(dst) = v;
}

// Row of column col (new token i = col / G, head h = col % G) of segment s.
__device__ __forceinline__ size_t combine_row(const CombineParams& p, int s, int col) {
  const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
  const int i = col / p.group, h = col - i * p.group;
  return ((size_t)b * p.q_len + i) * p.num_q_heads + (size_t)kvh * p.group + h;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
  const int s = blockIdx.x;
  const int dq = (threadIdx.x & 31) * 4;
  const int ncols = p.group * p.q_len;
  const int n = p.header[1];
  const long long total = p.header[2];
  const int sb = p.seg_start[s], se = p.seg_start[s + 1];
  if (sb == se) return;  // empty: its row was written by the partial kernel
  // the CTAs holding the first and the last page, on the plan's cost line
  const long long line = total + p.seg_cc[p.header[3] - 1];
  const int ilo = cta_of_vpos((long long)sb + p.seg_cc[s], line, n);
  const int ihi = cta_of_vpos((long long)se - 1 + p.seg_cc[s], line, n);
  if (ilo == ihi) return;  // written whole by its partial CTA
  const bool bad = p.tickets[ilo] >= kTicketPoison;
  __syncthreads();  // every thread has read the ticket before it is cleared
  if (threadIdx.x == 0) p.tickets[ilo] = 0;
  const float v_scale = p.v_scale_ptr ? __ldg(p.v_scale_ptr) : p.v_scale;
  for (int col = threadIdx.x >> 5; col < ncols; col += kCombineThreads / 32) {
    __half* o = p.out + combine_row(p, s, col) * kHeadDim + dq;
    if (bad) {
      const float v = __int_as_float(0x7fc00000);
      store_half4(o, v, v, v, v);
      continue;
    }
    // the maxima 16 pieces at a time, then the weighted sums 8 at a time (every
    // load of a batch issued before any is used; the sums in piece order)
    float M = -INFINITY;
    for (int base = ilo; base <= ihi; base += 16) {
      float mb[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (base + k <= ihi) mb[k] = p.partials[(size_t)(base + k + s) * kSlotFloats + kSlotM + col];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (base + k <= ihi) M = fmaxf(M, mb[k]);
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = ilo; base <= ihi; base += 8) {
      float mb[8], lb[8];
      float4 vb[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (base + k <= ihi) {
          const float* slot = p.partials + (size_t)(base + k + s) * kSlotFloats;
          mb[k] = slot[kSlotM + col];
          lb[k] = slot[kSlotL + col];
          vb[k] = *reinterpret_cast<const float4*>(slot + col * kHeadDim + dq);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (base + k <= ihi) {
          const float w = (mb[k] == -INFINITY) ? 0.f : ex2(mb[k] - M);
          L += w * lb[k];
          acc.x += w * vb[k].x;
          acc.y += w * vb[k].y;
          acc.z += w * vb[k].z;
          acc.w += w * vb[k].w;
        }
      }
    }
    const float r = (L > 0.f) ? v_scale / L : 0.f;  // a new token with no visible token: 0
    store_half4(o, acc.x * r, acc.y * r, acc.z * r, acc.w * r);
  }
}

cudaError_t launch_combine(const CombineParams& p, int num_segments, cudaStream_t stream) {
  if (num_segments <= 0) return cudaSuccess;
  combine_kernel<<<num_segments, kCombineThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace xqa
