// xqa_launch.h — host-side launch functions of the libxqa kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace xqa {

struct PartialParams {
  const __half* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  __half* out;
  int32_t* header;     // workspace header (CTAs launched, CTAs with work, pages, segments)
  int32_t* seg_start;  // [nseg + 1]; written here when the plan is derived in the kernel
  int32_t* seg_bad;    // [nseg] bad context-length flags (plan output)
  int32_t* seg_cc;     // [nseg] cost-line prefix (see seg_cost)
  int32_t* tickets;    // [kMaxCtas] merge tickets of split segments, zero between calls
  int32_t* status;     // [kMaxCtas] each CTA's status in this call
  float* partials;     // [(n_max + nseg) * kSlotFloats]
  int32_t* hints;      // [kMaxCtas * kHintPages] first pages of each CTA's range (null: none)
  int batch, num_q_heads, num_kv_heads, group, max_blocks_per_seq, num_blocks;
  int q_len;                 // new tokens per sequence (q, out: [B, q_len, Hq, D])
  int n_max, min_pages;      // split rule inputs (same values the planner got)
  int fused_merge;           // 1: the last CTA of a split segment merges it
  int merge_helpers;         // CTAs that may share a large segment's final merge (1: the
                             // last alone; more only if every CTA is resident at once)
  int kv_dtype, kv_layout;   // XQA_KV_* code format, XQA_LAYOUT_* cache layout
  double qk_scale_base;      // sm_scale * log2(e); the logit scale is this * k_scale
  float k_scale, v_scale;    // per-tensor scales (used when the pointers are null)
  const float* k_scale_ptr;  // optional device scalars, read when the kernel runs
  const float* v_scale_ptr;
};

struct CombineParams {
  __half* out;
  const int32_t* header;
  const int32_t* seg_start;
  const int32_t* seg_cc;
  int32_t* tickets;  // read for the bad-piece count, then cleared
  const float* partials;
  int num_q_heads, num_kv_heads, group, q_len;
  float v_scale;
  const float* v_scale_ptr;  // optional device scalar (overrides v_scale)
};

cudaError_t launch_plan(const int32_t* context_lens, int batch, int num_kv_heads,
                        int max_blocks_per_seq, int n_max, int min_pages_per_cta,
                        int32_t* workspace, cudaStream_t stream);
cudaError_t launch_partial(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const PartialParams& p, int n_max, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int num_segments, cudaStream_t stream);
cudaError_t launch_wait_timeout(int32_t* status, unsigned long long budget_ns,
                                cudaStream_t stream);
cudaError_t launch_dequant(int kv_dtype, const uint8_t* in, size_t n, float scale,
                           uint16_t* out16, float* out32, cudaStream_t stream);

}  // namespace xqa
