// plan.cu — the split-KV planner (one CTA).
//
// Reads context_lens[B] and publishes, in the workspace, the pages of every
// (sequence, kv head) segment as an exclusive prefix sum, the bad-segment
// flags, the cost-line prefix, the total page count and the number of
// partial-kernel CTAs. The cost line lays the segments end to end, each
// preceded by its switch cost (seg_cost: 32 page units for a non-empty
// segment); CTA i of the partial kernel owns the pages at positions
// [floor(i*V/n), floor((i+1)*V/n)) of that line. Every CTA gets the same cost
// whatever the length mix: long sequences are split across CTAs, short ones
// share a CTA, and many tiny segments are spread over several. This answers the two failure
// modes recorded on the page "[Kernel][WIP] Follow up FlashNext batch HC fusion
// and QSA route audit" (section "Test Result"): a capacity-sized grid with
// empty CTAs on short contexts, and fixed grids that regress long ones. The
// plan is computed on the device so the decode step needs no host sync.
//
// The partial kernel derives the same plan itself whenever the segment table
// fits in its shared memory; this kernel is launched only for larger batches
// (and on request, through xqa_plan). It is launched as a programmatic
// dependent of the previous kernel on the stream: it becomes resident early
// and waits for that kernel to complete before it reads or writes anything;
// the partial kernel, its own programmatic dependent, waits for it in turn.
#include "xqa_device.cuh"
#include "xqa_launch.h"

namespace xqa {

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += u;
  }
  return v;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ context_lens,
                                                            int batch, int num_kv_heads,
                                                            int max_blocks_per_seq, int n_max,
                                                            int min_pages, int32_t* ws) {
  griddep_wait();               // everything earlier on the stream is complete
  griddep_launch_dependents();  // the partial kernel may start its prologue now
  constexpr int kPlanWarps = kPlanThreads / 32;
  const int nseg = batch * num_kv_heads;
  const WsLayout lay = ws_layout(nseg, 0);
  int32_t* header = ws;
  int32_t* seg_start = ws + lay.seg_start_off / 4;
  int32_t* seg_bad = ws + lay.seg_bad_off / 4;
  int32_t* seg_cc = ws + lay.seg_cc_off / 4;
  __shared__ int warp_total[kPlanWarps], warp_cost[kPlanWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long max_ctx = (long long)max_blocks_per_seq * kBlockSize;
  auto pages_of = [&](int s, bool& bad) {
    const int ctx = context_lens[s / num_kv_heads];
    bad = ctx < 0 || (long long)ctx > max_ctx;
    return bad ? 0 : (ctx + kBlockSize - 1) / kBlockSize;
  };
  // Thread tid owns the consecutive segments [s0, s1). Its pages and costs
  // are summed first (independent loads, no stores in between), one block
  // scan turns the sums into the thread's offsets, and a second pass writes
  // the rows: one scan and a single round of load latency for any batch.
  const int per = (nseg + kPlanThreads - 1) / kPlanThreads;
  const int s0 = min(nseg, tid * per), s1 = min(nseg, s0 + per);
  int my_pages = 0, my_cost = 0;
#pragma unroll 8
  for (int s = s0; s < s1; ++s) {
    bool bad;
    const int pg = pages_of(s, bad);
    my_pages += pg;
    my_cost += seg_cost(pg);
  }
  const int incl = warp_inclusive_scan(my_pages);
  const int incl_cost = warp_inclusive_scan(my_cost);
  if (lane == 31) {
    warp_total[warp] = incl;
    warp_cost[warp] = incl_cost;
  }
  __syncthreads();
  if (warp == 0) {
    const int t = warp_inclusive_scan(lane < kPlanWarps ? warp_total[lane] : 0);
    const int tc = warp_inclusive_scan(lane < kPlanWarps ? warp_cost[lane] : 0);
    if (lane < kPlanWarps) {
      warp_total[lane] = t;
      warp_cost[lane] = tc;
    }
  }
  __syncthreads();
  int start = incl - my_pages + (warp > 0 ? warp_total[warp - 1] : 0);  // exclusive
  int cc = incl_cost - my_cost + (warp > 0 ? warp_cost[warp - 1] : 0);
  for (int s = s0; s < s1; ++s) {
    bool bad;
    const int pg = pages_of(s, bad);
    seg_bad[s] = bad ? 1 : 0;
    seg_start[s] = start;
    cc += seg_cost(pg);
    seg_cc[s] = cc;  // inclusive: the switch costs of segments 0 .. s
    start += pg;
  }
  if (tid == kPlanThreads - 1) {
    const int total = warp_total[kPlanWarps - 1];
    seg_start[nseg] = total;
    header[2] = total;
    header[3] = nseg;
    header[1] = num_ctas_for(total, n_max, min_pages);
  }
}

cudaError_t launch_plan(const int32_t* context_lens, int batch, int num_kv_heads,
                        int max_blocks_per_seq, int n_max, int min_pages_per_cta,
                        int32_t* workspace, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, context_lens, batch, num_kv_heads,
                            max_blocks_per_seq, n_max, min_pages_per_cta, workspace);
}

}  // namespace xqa
