// partial.cu — the split-KV partial attention kernel (the hot loop).
//
// One persistent CTA per planner share of the flattened (sequence, kv head,
// page) order. Its phases are the ones profiled on the page "[Kernel][SM70]
// Pipeline batched E5M2 XQA decode" (section "Pending work and gates"): K load +
// E5M2 conversion, shared-memory publication, QK, V load + conversion, PV and
// synchronization. That page's starting kernel was memory-latency bound
// (long-scoreboard stalls at low occupancy, section "Starting bottleneck"); on
// sm_103a this kernel keeps kStages pages in flight per SM instead.
//
// Every one of the 8 warps both loads and computes. Warp w owns the CTA-local
// pages w, w+8, w+16, ... and the ring slots w, w+8, w+16, w+24 they map to
// (slot = page % kStages). It keeps kLookahead of its pages in flight: after
// computing page q it issues the two 2-D TMA loads (K and V slice, 2048 B each,
// 128-byte swizzle) of its page q + kStages into the slot it just freed, so no
// empty-slot barrier is needed and TMA issue is spread over all warps. Block ids
// are fetched 32 owned pages at a time, one batch ahead (bounds-checked).
//
// Per 16-token page a warp
//   - reads K and V with conflict-free 16-byte shared loads,
//   - dequantises exactly (fp16 pattern = code << 8, a byte permutation),
//   - S^T[16 tok x 8 heads] = K * Q^T with 8 m16n8k16 MMAs (fp32 accumulate),
//   - runs the online softmax in the log2 domain (k_scale and sm_scale folded
//     into one fp32 logit scale; the running max only moves when a logit
//     exceeds it by more than 8, so most pages skip the rescale),
//   - moves P^T to the B-operand layout with two movmatrix transposes,
//   - O^T[128 x 8] += V^T * P^T with 8 MMAs plus one MMA against ones for the
//     row sums l (so l sums exactly the fp16 P used for O).
// At the end of every segment the 8 warps' (m, l, O) are merged in shared
// memory; a segment owned whole by this CTA is normalised and written as fp16
// (out = O * (v_scale / l)); otherwise the piece goes to partial slot i + s for
// the combine kernel.
//
// Contraction-index permutation: the MMA result does not depend on how the
// contraction index is laid out, as long as both operands use the same layout.
// QK lane (g, c) owns dims [32c, 32c+32) of its two token rows; PV lane (g, c)
// owns dims [16g, 16g+16) of tokens {2c, 2c+1, 2c+8, 2c+9}. Both read 16 B per
// shared load, and the TMA 128-byte swizzle (chunk ^= row & 7) makes every
// 8-lane phase hit 8 distinct 16-byte chunks.
#include <math.h>

#include "xqa_device.cuh"
#include "xqa_launch.h"

namespace xqa {

namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kOnesHalf2 = 0x3C003C00u;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

__device__ __forceinline__ int consumer_bar_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kThreads)
      : "memory");
  return r;
}

// Largest s in [lo, nseg) with seg_start[s] <= page, given seg_start[lo] <= page
// < seg_start[nseg]. `seg_start` may point to shared or global memory.
__device__ __forceinline__ int find_segment(const int32_t* seg_start, int lo, int nseg, int page) {
  int hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seg_start[mid] <= page) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// TMA coordinates of 32 consecutive owned pages of one warp, one per lane.
struct PageBatch {
  int y;    // row of the (page, kv head) slice in the [NB*Hkv*16, 128] view
  int bad;  // block id outside [0, NB)
  int seg;  // segment of the page
};

__device__ __forceinline__ PageBatch load_batch(const PartialParams& p, const int32_t* segs,
                                                int s_first, int nseg, int cbeg, int npages,
                                                int warp, int base, int lane) {
  PageBatch r{0, 0, s_first};
  const int q = warp + kWarps * (base + lane);
  if (q < npages) {
    const int pg = cbeg + q;
    const int s = find_segment(segs, s_first, nseg, pg);
    const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
    const int j = pg - segs[s];
    const int id = __ldg(&p.block_tables[(size_t)b * p.max_blocks_per_seq + j]);
    r.bad = (id < 0 || id >= p.num_blocks) ? 1 : 0;
    // HND: row of the (page, kv head) slice; NHD: first token row of the page
    r.y = r.bad ? 0 : (p.kv_layout == XQA_LAYOUT_HND ? (id * p.num_kv_heads + kvh) : id) * kBlockSize;
    r.seg = s;
  }
  return r;
}

// Q of segment s as B fragments: lane (g, c) holds head g, dims [32c, 32c+32).
__device__ __forceinline__ void load_q(const PartialParams& p, int s, int g, int c,
                                       uint32_t (&qf)[16]) {
  const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
  if (g < p.group) {
    const uint4* qp = reinterpret_cast<const uint4*>(
        p.q + ((size_t)b * p.num_q_heads + (size_t)kvh * p.group + g) * kHeadDim + 32 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(qp + i);
      qf[4 * i] = v.x;
      qf[4 * i + 1] = v.y;
      qf[4 * i + 2] = v.z;
      qf[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) qf[i] = 0u;
  }
}

struct WarpState {
  float o[8][4];  // O^T tiles: [tile i][c-frag]; rows d = 16g + 2i (+1), cols heads 2c (+1)
  float l[4];     // row sums per head (cols 2c, 2c+1), replicated over rows
  float m0, m1;   // running max (log2 domain) of heads 2c and 2c+1
};

__device__ __forceinline__ void reset_state(WarpState& st) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) st.o[i][k] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) st.l[k] = 0.f;
  st.m0 = -INFINITY;
  st.m1 = -INFINITY;
}

// One page's K and V bytes as this lane needs them (see the layout note above).
struct PageRegs {
  uint4 ka0, ka1, kb0, kb1;  // K rows g and g+8, dims [32c, 32c+32)
  uint4 vx, vy, vz, vw;      // V tokens 2c, 2c+1, 2c+8, 2c+9, dims [16g, 16g+16)
};

// Shared loads of one stage (swizzled 16-byte chunks, conflict-free).
__device__ __forceinline__ PageRegs load_page(const uint8_t* ks, const uint8_t* vs, int g, int c) {
  PageRegs r;
  const int kc0 = ((2 * c) ^ g) << 4, kc1 = ((2 * c + 1) ^ g) << 4;
  r.ka0 = lds128(ks + g * 128 + kc0);
  r.ka1 = lds128(ks + g * 128 + kc1);
  r.kb0 = lds128(ks + (g + 8) * 128 + kc0);
  r.kb1 = lds128(ks + (g + 8) * 128 + kc1);
  const int ve = (g ^ (2 * c)) << 4, vo = (g ^ (2 * c + 1)) << 4;
  r.vx = lds128(vs + (2 * c) * 128 + ve);
  r.vy = lds128(vs + (2 * c + 1) * 128 + vo);
  r.vz = lds128(vs + (2 * c + 8) * 128 + ve);
  r.vw = lds128(vs + (2 * c + 9) * 128 + vo);
  return r;
}

// NP (1 or 2) 16-token pages of one kv head: QK, one online-softmax update for
// all NP pages, PV. With two pages the two independent QK and PV chains
// interleave, which hides the fixed latencies of one page's chain behind the
// other's.
template <int kFmt, int NP>
__device__ __forceinline__ void process_pages(WarpState& st, const PageRegs (&r)[NP],
                                              const uint32_t (&qf)[16], const int (&nvalid)[NP],
                                              float scale_log2, int g, int c) {
  // ---- S^T = K * Q^T : rows tokens (g, g+8), cols heads (2c, 2c+1) ----
  float s[NP][4];
#pragma unroll
  for (int pi = 0; pi < NP; ++pi) {
    const uint32_t kr0[8] = {r[pi].ka0.x, r[pi].ka0.y, r[pi].ka0.z, r[pi].ka0.w,
                             r[pi].ka1.x, r[pi].ka1.y, r[pi].ka1.z, r[pi].ka1.w};
    const uint32_t kr1[8] = {r[pi].kb0.x, r[pi].kb0.y, r[pi].kb0.z, r[pi].kb0.w,
                             r[pi].kb1.x, r[pi].kb1.y, r[pi].kb1.z, r[pi].kb1.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) s[pi][k] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mma_16816(s[pi], KvConv<kFmt>::k_lo(kr0[j]), KvConv<kFmt>::k_lo(kr1[j]),
                KvConv<kFmt>::k_hi(kr0[j]), KvConv<kFmt>::k_hi(kr1[j]), qf[2 * j],
                qf[2 * j + 1]);
    }
  }

  // ---- online softmax (log2 domain), one update for all NP pages ----
  float t[NP][4];
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int pi = 0; pi < NP; ++pi) {
#pragma unroll
    for (int k = 0; k < 4; ++k) t[pi][k] = s[pi][k] * scale_log2;
    if (nvalid[pi] < kBlockSize) {
      if (g >= nvalid[pi]) t[pi][0] = t[pi][1] = -INFINITY;
      if (g + 8 >= nvalid[pi]) t[pi][2] = t[pi][3] = -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(t[pi][0], t[pi][2]));
    mx1 = fmaxf(mx1, fmaxf(t[pi][1], t[pi][3]));
  }
  const bool need = (mx0 > st.m0 + kRescaleThreshold) || (mx1 > st.m1 + kRescaleThreshold);
  if (__any_sync(kFull, need)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
    }
    const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
    const float a0 = ex2(st.m0 - n0), a1 = ex2(st.m1 - n1);
    st.m0 = n0;
    st.m1 = n1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.o[i][0] *= a0;
      st.o[i][2] *= a0;
      st.o[i][1] *= a1;
      st.o[i][3] *= a1;
    }
    st.l[0] *= a0;
    st.l[2] *= a0;
    st.l[1] *= a1;
    st.l[3] *= a1;
  }

#pragma unroll
  for (int pi = 0; pi < NP; ++pi) {
    const float p0 = ex2(t[pi][0] - st.m0), p1 = ex2(t[pi][1] - st.m1);
    const float p2 = ex2(t[pi][2] - st.m0), p3 = ex2(t[pi][3] - st.m1);
    // P^T B-fragments: lane (g, c) gets P[tokens 2c, 2c+1 | 2c+8, 2c+9][head g]
    const uint32_t pb0 = movmatrix_trans(pack_half2(p0, p1));
    const uint32_t pb1 = movmatrix_trans(pack_half2(p2, p3));

    // ---- O^T += V^T * P^T ----
    uint4 vx = r[pi].vx, vy = r[pi].vy, vz = r[pi].vz, vw = r[pi].vw;
    if (nvalid[pi] < kBlockSize) {  // zero V rows past the context (0 * NaN would poison O)
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (2 * c >= nvalid[pi]) vx = z;
      if (2 * c + 1 >= nvalid[pi]) vy = z;
      if (2 * c + 8 >= nvalid[pi]) vz = z;
      if (2 * c + 9 >= nvalid[pi]) vw = z;
    }
    const uint32_t X[4] = {vx.x, vx.y, vx.z, vx.w}, Y[4] = {vy.x, vy.y, vy.z, vy.w};
    const uint32_t Z[4] = {vz.x, vz.y, vz.z, vz.w}, W[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t xy[4], zw[4];  // {x_k, y_k}: tokens 2c, 2c+1 / 2c+8, 2c+9 at dim byte k
      KvConv<kFmt>::v_pairs(X[u], Y[u], xy);
      KvConv<kFmt>::v_pairs(Z[u], W[u], zw);
      mma_16816(st.o[2 * u], xy[0], xy[1], zw[0], zw[1], pb0, pb1);
      mma_16816(st.o[2 * u + 1], xy[2], xy[3], zw[2], zw[3], pb0, pb1);
    }
    mma_16816(st.l, kOnesHalf2, kOnesHalf2, kOnesHalf2, kOnesHalf2, pb0, pb1);
  }
}

// LSE merge of all pieces of split segment s into fp16 rows (thread: head h,
// dims dq..dq+3). Pieces were written by other CTAs: read through L2.
__device__ __forceinline__ void merge_pieces(const PartialParams& p, int s, int sb, int se,
                                             int total, int n, int h, int dq, float v_scale) {
  if (h >= p.group) return;
  const int ilo = cta_of_page(sb, total, n), ihi = cta_of_page(se - 1, total, n);
  const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
  __half* o = p.out + ((size_t)b * p.num_q_heads + (size_t)kvh * p.group + h) * kHeadDim + dq;
  uint2 v;
  if (__ldcg(&p.seg_bad[s]) != 0) {
    const float nan = __int_as_float(0x7fc00000);
    v.x = pack_half2(nan, nan);
    v.y = v.x;
    *reinterpret_cast<uint2*>(o) = v;
    return;
  }
  float M = -INFINITY;
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kFew = 4;
  if (ihi - ilo < kFew) {
    // usual case: every load issued before any is used (one L2 round trip)
    float mi[kFew], li[kFew];
    float4 oi[kFew];
#pragma unroll
    for (int k = 0; k < kFew; ++k) {
      if (ilo + k <= ihi) {
        const float* slot = p.partials + (size_t)(ilo + k + s) * kSlotFloats;
        mi[k] = __ldcg(slot + kMaxGroup * kHeadDim + h);
        li[k] = __ldcg(slot + kMaxGroup * kHeadDim + kMaxGroup + h);
        oi[k] = __ldcg(reinterpret_cast<const float4*>(slot + h * kHeadDim + dq));
      }
    }
#pragma unroll
    for (int k = 0; k < kFew; ++k)
      if (ilo + k <= ihi) M = fmaxf(M, mi[k]);
#pragma unroll
    for (int k = 0; k < kFew; ++k) {
      if (ilo + k <= ihi) {
        const float w = (mi[k] == -INFINITY) ? 0.f : ex2(mi[k] - M);
        L += w * li[k];
        acc.x += w * oi[k].x;
        acc.y += w * oi[k].y;
        acc.z += w * oi[k].z;
        acc.w += w * oi[k].w;
      }
    }
    const float r = v_scale / L;
    v.x = pack_half2(acc.x * r, acc.y * r);
    v.y = pack_half2(acc.z * r, acc.w * r);
    *reinterpret_cast<uint2*>(o) = v;
    return;
  }
  for (int i = ilo; i <= ihi; ++i)
    M = fmaxf(M, __ldcg(p.partials + (size_t)(i + s) * kSlotFloats + kMaxGroup * kHeadDim + h));
  for (int i = ilo; i <= ihi; ++i) {
    const float* slot = p.partials + (size_t)(i + s) * kSlotFloats;
    const float mi = __ldcg(slot + kMaxGroup * kHeadDim + h);
    const float w = (mi == -INFINITY) ? 0.f : ex2(mi - M);
    L += w * __ldcg(slot + kMaxGroup * kHeadDim + kMaxGroup + h);
    const float4 x = __ldcg(reinterpret_cast<const float4*>(slot + h * kHeadDim + dq));
    acc.x += w * x.x;
    acc.y += w * x.y;
    acc.z += w * x.z;
    acc.w += w * x.w;
  }
  const float r = v_scale / L;
  v.x = pack_half2(acc.x * r, acc.y * r);
  v.y = pack_half2(acc.z * r, acc.w * r);
  *reinterpret_cast<uint2*>(o) = v;
}

}  // namespace

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ int stage_bad[kStages];
  __shared__ int abort_flag;

  __shared__ int scan_warp[kWarps];
  __shared__ int scan_carry;
  // split pieces of this CTA (at most its first and last segment), whose
  // merge tickets are taken once the whole range is done
  __shared__ int pend_seg[2], pend_poison[2], pend_last[2];
  __shared__ int npend;
  // the segment each merge buffer holds, whether this CTA owns it whole, and
  // each warp's "met a bad page" flag for it
  __shared__ int buf_seg[kMergeBufs], buf_whole[kMergeBufs], buf_poison[kMergeBufs][kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int nseg = p.batch * p.num_kv_heads;
  // per-tensor scales: host values, or device scalars read when the kernel runs
  const float k_scale = p.k_scale_ptr ? __ldg(p.k_scale_ptr) : p.k_scale;
  const float v_scale = p.v_scale_ptr ? __ldg(p.v_scale_ptr) : p.v_scale;
  const float scale_log2 = static_cast<float>(p.qk_scale_base * static_cast<double>(k_scale));

  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* merge_bufs = reinterpret_cast<float*>(stages + kStages * kStageBytes);
  int32_t* seg_cache = reinterpret_cast<int32_t*>(merge_bufs + kMergeBufs * kMergeBufFloats);

  // ---- the plan: computed here when the segment table fits in shared memory
  // (same integer rule as the planner kernel), else read from the planner ----
  const bool segs_in_smem = nseg + 1 <= kSegCache;
  const int32_t* segs;
  int total, n;
  if (segs_in_smem) {
    if (tid == 0) scan_carry = 0;
    __syncthreads();
    const long long max_ctx = (long long)p.max_blocks_per_seq * kBlockSize;
    for (int base = 0; base < p.batch; base += kThreads) {
      const int b = base + tid;
      int pages = 0;
      if (b < p.batch) {
        const int ctx = __ldg(&p.context_lens[b]);
        pages = (ctx < 0 || (long long)ctx > max_ctx) ? 0 : (ctx + kBlockSize - 1) / kBlockSize;
      }
      int incl = pages;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += u;
      }
      if (lane == 31) scan_warp[warp] = incl;
      __syncthreads();
      int before = scan_carry;
      for (int w = 0; w < warp; ++w) before += scan_warp[w];
      const int excl = before + incl - pages;
      if (b < p.batch)
        for (int h = 0; h < p.num_kv_heads; ++h)
          seg_cache[b * p.num_kv_heads + h] = excl * p.num_kv_heads + h * pages;
      __syncthreads();
      if (tid == kThreads - 1) scan_carry = excl + pages;
      __syncthreads();
    }
    total = scan_carry * p.num_kv_heads;
    if (tid == 0) seg_cache[nseg] = total;
    n = num_ctas_for(total, p.n_max, p.min_pages);
    segs = seg_cache;
  } else {
    griddep_wait();
    total = p.header[2];
    n = p.header[1];
    segs = p.seg_start;
  }
  __syncthreads();

  // ---- rows of empty segments (context length 0, or invalid -> NaN) ----
  if (cta == 0) {
    const long long max_ctx = (long long)p.max_blocks_per_seq * kBlockSize;
    for (int s = warp; s < nseg; s += kWarps) {
      if (segs[s] != segs[s + 1]) continue;
      const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
      const int ctx = __ldg(&p.context_lens[b]);
      const bool bad = ctx < 0 || (long long)ctx > max_ctx;
      const float v = bad ? __int_as_float(0x7fc00000) : 0.0f;
      uint4 val;
      val.x = val.y = val.z = val.w = pack_half2(v, v);
      for (int i = lane; i < p.group * (kHeadDim / 8); i += 32) {
        const int h = i / (kHeadDim / 8), d8 = i - h * (kHeadDim / 8);
        __half* o = p.out + ((size_t)b * p.num_q_heads + (size_t)kvh * p.group + h) * kHeadDim;
        reinterpret_cast<uint4*>(o)[d8] = val;
      }
    }
  }
  if (cta >= n) return;
  const int cbeg = (int)(((long long)cta * total) / n);
  const int cend = (int)(((long long)(cta + 1) * total) / n);
  const int npages = cend - cbeg;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full_bar[i], 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  __syncthreads();
  const int s_first = find_segment(segs, 0, nseg, cbeg);
  volatile int* abort = &abort_flag;
  const uint64_t policy = l2_evict_first_policy();
  const int g = lane >> 2, c = lane & 3;

  // ---- this warp's loads: owned page k is CTA-local page warp + 8k ----
  const int owned = npages > warp ? (npages - warp + kWarps - 1) / kWarps : 0;
  PageBatch cur = load_batch(p, segs, s_first, nseg, cbeg, npages, warp, 0, lane);
  PageBatch nxt = load_batch(p, segs, s_first, nseg, cbeg, npages, warp, 32, lane);
  int cur_base = 0;
  int issued = 0;  // owned pages whose loads have been issued
  auto issue_next = [&]() {
    if (issued >= owned) return;
    const int k = issued++;
    if (k >= cur_base + 32) {
      cur = nxt;
      cur_base += 32;
      nxt = load_batch(p, segs, s_first, nseg, cbeg, npages, warp, cur_base + 32, lane);
    }
    const int y = __shfl_sync(kFull, cur.y, k - cur_base);
    const int bad = __shfl_sync(kFull, cur.bad, k - cur_base);
    const int sg = __shfl_sync(kFull, cur.seg, k - cur_base);
    const int slot = (warp + kWarps * k) % kStages;
    __syncwarp();  // all lanes' reads of this slot's previous page are done
    if (lane == 0) {
      uint8_t* st = stages + slot * kStageBytes;
      stage_bad[slot] = bad;
      fence_proxy_async_smem();  // this slot's earlier shared reads come before the TMA writes
      if (bad) {
        griddep_wait();  // the planner resets seg_bad and the status word
        atomicOr(&p.seg_bad[sg], 1);
        record_status(&p.header[0], XQA_ERR_BAD_BLOCK_ID);
        mbar_arrive(&full_bar[slot]);
      } else {
        mbar_arrive_expect_tx(&full_bar[slot], kStageBytes);
        if (p.kv_layout == XQA_LAYOUT_HND) {
          tma_load_2d(st, &tm_k, &full_bar[slot], 0, y, policy);
          tma_load_2d(st + kPageBytes, &tm_v, &full_bar[slot], 0, y, policy);
        } else {  // NHD: box (128 dims, 1 kv head, 16 tokens) at (0, kvh, page*16)
          const int kvh = sg - (sg / p.num_kv_heads) * p.num_kv_heads;
          tma_load_3d(st, &tm_k, &full_bar[slot], 0, kvh, y, policy);
          tma_load_3d(st + kPageBytes, &tm_v, &full_bar[slot], 0, kvh, y, policy);
        }
      }
    }
    __syncwarp();
  };
#pragma unroll 1
  for (int i = 0; i < kLookahead; ++i) issue_next();

  if (tid == 0) npend = 0;
  WarpState st;
  uint32_t qf[16], qf_next[16];
  int q_next_seg = -1;
  // Merge of one buffered segment by all threads (head h, dims dq..dq+3): the
  // 8 warps' (m, l, O) combine in shared memory; a segment owned whole is
  // normalised and written as fp16, a split piece goes to partial slot cta + s.
  auto merge_buffer = [&](int mb) {
    const int ms = buf_seg[mb];
    const bool mwhole = buf_whole[mb] != 0;
    int any_poison = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) any_poison |= buf_poison[mb][w];
    const float* base = merge_bufs + mb * kMergeBufFloats;
    const float* bm = base + kScratchFloats;
    const float* bl = bm + kWarps * kMaxGroup;
    const int h = tid >> 5;         // 0..7
    const int dq = (tid & 31) * 4;  // 0..124
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, bm[w * kMaxGroup + h]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = bm[w * kMaxGroup + h];
      const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      L += sc * bl[w * kMaxGroup + h];
      const float4 v =
          *reinterpret_cast<const float4*>(base + (w * kMaxGroup + h) * kScratchStride + dq);
      acc.x += sc * v.x;
      acc.y += sc * v.y;
      acc.z += sc * v.z;
      acc.w += sc * v.w;
    }
    const int mb_b = ms / p.num_kv_heads, mb_kvh = ms - mb_b * p.num_kv_heads;
    if (h < p.group) {
      if (mwhole) {
        __half* o = p.out +
                    ((size_t)mb_b * p.num_q_heads + (size_t)mb_kvh * p.group + h) * kHeadDim + dq;
        const float r = v_scale / L;
        uint2 v;
        if (any_poison) {
          const float nan = __int_as_float(0x7fc00000);
          v.x = pack_half2(nan, nan);
          v.y = v.x;
        } else {
          v.x = pack_half2(acc.x * r, acc.y * r);
          v.y = pack_half2(acc.z * r, acc.w * r);
        }
        *reinterpret_cast<uint2*>(o) = v;
      } else {
        float* slotp = p.partials + (size_t)(cta + ms) * kSlotFloats;
        *reinterpret_cast<float4*>(slotp + h * kHeadDim + dq) = acc;
        if (dq == 0) {
          slotp[kMaxGroup * kHeadDim + h] = M;
          slotp[kMaxGroup * kHeadDim + kMaxGroup + h] = L;
        }
      }
    }
    if (!mwhole && tid == 0) {  // a split piece: its ticket is taken after the range
      pend_seg[npend] = ms;
      pend_poison[npend] = any_poison;
      ++npend;
    }
  };

  int kseg = 0;  // segments of this range finished so far
  int s = s_first;
  int q0 = 0;
  while (q0 < npages) {
    while (segs[s + 1] <= cbeg + q0) ++s;
    const int sb = segs[s], se = segs[s + 1];
    const int qe = min(se, cend) - cbeg;
    const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
    const int ctx = __ldg(&p.context_lens[b]);
    const bool whole = (sb >= cbeg) && (se <= cend);
    if (q_next_seg == s) {
#pragma unroll
      for (int i = 0; i < 16; ++i) qf[i] = qf_next[i];
    } else {
      load_q(p, s, g, c, qf);
    }
    if (qe < npages) {  // prefetch Q of the next segment this CTA works on
      q_next_seg = find_segment(segs, s, nseg, cbeg + qe);
      load_q(p, q_next_seg, g, c, qf_next);
    }
    reset_state(st);
    int poisoned = 0;

    // this warp's pages of the segment, two at a time (q and q + kWarps)
    for (int q = q0 + ((warp - q0 % kWarps) + kWarps) % kWarps; q < qe; q += 2 * kWarps) {
      const bool pair = q + kWarps < qe;
      const int slot0 = q % kStages, slot1 = (q + kWarps) % kStages;
      bool ready = mbar_wait_bounded(&full_bar[slot0], (q / kStages) & 1, abort);
      if (pair) ready = ready && mbar_wait_bounded(&full_bar[slot1], ((q + kWarps) / kStages) & 1, abort);
      if (!__all_sync(kFull, ready)) {  // warp-uniform outcome
        poisoned = 1;
        if (lane == 0) {
          *abort = 1;
          griddep_wait();
          record_status(&p.header[0], XQA_ERR_DEVICE_TIMEOUT);
        }
        continue;
      }
      const uint8_t* stg0 = stages + slot0 * kStageBytes;
      const uint8_t* stg1 = stages + slot1 * kStageBytes;
      const bool bad0 = stage_bad[slot0] != 0, bad1 = pair && stage_bad[slot1] != 0;
      PageRegs regs[2];
      regs[0] = load_page(stg0, stg0 + kPageBytes, g, c);
      if (pair) regs[1] = load_page(stg1, stg1 + kPageBytes, g, c);
      // The pages are in registers: refill their slots with the pages kStages
      // ahead right away (warp-uniform decision), before the math.
      if (!__any_sync(kFull, *abort != 0)) {
        issue_next();
        if (pair) issue_next();
      }
      const int j0 = cbeg + q - sb;
      const int nv0 = min(kBlockSize, ctx - j0 * kBlockSize);
      const int nv1 = min(kBlockSize, ctx - (j0 + kWarps) * kBlockSize);
      if (pair && !bad0 && !bad1) {
        const int nv[2] = {nv0, nv1};
        process_pages<kFmt, 2>(st, regs, qf, nv, scale_log2, g, c);
      } else {
        if (bad0 || bad1) poisoned = 1;
        if (!bad0) {
          const PageRegs one[1] = {regs[0]};
          const int nv[1] = {nv0};
          process_pages<kFmt, 1>(st, one, qf, nv, scale_log2, g, c);
        }
        if (pair && !bad1) {
          const PageRegs one[1] = {regs[1]};
          const int nv[1] = {nv1};
          process_pages<kFmt, 1>(st, one, qf, nv, scale_log2, g, c);
        }
      }
    }

    // ---- hand this segment's per-warp state to a merge buffer; no CTA-wide
    // barrier unless the buffer still holds the segment before the previous
    // one (so a range with at most two segments never stops mid-way) ----
    const int buf = kseg & 1;
    if (kseg >= 2) {
      consumer_bar();
      merge_buffer(buf);
      consumer_bar();
    }
    {
      float* my = merge_bufs + buf * kMergeBufFloats + warp * kMaxGroup * kScratchStride;
      float* bm = merge_bufs + buf * kMergeBufFloats + kScratchFloats;
      float* bl = bm + kWarps * kMaxGroup;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d0 = 16 * g + 2 * i;
        my[(2 * c) * kScratchStride + d0] = st.o[i][0];
        my[(2 * c + 1) * kScratchStride + d0] = st.o[i][1];
        my[(2 * c) * kScratchStride + d0 + 1] = st.o[i][2];
        my[(2 * c + 1) * kScratchStride + d0 + 1] = st.o[i][3];
      }
      if (g == 0) {
        bm[warp * kMaxGroup + 2 * c] = st.m0;
        bm[warp * kMaxGroup + 2 * c + 1] = st.m1;
        bl[warp * kMaxGroup + 2 * c] = st.l[0];
        bl[warp * kMaxGroup + 2 * c + 1] = st.l[1];
      }
      if (lane == 0) buf_poison[buf][warp] = poisoned;
      if (tid == 0) {
        buf_seg[buf] = s;
        buf_whole[buf] = whole ? 1 : 0;
      }
    }
    ++kseg;
    q0 = qe;
    ++s;
  }

  // ---- merges still buffered (the range's last one or two segments) ----
  consumer_bar();
  if (kseg >= 2) merge_buffer(kseg & 1);
  if (kseg >= 1) merge_buffer((kseg - 1) & 1);
  consumer_bar();

  // ---- split pieces: flag, ticket, and merge by the CTA that finishes last ----
  // The ticket (a device-wide atomic round trip) is taken once per piece after
  // the whole range, so no mid-range segment boundary stalls the CTA on it.
  // The CTA whose ticket completes a segment merges all its pieces in slot
  // order, exactly as the combine kernel would.
  if (npend > 0) {
    griddep_wait();  // the planner's resets of seg_bad / seg_count are visible
    consumer_bar();  // all of this CTA's partial-slot writes precede the tickets
    if (tid < npend) {
      const int s = pend_seg[tid];
      if (pend_poison[tid]) atomicOr(&p.seg_bad[s], 1);
      int last = 0;
      if (p.fused_merge) {
        const int ilo = cta_of_page(segs[s], total, n), ihi = cta_of_page(segs[s + 1] - 1, total, n);
        // release: this CTA's slots (ordered before by the barrier) are visible
        // to whoever takes a later ticket; acquire: the earlier pieces are
        // visible to this CTA after the next barrier
        last = (atom_add_acq_rel_gpu(&p.seg_count[s], 1) == ihi - ilo) ? 1 : 0;
      }
      pend_last[tid] = last;
    }
    consumer_bar();
    for (int i = 0; i < npend; ++i) {
      if (!pend_last[i]) continue;
      const int s = pend_seg[i];
      merge_pieces(p, s, segs[s], segs[s + 1], total, n, tid >> 5, (tid & 31) * 4, v_scale);
    }
  }

  // Drain: after an abort some issued copies may not have been waited for; every
  // copy must land before the CTA's shared memory is released.
  if (*abort) {
    int never = 0;
    volatile int* no_abort = &never;
    // only the last kLookahead issued pages can still be in flight: every
    // earlier one was waited for before its slot was reissued
    const int first = issued > kLookahead ? issued - kLookahead : 0;
    for (int k = first; k < issued; ++k) {
      const int q = warp + kWarps * k;
      const bool ok = mbar_wait_bounded(&full_bar[q % kStages], (q / kStages) & 1, no_abort);
      if (!__all_sync(kFull, ok)) break;
    }
  }
}

cudaError_t launch_partial(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const PartialParams& p, int n_max, cudaStream_t stream) {
  // Programmatic dependent launch: CTAs may start while the planner (the
  // previous kernel on the stream) still runs; the kernel waits for it with
  // griddepcontrol.wait before reading or writing anything the planner writes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_max);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPartialSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.kv_dtype == XQA_KV_E4M3)
    return cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E4M3>, tm_k, tm_v, p);
  return cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E5M2>, tm_k, tm_v, p);
}

cudaError_t set_partial_attributes() {
  cudaError_t e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E5M2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPartialSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(partial_kernel<XQA_KV_E4M3>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kPartialSmem);
}

}  // namespace xqa
