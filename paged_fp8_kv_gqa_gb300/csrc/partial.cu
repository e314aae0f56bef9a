// partial.cu — the split-KV partial attention kernel (the hot loop).
//
// One persistent CTA per planner share of the flattened (sequence, kv head,
// page) order, cut on the planner's cost line (each segment's switch cost
// counted beside its pages; the CTA derives the plan itself from the context
// lengths when the segment table fits in shared memory). Its steps are the
// phases whose cost the page "[Kernel][SM70] Pipeline batched E5M2 XQA decode"
// (section "Pending work and gates") sets out to attribute: bringing in K and
// decoding it from E5M2, making it visible to the other warps through shared
// memory, the QK product, bringing in and decoding V, the PV product, and the
// waits between them. That page's starting kernel was memory-latency bound
// (long-scoreboard stalls at low occupancy, section "Starting bottleneck"); on
// sm_103a this kernel keeps kStages pages in flight per SM instead.
//
// Every one of the 8 warps both loads and computes. Warp w owns the CTA-local
// pages w, w+8, w+16, ... and the ring slots w, w+8, w+16, w+24 they map to
// (slot = page % kStages). It keeps kLookahead of its pages in flight: once a
// page is in registers it issues the two TMA loads (K and V slice, 2048 B each,
// 128-byte swizzle) of its page q + kStages into the slot just freed, so no
// empty-slot barrier is needed and TMA issue is spread over all warps. Block ids
// are fetched 32 owned pages at a time, one batch ahead (bounds-checked).
//
// Columns: the MMA N dimension holds (new token i, q head h) pairs of one kv
// head, column = i * G + h, 8 per tile; single-token decode has G columns and
// one tile, multi-token decode up to 16 columns in two tiles (NT).
//
// Per 16-token page a warp
//   - reads K and V with conflict-free 16-byte shared loads,
//   - dequantises exactly (E5M2: fp16 pattern = code << 8, a byte permutation;
//     E4M3: the hardware pair conversion),
//   - S^T[16 tok x 8 cols] = K * Q^T with 8 m16n8k16 MMAs per tile (fp32 acc),
//   - masks tokens past each column's causal limit (ctx - 1 for single-token
//     decode), then runs the online softmax in the log2 domain (k_scale and
//     sm_scale folded into one fp32 logit scale; the running max only moves
//     when a logit exceeds it by more than 8, so most pages skip the rescale),
//   - moves P^T to the B-operand layout with two movmatrix transposes per tile,
//   - O^T[128 x 8] += V^T * P^T with 8 MMAs per tile (V converted once for all
//     tiles) plus one MMA against ones for the row sums l (so l sums exactly
//     the fp16 P used for O).
// A warp takes its pages two at a time, interleaving two independent
// dependency chains (two-tile kernels load Q per segment instead of
// prefetching it, to stay within 255 registers). At the end of a segment each
// warp hands its (m, l, O) to a shared merge buffer and moves on; the buffered
// segments are merged across warps when a buffer is reused and at the end of
// the range. A segment owned whole by this CTA is normalised and written as
// fp16 (out = O * (v_scale / l)); a split piece goes to partial slot i + s, and
// the CTA whose ticket completes the segment merges all its pieces, loading
// them (and those of its other completed segment) before using any.
//
// Bookkeeping across calls needs no reset kernel: a split segment's merge
// ticket (the workspace word of the CTA holding its first page) counts the
// pieces and the pieces that met a bad page, and the CTA that completes it
// clears it; every CTA writes its own status word as it exits. So with the
// segment table in shared memory a decode step is this one launch, which may
// become resident while the previous kernel on the stream still runs and
// waits for it before reading any input.
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
// Running-max start value: finite, so a column that has seen no visible token
// yet needs no special case: 2^(-inf - kNoMax) = 0 for its masked logits, its
// rescale factor stays 2^0 = 1, and the first real maximum rescales its
// all-zero state by 2^(kNoMax - m) = 0.
constexpr float kNoMax = -1e30f;
constexpr uint32_t kOnesHalf2 = 0x3C003C00u;
constexpr unsigned kFull = 0xffffffffu;

}  // namespace

// Phase stamps, in diagnostic builds only (compiled with -DXQA_STAMPS; the
// library itself is built without them): thread 0 of every CTA records
// %globaltimer at fixed points of the kernel, kStampsPerCta per CTA, which
// xqa_diag_read_stamps copies out. They add a few stores and skip no work.
//   0 entry                 1 inputs readable (after the wait for the
//   2 range known             previous kernels)
//   3 first pages in warp 0's registers
//   4 every warp done with its pages      5 buffered merges written
//   6 merge tickets taken                 7 exit
// and two counts: 8 the CTA's pages, 9 the segments its range touches; then
//   10 context lengths in registers   11 first block ids in registers
//   12 every warp past the wait       13 plan done (before the range search)
//   14 page loop entered              15 first segment search done
//   16 final merge: piece range known 17 final merge: first segment's loads in
constexpr int kStampsPerCta = 18;
#ifdef XQA_STAMPS
__device__ unsigned long long g_stamps[kMaxCtas * kStampsPerCta];
__device__ __forceinline__ void stamp(int i) {
  if (threadIdx.x == 0) g_stamps[blockIdx.x * kStampsPerCta + i] = global_timer_ns();
}
__device__ __forceinline__ void stamp_count(int i, int v) {
  if (threadIdx.x == 0) g_stamps[blockIdx.x * kStampsPerCta + i] = (unsigned long long)v;
}
// the time once v (a load's result) is in thread 0's registers
__device__ __forceinline__ void stamp_after(int i, int v) {
  if (threadIdx.x == 0) {
    asm volatile("" ::"r"(v));
    g_stamps[blockIdx.x * kStampsPerCta + i] = global_timer_ns();
  }
}
#else
__device__ __forceinline__ void stamp(int) {}
__device__ __forceinline__ void stamp_count(int, int) {}
__device__ __forceinline__ void stamp_after(int, int) {}
#endif

namespace {

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
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
  int y;    // HND: row of the (page, kv head) slice; NHD: first token row of the page
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
    if (base == 0) stamp_after(15, s);
    const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
    const int j = pg - segs[s];
    const int id = __ldg(&p.block_tables[(size_t)b * p.max_blocks_per_seq + j]);
    r.bad = (id < 0 || id >= p.num_blocks) ? 1 : 0;
    r.y = r.bad ? 0 : (p.kv_layout == XQA_LAYOUT_HND ? (id * p.num_kv_heads + kvh) : id) * kBlockSize;
    r.seg = s;
  }
  return r;
}

// Output / query row of column col (new token i = col / G, head h = col % G)
// of segment s: ((b * T + i) * Hq + kvh * G + h).
__device__ __forceinline__ size_t col_row(const PartialParams& p, int s, int col) {
  const int b = s / p.num_kv_heads, kvh = s - b * p.num_kv_heads;
  const int i = col / p.group, h = col - i * p.group;
  return ((size_t)b * p.q_len + i) * p.num_q_heads + (size_t)kvh * p.group + h;
}

// Q of segment s as B fragments: lane (g, c) holds column 8j + g of tile j,
// dims [32c, 32c+32); columns past G * q_len are zero.
template <int NT>
__device__ __forceinline__ void load_q(const PartialParams& p, int s, int g, int c,
                                       uint32_t (&qf)[NT][16]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int col = 8 * j + g;
    if (col < p.group * p.q_len) {
      const uint4* qp = reinterpret_cast<const uint4*>(p.q + col_row(p, s, col) * kHeadDim + 32 * c);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(qp + i);
        qf[j][4 * i] = v.x;
        qf[j][4 * i + 1] = v.y;
        qf[j][4 * i + 2] = v.z;
        qf[j][4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) qf[j][i] = 0u;
    }
  }
}

template <int NT>
struct WarpState {
  float o[NT][8][4];  // O^T tiles per column tile: rows d = 16g + 2i (+1), cols 2c (+1)
  float l[NT][4];     // row sums per column (2c, 2c+1), replicated over rows
  float m[NT][2];     // running max (log2 domain) of columns 2c and 2c+1
};

template <int NT>
__device__ __forceinline__ void reset_state(WarpState<NT>& st) {
#pragma unroll
  for (int j = 0; j < NT; ++j) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) st.o[j][i][k] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) st.l[j][k] = 0.f;
    st.m[j][0] = st.m[j][1] = kNoMax;
  }
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

// Causal limits of one segment for this lane: token t is visible to column
// 8j + 2c + e iff t <= lim[j][e] (ctx - T + i; ctx - 1 for single-token
// decode). Padding columns never mask. min_lim is the smallest limit of a real
// column: a page whose last token is at most min_lim needs no mask at all.
template <int NT>
struct SegLimits {
  int lim[NT][2];
  int min_lim;
};

// NP (1 or 2) 16-token pages of one kv head: QK for
// every column tile, one online-softmax update, PV for every tile. The V
// fragments are converted once and shared by all tiles. With two pages the two
// independent chains interleave and hide each other's fixed latencies.
template <int kFmt, int NP, int NT, bool kMulti>
__device__ __forceinline__ void process_pages(WarpState<NT>& st, const PageRegs (&r)[NP],
                                              const uint32_t (&qf)[NT][16], const int (&tok0)[NP],
                                              const int (&nvalid)[NP], const SegLimits<NT>& sl,
                                              float scale_log2, int g, int c) {
  // ---- S^T = K * Q^T : rows tokens (g, g+8), cols 2c, 2c+1 of each tile ----
  float s[NP][NT][4];
#pragma unroll
  for (int pi = 0; pi < NP; ++pi) {
    const uint32_t kr0[8] = {r[pi].ka0.x, r[pi].ka0.y, r[pi].ka0.z, r[pi].ka0.w,
                             r[pi].ka1.x, r[pi].ka1.y, r[pi].ka1.z, r[pi].ka1.w};
    const uint32_t kr1[8] = {r[pi].kb0.x, r[pi].kb0.y, r[pi].kb0.z, r[pi].kb0.w,
                             r[pi].kb1.x, r[pi].kb1.y, r[pi].kb1.z, r[pi].kb1.w};
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) s[pi][j][k] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a0 = KvConv<kFmt>::k_lo(kr0[kk]), a1 = KvConv<kFmt>::k_lo(kr1[kk]);
      const uint32_t a2 = KvConv<kFmt>::k_hi(kr0[kk]), a3 = KvConv<kFmt>::k_hi(kr1[kk]);
#pragma unroll
      for (int j = 0; j < NT; ++j)
        mma_16816(s[pi][j], a0, a1, a2, a3, qf[j][2 * kk], qf[j][2 * kk + 1]);
    }
  }

  // ---- online softmax (log2 domain), one update for all NP pages ----
  float t[NP][NT][4];
  float mx[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) mx[j][0] = mx[j][1] = -INFINITY;
#pragma unroll
  for (int pi = 0; pi < NP; ++pi) {
    const bool masked = tok0[pi] + kBlockSize - 1 > sl.min_lim;
    const int r0 = tok0[pi] + g, r1 = tok0[pi] + g + 8;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int k = 0; k < 4; ++k) t[pi][j][k] = s[pi][j][k] * scale_log2;
      if (!kMulti) {  // one new token: every column's limit is ctx - 1
        if (nvalid[pi] < kBlockSize) {
          if (g >= nvalid[pi]) t[pi][j][0] = t[pi][j][1] = -INFINITY;
          if (g + 8 >= nvalid[pi]) t[pi][j][2] = t[pi][j][3] = -INFINITY;
        }
      } else if (masked) {
        if (r0 > sl.lim[j][0]) t[pi][j][0] = -INFINITY;
        if (r0 > sl.lim[j][1]) t[pi][j][1] = -INFINITY;
        if (r1 > sl.lim[j][0]) t[pi][j][2] = -INFINITY;
        if (r1 > sl.lim[j][1]) t[pi][j][3] = -INFINITY;
      }
      mx[j][0] = fmaxf(mx[j][0], fmaxf(t[pi][j][0], t[pi][j][2]));
      mx[j][1] = fmaxf(mx[j][1], fmaxf(t[pi][j][1], t[pi][j][3]));
    }
  }
  bool need = false;
#pragma unroll
  for (int j = 0; j < NT; ++j)
    need = need || (mx[j][0] > st.m[j][0] + kRescaleThreshold) ||
           (mx[j][1] > st.m[j][1] + kRescaleThreshold);
  if (__any_sync(kFull, need)) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx[j][0] = fmaxf(mx[j][0], __shfl_xor_sync(kFull, mx[j][0], off));
        mx[j][1] = fmaxf(mx[j][1], __shfl_xor_sync(kFull, mx[j][1], off));
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float nm = fmaxf(st.m[j][e], mx[j][e]);
        const float a = ex2(st.m[j][e] - nm);
        st.m[j][e] = nm;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          st.o[j][i][e] *= a;
          st.o[j][i][e + 2] *= a;
        }
        st.l[j][e] *= a;
        st.l[j][e + 2] *= a;
      }
    }
  }

#pragma unroll
  for (int pi = 0; pi < NP; ++pi) {
    // P^T B-fragments per tile: lane (g, c) gets P[tokens 2c, 2c+1 | 2c+8, 2c+9][col g]
    uint32_t pb0[NT], pb1[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float p0 = ex2(t[pi][j][0] - st.m[j][0]), p1 = ex2(t[pi][j][1] - st.m[j][1]);
      const float p2 = ex2(t[pi][j][2] - st.m[j][0]), p3 = ex2(t[pi][j][3] - st.m[j][1]);
      pb0[j] = movmatrix_trans(pack_half2(p0, p1));
      pb1[j] = movmatrix_trans(pack_half2(p2, p3));
    }

    // ---- O^T += V^T * P^T for every tile ----
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
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        mma_16816(st.o[j][2 * u], xy[0], xy[1], zw[0], zw[1], pb0[j], pb1[j]);
        mma_16816(st.o[j][2 * u + 1], xy[2], xy[3], zw[2], zw[3], pb0[j], pb1[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
      mma_16816(st.l[j], kOnesHalf2, kOnesHalf2, kOnesHalf2, kOnesHalf2, pb0[j], pb1[j]);
  }
}

__device__ __forceinline__ void store_half4(__half* o, float a, float b, float c, float d) {
  uint2 v;
  v.x = pack_half2(a, b);
  v.y = pack_half2(c, d);
  *reinterpret_cast<uint2*>(o) = v;
}

// LSE merge of the split segments this CTA completed alone (at most two: the
// first and the last of its range) into fp16 rows, thread: column col, dims
// dq..dq+3 (col is uniform over a warp). Pieces were written by other CTAs:
// read through L2. The bad flags come from the merge tickets (a bad segment
// gets NaN rows whatever its piece count). For segments of at most kFew
// pieces, every piece of both segments is loaded before any is used (one
// round trip for the whole merge). In one-tile kernels a segment of up to
// kWidePieces pieces takes one round trip of its own: lane k loads piece k's
// maximum and sum and the warp shares them by shuffles, so a lane holds only
// its dims of each piece's O (fewer registers, so every load of the batch
// stays in flight). Larger segments are merged by merge_staged. The sums run
// in piece order with the combine kernel's arithmetic (bitwise equal results).
template <bool kWide>  // one round trip for up to kWidePieces pieces (else kFewPieces)
__device__ __forceinline__ void merge_segments(const PartialParams& p, const int (&ms)[2],
                                               const int (&mbad)[2], const int (&milo)[2],
                                               const int (&mihi)[2], int nm, int col, int dq,
                                               float v_scale) {
  if (col >= p.group * p.q_len) return;
  constexpr int kFew = kFewPieces;
  int ilo[2], ihi[2], bad[2];
  float mi[2][kFew], li[2][kFew];
  float4 oi[2][kFew];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j < nm) {
      const int s = ms[j];
      ilo[j] = milo[j];
      ihi[j] = mihi[j];
      if (j == 0) stamp_after(16, ihi[j] - ilo[j]);
      bad[j] = mbad[j];
#pragma unroll
      for (int k = 0; k < kFew; ++k) {
        if (ilo[j] + k <= ihi[j] && ihi[j] - ilo[j] < kFew) {  // larger segments load their own batch
          const float* slot = p.partials + (size_t)(ilo[j] + k + s) * kSlotFloats;
          mi[j][k] = __ldcg(slot + kSlotM + col);
          li[j][k] = __ldcg(slot + kSlotL + col);
          oi[j][k] = __ldcg(reinterpret_cast<const float4*>(slot + col * kHeadDim + dq));
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j >= nm) continue;
    const int s = ms[j];
    __half* o = p.out + col_row(p, s, col) * kHeadDim + dq;
    if (bad[j] != 0) {
      const float nan = __int_as_float(0x7fc00000);
      store_half4(o, nan, nan, nan, nan);
      continue;
    }
    float M = -INFINITY;
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ihi[j] - ilo[j] < kFew) {
#pragma unroll
      for (int k = 0; k < kFew; ++k)
        if (ilo[j] + k <= ihi[j]) M = fmaxf(M, mi[j][k]);
#pragma unroll
      for (int k = 0; k < kFew; ++k) {
        if (ilo[j] + k <= ihi[j]) {
          const float w = (mi[j][k] == -INFINITY) ? 0.f : ex2(mi[j][k] - M);
          L += w * li[j][k];
          acc.x += w * oi[j][k].x;
          acc.y += w * oi[j][k].y;
          acc.z += w * oi[j][k].z;
          acc.w += w * oi[j][k].w;
        }
      }
    } else if (kWide && ihi[j] - ilo[j] < kWidePieces) {  // still one round trip
      // lane k loads piece k's maximum and sum; the warp shares them by shuffles
      const int lane = threadIdx.x & 31, np = ihi[j] - ilo[j] + 1;
      float mk = -INFINITY, lk = 0.f;
      if (lane < np) {
        const float* slot = p.partials + (size_t)(ilo[j] + lane + s) * kSlotFloats;
        mk = __ldcg(slot + kSlotM + col);
        lk = __ldcg(slot + kSlotL + col);
      }
      float4 ob[kWidePieces];
#pragma unroll
      for (int k = 0; k < kWidePieces; ++k)
        if (k < np)
          ob[k] = __ldcg(reinterpret_cast<const float4*>(p.partials + (size_t)(ilo[j] + k + s) * kSlotFloats +
                                                         col * kHeadDim + dq));
      if (j == 0) stamp_after(17, __float_as_int(ob[0].x) ^ __float_as_int(lk));
      float mx = mk;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      M = mx;
      const float wk = (mk == -INFINITY) ? 0.f : ex2(mk - M);
#pragma unroll
      for (int k = 0; k < kWidePieces; ++k) {
        if (k < np) {
          const float w = __shfl_sync(kFull, wk, k), l = __shfl_sync(kFull, lk, k);
          L += w * l;
          acc.x += w * ob[k].x;
          acc.y += w * ob[k].y;
          acc.z += w * ob[k].z;
          acc.w += w * ob[k].w;
        }
      }
    }
    const float rr = (L > 0.f) ? v_scale / L : 0.f;  // a new token with no visible token: 0
    store_half4(o, acc.x * rr, acc.y * rr, acc.z * rr, acc.w * rr);
  }
}

// ---------------------------------------------------------------------------
// The parts of a partial CTA's work that both kernels below share.
// ---------------------------------------------------------------------------

// Static shared state of one partial CTA (the ring, the merge buffers and the
// segment caches live in dynamic shared memory).
template <int NT>
struct CtaShared {
  static constexpr int kBufs = PartialGeom<NT>::kMergeBufs;
  uint64_t full_bar[kStages];  // one per ring slot: the slot's K and V pages landed
  int stage_bad[kStages];      // the slot's page had a block id outside [0, NB)
  int abort_flag;              // a wait ran out of time: stop issuing, drain
  int scan_warp[kWarps], scan_warp_cost[kWarps];
  int scan_carry, scan_carry_cost;
  long long cost_line;  // the line's length, for piece_owners
  int range_lo, range_hi, range_seg, range_seg_hi;  // pages; first, last segment
  // split pieces of this CTA (at most its first and last segment), whose
  // merge tickets are taken once the whole range is done
  int pend_seg[2], pend_poison[2], pend_last[2], pend_bad[2];
  // pieces of segments merged by merge_shared: rank (-1: none; 0: the last
  // piece to arrive) and merging CTAs
  int pend_rank[2], pend_nh[2];
  int arrived[2];  // old arrival counts of the range's first and last segment (-1: none)
  int wait_word;  // the ticket word a helper saw complete (-1: it did not)
  int npend;
  // the range's first and last segment (the only ones a range can share with
  // other CTAs) and the CTAs holding their first and last page
  int own_seg[2], own_ilo[2], own_ihi[2];
  int cta_status;  // first error this CTA met (XQA_OK if none), published at exit
#ifdef XQA_STAMPS
  int first_stamped;
#endif
  // the segment each merge buffer holds, whether this CTA owns it whole, and
  // each warp's "met a bad page" flag for it
  int buf_seg[kBufs], buf_whole[kBufs], buf_poison[kBufs][kWarps];
};

// Dynamic shared memory of a partial CTA: the 1024-byte aligned ring of
// kStages (K, V) page slots, then the merge buffers and the three segment
// caches (segment starts, context lengths, cost-line prefix).
template <int NT>
struct CtaSmem {
  uint8_t* stages;
  float* merge_bufs;
  int32_t* seg_cache;
  int32_t* ctx_cache;
  int32_t* cc_cache;
};

template <int NT>
__device__ __forceinline__ CtaSmem<NT> carve_smem(uint8_t* smem_raw) {
  CtaSmem<NT> m;
  m.stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  m.merge_bufs = reinterpret_cast<float*>(m.stages + kStages * kStageBytes);
  m.seg_cache = reinterpret_cast<int32_t*>(m.merge_bufs +
                                           PartialGeom<NT>::kMergeBufs * PartialGeom<NT>::kMergeBufFloats);
  m.ctx_cache = m.seg_cache + kSegCache;  // context length per sequence
  m.cc_cache = m.ctx_cache + kSegCache;   // cost-line prefix per segment
  return m;
}

// This CTA's range of the flattened (segment, page) order and the tables it
// reads them through. segs / cc / ctxs index by global segment (sequence)
// number even when they point into a shared window of the tables.
struct RangeView {
  const int32_t* segs;  // segment starts
  const int32_t* cc;    // cost-line prefix
  const int32_t* ctxs;  // context lengths
  int total, n;         // pages of the step, CTAs that hold work
  int cbeg, cend, npages;
  int s_first, s_hi;  // the range's first segment, the last any lookup can reach
};

// The plan (computed here when the segment table fits in shared memory, with
// the same integer rule as the planner kernel, else read from the planner),
// the rows of empty segments, and this CTA's range on the cost line. Also
// initialises the ring barriers and waits for the kernels before this one on
// the stream. Returns false when this CTA holds no page.
template <int NT>
__device__ __forceinline__ bool setup_range(const PartialParams& p, const CUtensorMap* tm_k,
                                            const CUtensorMap* tm_v, CtaShared<NT>& sh,
                                            const CtaSmem<NT>& sm, RangeView& rv) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int nseg = p.batch * p.num_kv_heads;
  const int ncols = p.group * p.q_len;
  const bool segs_in_smem = nseg + 1 <= kSegCache;
  const int32_t* segs;
  const int32_t* cc;
  int total, n;
  if (tid == 0) {  // before the wait: nothing here reads or writes global memory
    for (int i = 0; i < kStages; ++i) mbar_init(&sh.full_bar[i], 1);
    sh.abort_flag = 0;
    sh.npend = 0;
    sh.cta_status = XQA_OK;
    sh.scan_carry = sh.scan_carry_cost = 0;
#ifdef XQA_STAMPS
    sh.first_stamped = 0;
#endif
    fence_mbar_init();
    prefetch_tensormap(tm_k);
    prefetch_tensormap(tm_v);
  }
  // Also before the wait, and only a hint: the first pages this CTA index
  // streamed in the previous call (usually the same pages), fetched into L2
  // so that the first loads after the wait find them there. The hint words
  // may be being written by that call; any value is harmless (a row outside
  // the tensor fetches nothing).
  if (p.hints != nullptr && tid < kHintPages) {
    const int y = ld_relaxed_gpu(p.hints + (size_t)cta * kHintPages + tid);
    if (y >= 0) {
      if (p.kv_layout == XQA_LAYOUT_HND) {
        tma_prefetch_2d(tm_k, 0, y);
        tma_prefetch_2d(tm_v, 0, y);
      } else {  // NHD: box (128 dims, 1 kv head, 16 tokens) at (0, kvh, page * 16)
        const int row = y / kBlockSize, id = row / p.num_kv_heads, kvh = row - id * p.num_kv_heads;
        tma_prefetch_3d(tm_k, 0, kvh, id * kBlockSize);
        tma_prefetch_3d(tm_v, 0, kvh, id * kBlockSize);
      }
    }
  }
  // Every input (and the planner's table, when it ran) is read after the
  // kernels before this one on the stream have completed; this kernel may have
  // become resident while they still ran (programmatic dependent launch).
  griddep_wait();
  stamp(1);
  if (cta == 0 && tid == 0) p.header[0] = gridDim.x;  // status words this call writes
  __syncthreads();
  stamp(12);
  if (segs_in_smem) {
    const long long max_ctx = (long long)p.max_blocks_per_seq * kBlockSize;
    for (int base = 0; base < p.batch; base += kThreads) {
      const int b = base + tid;
      int pages = 0;
      if (b < p.batch) {
        const int ctx = __ldg(&p.context_lens[b]);
        if (base == 0) stamp_after(10, ctx);
        sm.ctx_cache[b] = ctx;
        pages = (ctx < 0 || (long long)ctx > max_ctx) ? 0 : (ctx + kBlockSize - 1) / kBlockSize;
      }
      const int cost = seg_cost(pages);  // every kv head's segment of sequence b
      int incl = pages, incl_cost = cost;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(kFull, incl, off);
        const int uc = __shfl_up_sync(kFull, incl_cost, off);
        if (lane >= off) {
          incl += u;
          incl_cost += uc;
        }
      }
      if (lane == 31) {
        sh.scan_warp[warp] = incl;
        sh.scan_warp_cost[warp] = incl_cost;
      }
      __syncthreads();
      int before = sh.scan_carry, before_cost = sh.scan_carry_cost;
      for (int w = 0; w < warp; ++w) {
        before += sh.scan_warp[w];
        before_cost += sh.scan_warp_cost[w];
      }
      const int excl = before + incl - pages;
      const int excl_cost = before_cost + incl_cost - cost;
      if (b < p.batch)
        for (int h = 0; h < p.num_kv_heads; ++h) {
          sm.seg_cache[b * p.num_kv_heads + h] = excl * p.num_kv_heads + h * pages;
          sm.cc_cache[b * p.num_kv_heads + h] = excl_cost * p.num_kv_heads + (h + 1) * cost;
        }
      __syncthreads();
      if (tid == kThreads - 1) {
        sh.scan_carry = excl + pages;
        sh.scan_carry_cost = excl_cost + cost;
      }
      __syncthreads();
    }
    total = sh.scan_carry * p.num_kv_heads;
    if (tid == 0) sm.seg_cache[nseg] = total;
    n = num_ctas_for(total, p.n_max, p.min_pages);
    segs = sm.seg_cache;
    cc = sm.cc_cache;
    if (cta == 0) {  // publish the plan (read back by xqa_read_plan and the combine kernel)
      for (int s = tid; s < nseg; s += kThreads) {
        const int ctx = sm.ctx_cache[s / p.num_kv_heads];
        p.seg_start[s] = sm.seg_cache[s];
        p.seg_cc[s] = sm.cc_cache[s];
        p.seg_bad[s] = (ctx < 0 || (long long)ctx > max_ctx) ? 1 : 0;
      }
      if (tid == 0) {
        p.seg_start[nseg] = total;
        p.header[1] = n;
        p.header[2] = total;
        p.header[3] = nseg;
      }
    }
  } else {
    total = p.header[2];
    n = p.header[1];
    segs = p.seg_start;
    cc = p.seg_cc;
  }
  __syncthreads();

  // ---- rows of empty segments (context length 0, or invalid -> NaN), the
  // segments spread over every warp of every CTA (a few each) ----
  {
    const long long max_ctx = (long long)p.max_blocks_per_seq * kBlockSize;
    for (int s = cta * kWarps + warp; s < nseg; s += gridDim.x * kWarps) {
      if (segs[s] != segs[s + 1]) continue;
      const int ctx = __ldg(&p.context_lens[s / p.num_kv_heads]);
      const bool bad = ctx < 0 || (long long)ctx > max_ctx;
      const float v = bad ? __int_as_float(0x7fc00000) : 0.0f;
      if (bad && lane == 0) record_status(&sh.cta_status, XQA_ERR_CTX_TOO_LONG);
      uint4 val;
      val.x = val.y = val.z = val.w = pack_half2(v, v);
      for (int i = lane; i < ncols * (kHeadDim / 8); i += 32) {
        const int col = i / (kHeadDim / 8), d8 = i - col * (kHeadDim / 8);
        reinterpret_cast<uint4*>(p.out + col_row(p, s, col) * kHeadDim)[d8] = val;
      }
    }
  }
  if (cta >= n) return false;
  stamp(13);
  // This CTA's positions [vlo, vhi) on the cost line, and the pages there: the
  // first page at a position >= a lies in the first segment whose pages end
  // past a. One parallel pass over the segments finds both ends (and the
  // first segment) in shared memory, in place of two dependent searches.
  const long long line = (long long)total + (nseg > 0 ? cc[nseg - 1] : 0);
  long long vlo, vhi;  // floor(cta * line / n), floor((cta + 1) * line / n)
  if (line <= 0xffffffffll) {
    // exact in 32 bits: line = q n + r, so cta line / n = cta q + cta r / n
    // with cta r < n^2 <= 2^20 (a 64-bit division is a long software routine)
    const uint32_t q = (uint32_t)line / (uint32_t)n, r = (uint32_t)line - q * (uint32_t)n;
    vlo = (long long)((uint32_t)cta * q + ((uint32_t)cta * r) / (uint32_t)n);
    vhi = (long long)((uint32_t)(cta + 1) * q + ((uint32_t)(cta + 1) * r) / (uint32_t)n);
  } else {
    vlo = ((long long)cta * line) / n;
    vhi = ((long long)(cta + 1) * line) / n;
  }
  if (tid == 0) {
    sh.cost_line = line;
    sh.range_lo = sh.range_hi = total;  // no segment ends past the position
    sh.range_seg = nseg;
    sh.range_seg_hi = nseg - 1;
  }
  __syncthreads();
  for (int s = tid; s < nseg; s += kThreads) {
    const long long end = (long long)segs[s + 1] + cc[s];                 // past its last page
    const long long prev = s > 0 ? (long long)segs[s] + cc[s - 1] : -1;  // previous one's end
    const long long first = (long long)segs[s] + cc[s];                   // its first page
    if (end > vlo && prev <= vlo) {
      sh.range_lo = vlo <= first ? segs[s] : (int)(segs[s] + (vlo - first));
      sh.range_seg = s;
    }
    if (end > vhi && prev <= vhi) {
      sh.range_hi = vhi <= first ? segs[s] : (int)(segs[s] + (vhi - first));
      sh.range_seg_hi = s;  // the range's last segment is this one or an earlier one
    }
  }
  __syncthreads();
  rv.cbeg = sh.range_lo;
  rv.cend = sh.range_hi;
  rv.npages = rv.cend - rv.cbeg;
  if (rv.npages <= 0) return false;  // its share of the line is segment switch cost only
  rv.s_first = sh.range_seg;
  rv.total = total;
  rv.n = n;
  // With the planner's table in global memory, the few segments this range
  // touches (a contiguous run) are copied into the shared caches, and the
  // table pointers are shifted so that segment s still reads entry s.
  rv.s_hi = nseg - 1;
  rv.ctxs = segs_in_smem ? sm.ctx_cache : p.context_lens;
  if (!segs_in_smem) {
    const int s_first = rv.s_first;
    const int wn = sh.range_seg_hi - s_first + 1;
    const int b_first = s_first / p.num_kv_heads;
    const int wb = sh.range_seg_hi / p.num_kv_heads - b_first + 1;
    if (wn + 1 <= kSegCache && wb <= kSegCache) {
      for (int i = tid; i <= wn; i += kThreads) {
        sm.seg_cache[i] = segs[s_first + i];
        if (i < wn) sm.cc_cache[i] = cc[s_first + i];
      }
      for (int i = tid; i < wb; i += kThreads) sm.ctx_cache[i] = __ldg(&p.context_lens[b_first + i]);
      __syncthreads();
      segs = sm.seg_cache - s_first;
      cc = sm.cc_cache - s_first;
      rv.ctxs = sm.ctx_cache - b_first;
      rv.s_hi = sh.range_seg_hi;
    }
  }
  rv.segs = segs;
  rv.cc = cc;
  stamp(2);
  stamp_count(8, rv.npages);
  stamp_count(9, sh.range_seg_hi - rv.s_first + 1);
  return true;
}

// One thread, once the range's first pages are in flight: the CTAs holding the
// first and the last page of the range's first and last segment (two 64-bit
// divisions each), which the end of the range needs for the merge tickets and
// the final merge and would otherwise compute on its critical path.
template <int NT>
__device__ __forceinline__ void piece_owners(CtaShared<NT>& sh, const RangeView& rv) {
  const long long line = sh.cost_line;
  const int s_last = find_segment(rv.segs, rv.s_first, rv.s_hi + 1, rv.cend - 1);
#pragma unroll 1
  for (int e = 0; e < 2; ++e) {
    const int sg = e == 0 ? rv.s_first : s_last;
    sh.own_seg[e] = sg;
    sh.own_ilo[e] = cta_of_vpos((long long)rv.segs[sg] + rv.cc[sg], line, rv.n);
    sh.own_ihi[e] = cta_of_vpos((long long)rv.segs[sg + 1] - 1 + rv.cc[sg], line, rv.n);
  }
}

// Lane 0 of a warp: the two TMA loads (K and V slice of one page) into ring
// slot `slot`, completing on its barrier; a page with a bad block id is
// flagged instead (the slot's barrier completes without data).
template <int NT>
__device__ __forceinline__ void issue_page(const PartialParams& p, const CUtensorMap* tm_k,
                                           const CUtensorMap* tm_v, CtaShared<NT>& sh,
                                           uint8_t* stages, int slot, int y, int bad, int sg,
                                           uint64_t policy) {
  uint8_t* st = stages + slot * kStageBytes;
  sh.stage_bad[slot] = bad;
  fence_proxy_async_smem();  // this slot's earlier shared reads come before the TMA writes
  if (bad) {
    record_status(&sh.cta_status, XQA_ERR_BAD_BLOCK_ID);
    mbar_arrive(&sh.full_bar[slot]);
  } else {
    mbar_arrive_expect_tx(&sh.full_bar[slot], kStageBytes);
    if (p.kv_layout == XQA_LAYOUT_HND) {
      tma_load_2d(st, tm_k, &sh.full_bar[slot], 0, y, policy);
      tma_load_2d(st + kPageBytes, tm_v, &sh.full_bar[slot], 0, y, policy);
    } else {  // NHD: box (128 dims, 1 kv head, 16 tokens) at (0, kvh, page*16)
      const int kvh = sg - (sg / p.num_kv_heads) * p.num_kv_heads;
      tma_load_3d(st, tm_k, &sh.full_bar[slot], 0, kvh, y, policy);
      tma_load_3d(st + kPageBytes, tm_v, &sh.full_bar[slot], 0, kvh, y, policy);
    }
  }
}

// One or two of a warp's pages (slots slot0 / slot1, ring phases ph0 / ph1):
// wait for them, move them into registers, refill their slots through
// `refill` (called once per page, before the math), then run the attention
// math on the pages whose block ids were good. t0 / t1 are the pages' first
// token within the sequence. A wait that runs out marks the warp's segment
// state poisoned and the CTA aborted.
template <int kFmt, int NT, bool kMulti, typename Refill>
__device__ __forceinline__ void consume_pages(const PartialParams& p, CtaShared<NT>& sh,
                                              const uint8_t* stages, int slot0, uint32_t ph0,
                                              int slot1, uint32_t ph1, bool pair, int t0, int t1,
                                              int ctx, WarpState<NT>& st,
                                              const uint32_t (&qf)[NT][16],
                                              const SegLimits<NT>& sl, float scale_log2, int g,
                                              int c, int lane, int& poisoned, Refill&& refill) {
  volatile int* abort = &sh.abort_flag;
  bool ready = mbar_wait_bounded(&sh.full_bar[slot0], ph0, abort);
  if (pair) ready = ready && mbar_wait_bounded(&sh.full_bar[slot1], ph1, abort);
  if (!__all_sync(kFull, ready)) {  // warp-uniform outcome
    poisoned = 1;
    if (lane == 0) {
      *abort = 1;
      record_status(&sh.cta_status, XQA_ERR_DEVICE_TIMEOUT);
    }
    return;
  }
#ifdef XQA_STAMPS
  if (threadIdx.x == 0 && !sh.first_stamped) {
    sh.first_stamped = 1;
    stamp(3);
  }
#endif
  const uint8_t* stg0 = stages + slot0 * kStageBytes;
  const uint8_t* stg1 = stages + slot1 * kStageBytes;
  const bool bad0 = sh.stage_bad[slot0] != 0, bad1 = pair && sh.stage_bad[slot1] != 0;
  PageRegs regs[2];
  regs[0] = load_page(stg0, stg0 + kPageBytes, g, c);
  if (pair) regs[1] = load_page(stg1, stg1 + kPageBytes, g, c);
  // The pages are in registers: refill their slots with the pages kStages
  // ahead right away (warp-uniform decision), before the math.
  if (!__any_sync(kFull, *abort != 0)) {
    refill();
    if (pair) refill();
  }
  const int nv0 = min(kBlockSize, ctx - t0), nv1 = min(kBlockSize, ctx - t1);
  if (pair && !bad0 && !bad1) {
    const int tk[2] = {t0, t1}, nv[2] = {nv0, nv1};
    process_pages<kFmt, 2, NT, kMulti>(st, regs, qf, tk, nv, sl, scale_log2, g, c);
  } else {
    if (bad0 || bad1) poisoned = 1;
    if (!bad0) {
      const PageRegs one[1] = {regs[0]};
      const int tk[1] = {t0}, nv[1] = {nv0};
      process_pages<kFmt, 1, NT, kMulti>(st, one, qf, tk, nv, sl, scale_log2, g, c);
    }
    if (pair && !bad1) {
      const PageRegs one[1] = {regs[1]};
      const int tk[1] = {t1}, nv[1] = {nv1};
      process_pages<kFmt, 1, NT, kMulti>(st, one, qf, tk, nv, sl, scale_log2, g, c);
    }
  }
}

// Causal limits of segment s's columns for this lane (see SegLimits).
template <int NT>
__device__ __forceinline__ SegLimits<NT> seg_limits(const PartialParams& p, int ctx, int ncols,
                                                    int c) {
  SegLimits<NT> sl;
  sl.min_lim = ctx - p.q_len;  // the first new token's last visible token
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = 8 * j + 2 * c + e;
      sl.lim[j][e] = col < ncols ? ctx - p.q_len + col / p.group : 0x7fffffff;
    }
  return sl;
}

// Merge of one buffered segment by all threads (column col, dims dq..dq+3):
// the 8 warps' (m, l, O) combine in shared memory; a segment owned whole is
// normalised and written as fp16, a split piece goes to partial slot cta + s.
template <int NT>
__device__ __forceinline__ void merge_buffer(const PartialParams& p, CtaShared<NT>& sh,
                                             const float* merge_bufs, int mb, int ncols,
                                             float v_scale) {
  using Geom = PartialGeom<NT>;
  constexpr int kCols = Geom::kCols;
  const int tid = threadIdx.x;
  const int ms = sh.buf_seg[mb];
  const bool mwhole = sh.buf_whole[mb] != 0;
  int any_poison = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) any_poison |= sh.buf_poison[mb][w];
  const float* base = merge_bufs + mb * Geom::kMergeBufFloats;
  const float* bm = base + Geom::kScratchFloats;
  const float* bl = bm + kWarps * kCols;
  const int dq = (tid & 31) * 4;  // 0..124
#pragma unroll
  for (int col = tid >> 5; col < kCols; col += kWarps) {
    if (col >= ncols) break;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, bm[w * kCols + col]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = bm[w * kCols + col];
      const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      L += sc * bl[w * kCols + col];
      const float4 v =
          *reinterpret_cast<const float4*>(base + (w * kCols + col) * kScratchStride + dq);
      acc.x += sc * v.x;
      acc.y += sc * v.y;
      acc.z += sc * v.z;
      acc.w += sc * v.w;
    }
    if (mwhole) {
      __half* o = p.out + col_row(p, ms, col) * kHeadDim + dq;
      if (any_poison) {
        const float nan = __int_as_float(0x7fc00000);
        store_half4(o, nan, nan, nan, nan);
      } else {
        const float rr = (L > 0.f) ? v_scale / L : 0.f;
        store_half4(o, acc.x * rr, acc.y * rr, acc.z * rr, acc.w * rr);
      }
    } else {
      float* slotp = p.partials + (size_t)(blockIdx.x + ms) * kSlotFloats;
      *reinterpret_cast<float4*>(slotp + col * kHeadDim + dq) = acc;
      if (dq == 0) {
        slotp[kSlotM + col] = M;
        slotp[kSlotL + col] = L;
      }
    }
  }
  if (!mwhole && tid == 0) {  // a split piece: its ticket is taken after the range
    sh.pend_seg[sh.npend] = ms;
    sh.pend_poison[sh.npend] = any_poison;
    ++sh.npend;
  }
}

// CTA mode: warp w takes the CTA-local pages w, w + 8, w + 16, ... of the
// range (two at a time), keeping kLookahead of them in flight; at the end of
// each segment every warp hands its (m, l, O) to a merge buffer, merged across
// warps when the buffer is next reused or at the end of the range.
template <int kFmt, int NT, bool kMulti>
__device__ __forceinline__ void cta_mode_range(const PartialParams& p, const CUtensorMap* tm_k,
                                               const CUtensorMap* tm_v, CtaShared<NT>& sh,
                                               const CtaSmem<NT>& sm, const RangeView& rv,
                                               float scale_log2, float v_scale, uint64_t policy,
                                               WarpState<NT>& st, uint32_t (&qf)[NT][16],
                                               uint32_t (&qf_next)[NT][16], int& q_next_seg,
                                               int& issued, int& kseg) {
  using Geom = PartialGeom<NT>;
  constexpr int kCols = Geom::kCols;
  constexpr int kBufs = Geom::kMergeBufs;
  constexpr bool kPrefetchQ = NT == 1;  // registers: two-tile kernels load Q per segment
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ncols = p.group * p.q_len;
  const int32_t* segs = rv.segs;
  const int cbeg = rv.cbeg, cend = rv.cend, npages = rv.npages;
  const int s_first = rv.s_first, s_hi = rv.s_hi;

  // ---- this warp's loads: owned page k is CTA-local page warp + 8k ----
  const int owned = npages > warp ? (npages - warp + kWarps - 1) / kWarps : 0;
  stamp(14);
  PageBatch cur = load_batch(p, segs, s_first, s_hi + 1, cbeg, npages, warp, 0, lane);
  PageBatch nxt = load_batch(p, segs, s_first, s_hi + 1, cbeg, npages, warp, 32, lane);
  stamp_after(11, cur.y ^ nxt.y);
  if (p.hints != nullptr && lane < 2) {  // this warp's first pair, for the next call's prefetch
    const int row = p.kv_layout == XQA_LAYOUT_HND
                        ? cur.y
                        : (cur.y / kBlockSize * p.num_kv_heads + cur.seg % p.num_kv_heads) * kBlockSize;
    p.hints[(size_t)blockIdx.x * kHintPages + 2 * warp + lane] = lane < owned && !cur.bad ? row : -1;
  }
  int cur_base = 0;
  auto issue_next = [&]() {
    if (issued >= owned) return;
    const int k = issued++;
    if (k >= cur_base + 32) {
      cur = nxt;
      cur_base += 32;
      nxt = load_batch(p, segs, s_first, s_hi + 1, cbeg, npages, warp, cur_base + 32, lane);
    }
    const int y = __shfl_sync(kFull, cur.y, k - cur_base);
    const int bad = __shfl_sync(kFull, cur.bad, k - cur_base);
    const int sg = __shfl_sync(kFull, cur.seg, k - cur_base);
    const int slot = (warp + kWarps * k) % kStages;
    __syncwarp();  // all lanes' reads of this slot's previous page are done
    if (lane == 0) issue_page<NT>(p, tm_k, tm_v, sh, sm.stages, slot, y, bad, sg, policy);
    __syncwarp();
  };
#pragma unroll 1
  for (int i = 0; i < kLookahead; ++i) issue_next();
  if (warp == kWarps - 1 && lane == 0) piece_owners<NT>(sh, rv);

  int s = s_first;
  int q0 = 0;
  while (q0 < npages) {
    while (segs[s + 1] <= cbeg + q0) ++s;
    const int sb = segs[s], se = segs[s + 1];
    const int qe = min(se, cend) - cbeg;
    const int b = s / p.num_kv_heads;
    // from shared memory (the whole table, or this range's window of it): no
    // global round trip at a segment switch
    const int ctx = rv.ctxs[b];
    const bool whole = (sb >= cbeg) && (se <= cend);
    if (kPrefetchQ && q_next_seg == s) {
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < 16; ++i) qf[j][i] = qf_next[j][i];
    } else {
      load_q<NT>(p, s, g, c, qf);
    }
    if (kPrefetchQ && qe < npages) {  // prefetch Q of the next segment this CTA works on
      q_next_seg = find_segment(segs, s, s_hi + 1, cbeg + qe);
      load_q<NT>(p, q_next_seg, g, c, qf_next);
    }
    const SegLimits<NT> sl = seg_limits<NT>(p, ctx, ncols, c);
    reset_state<NT>(st);
    int poisoned = 0;

    // this warp's pages of the segment (q, and q + kWarps when pairing)
    for (int q = q0 + ((warp - q0 % kWarps) + kWarps) % kWarps; q < qe; q += 2 * kWarps) {
      const bool pair = q + kWarps < qe;
      const int j0 = cbeg + q - sb;  // page index within the sequence
      consume_pages<kFmt, NT, kMulti>(p, sh, sm.stages, q % kStages, (q / kStages) & 1,
                                      (q + kWarps) % kStages, ((q + kWarps) / kStages) & 1, pair,
                                      j0 * kBlockSize, (j0 + kWarps) * kBlockSize, ctx, st, qf,
                                      sl, scale_log2, g, c, lane, poisoned, issue_next);
    }

    // ---- hand this segment's per-warp state to a merge buffer; a CTA-wide
    // barrier only when the buffer still holds an unmerged segment (with two
    // buffers a range of at most two segments never stops mid-way) ----
    const int buf = kseg % kBufs;
    if (kseg >= kBufs) {
      consumer_bar();
      merge_buffer<NT>(p, sh, sm.merge_bufs, buf, ncols, v_scale);
      consumer_bar();
    }
    {
      float* base = sm.merge_bufs + buf * Geom::kMergeBufFloats;
      float* bm = base + Geom::kScratchFloats;
      float* bl = bm + kWarps * kCols;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float* my = base + (warp * kCols + 8 * j) * kScratchStride;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d0 = 16 * g + 2 * i;
          my[(2 * c) * kScratchStride + d0] = st.o[j][i][0];
          my[(2 * c + 1) * kScratchStride + d0] = st.o[j][i][1];
          my[(2 * c) * kScratchStride + d0 + 1] = st.o[j][i][2];
          my[(2 * c + 1) * kScratchStride + d0 + 1] = st.o[j][i][3];
        }
        if (g == 0) {
          bm[warp * kCols + 8 * j + 2 * c] = st.m[j][0];
          bm[warp * kCols + 8 * j + 2 * c + 1] = st.m[j][1];
          bl[warp * kCols + 8 * j + 2 * c] = st.l[j][0];
          bl[warp * kCols + 8 * j + 2 * c + 1] = st.l[j][1];
        }
      }
      if (lane == 0) sh.buf_poison[buf][warp] = poisoned;
      if (tid == 0) {
        sh.buf_seg[buf] = s;
        sh.buf_whole[buf] = whole ? 1 : 0;
      }
    }
    ++kseg;
    q0 = qe;
    ++s;
  }
}

// Merge of the rows row0, row0 + rstride, ... (< G * q_len) of a good split
// segment too large for merge_segments, by every thread of the CTA. The
// pieces' rows and their (m, l) words are gathered into shared memory (the
// page ring and the merge buffers, free once the range is done) by all 256
// threads, kGatherLoads 16-byte loads in flight per thread, as many pieces per
// batch as fit; then warp w sums the CTA's rows w and w + kWarps over the
// pieces (lane: dims 4 * lane .. 4 * lane + 3). Each warp reads every
// piece's maximum for its row with lane-parallel loads issued with the first
// gather. The sums run in piece order with the combine kernel's arithmetic
// (bitwise equal results).
template <int NT>
__device__ __forceinline__ void merge_staged(const PartialParams& p, uint8_t* stage, int s,
                                             int ilo, int ihi, int row0, int rstride,
                                             float v_scale) {
  constexpr int kCap = kStages * kStageBytes +
                       PartialGeom<NT>::kMergeBufs * PartialGeom<NT>::kMergeBufFloats * 4;
  constexpr int kGatherLoads = 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, dq = lane * 4;
  const int ncols = p.group * p.q_len;
  const int nrows = (ncols - row0 + rstride - 1) / rstride;  // rows of this CTA (>= 1)
  const int np = ihi - ilo + 1;
  const int per = kCap / (nrows * (kHeadDim * 4 + 8));  // pieces per batch
  const float* first = p.partials + (size_t)(ilo + s) * kSlotFloats;
  stamp_after(16, np);
  float M[NT], L[NT];
  float4 acc[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    M[j] = -INFINITY;
    L[j] = 0.f;
    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int b0 = 0; b0 < np; b0 += per) {
    const int nb = min(per, np - b0);
    const int nchunks = nb * nrows * (kHeadDim / 4);  // 16-byte chunks: (piece, row, dims)
    float* ml = reinterpret_cast<float*>(stage + (size_t)nchunks * 16);  // (piece, row): m, l
    if (b0 > 0) __syncthreads();  // every warp is done with the previous batch
    for (int rp = tid; rp < nb * nrows; rp += kThreads) {  // (piece, row) pairs
      const int k = rp / nrows, i = rp - k * nrows;
      const float* slot = first + (size_t)(b0 + k) * kSlotFloats;
      ml[2 * rp] = __ldcg(slot + kSlotM + row0 + i * rstride);
      ml[2 * rp + 1] = __ldcg(slot + kSlotL + row0 + i * rstride);
    }
    if (b0 == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {  // the maximum over every piece, for this warp's row
        const int i = warp + kWarps * j, col = row0 + i * rstride;
        float mx = -INFINITY;
        if (i < nrows) {
          for (int base = 0; base < np; base += 128) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = base + 32 * u + lane;
              v[u] = k < np ? __ldcg(first + (size_t)k * kSlotFloats + kSlotM + col) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) mx = fmaxf(mx, v[u]);
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        }
        M[j] = mx;
      }
    }
    for (int c0 = 0; c0 < nchunks; c0 += kThreads * kGatherLoads) {
      float4 v[kGatherLoads];
#pragma unroll
      for (int u = 0; u < kGatherLoads; ++u) {
        const int c = c0 + u * kThreads + tid;
        if (c < nchunks) {
          const int rp = c >> 5, k = rp / nrows, i = rp - k * nrows;
          v[u] = __ldcg(reinterpret_cast<const float4*>(
              first + (size_t)(b0 + k) * kSlotFloats + (row0 + i * rstride) * kHeadDim + (c & 31) * 4));
        }
      }
#pragma unroll
      for (int u = 0; u < kGatherLoads; ++u) {
        const int c = c0 + u * kThreads + tid;
        if (c < nchunks) reinterpret_cast<float4*>(stage)[c] = v[u];
      }
    }
    __syncthreads();
    if (b0 == 0) stamp(17);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int i = warp + kWarps * j;
      if (i >= nrows) continue;
#pragma unroll 4
      for (int k = 0; k < nb; ++k) {
        const int rp = k * nrows + i;
        const float mk = ml[2 * rp], lk = ml[2 * rp + 1];
        const float4 o = reinterpret_cast<const float4*>(stage)[rp * 32 + lane];
        const float w = (mk == -INFINITY) ? 0.f : ex2(mk - M[j]);
        L[j] += w * lk;
        acc[j].x += w * o.x;
        acc[j].y += w * o.y;
        acc[j].z += w * o.z;
        acc[j].w += w * o.w;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int i = warp + kWarps * j, col = row0 + i * rstride;
    if (i >= nrows) continue;
    const float rr = (L[j] > 0.f) ? v_scale / L[j] : 0.f;  // a new token with no visible token: 0
    store_half4(p.out + col_row(p, s, col) * kHeadDim + dq, acc[j].x * rr, acc[j].y * rr,
                acc[j].z * rr, acc[j].w * rr);
  }
}

// The final merges this CTA takes part in for segments of more than kAlone
// pieces (at most two: its range's first and last segment), shared by each
// segment's last nh pieces to arrive: the piece of rank r (0 = the last)
// takes the rows r, r + nh, ... once every piece is written (acquire through
// the written count). The segments this CTA completes come first, then those
// it helps with. Each merging CTA adds kTicketRelease to the arrival word
// once it has seen every piece written; the one that brings the releases to
// nh (or the last piece, when it merges alone) clears both words for the next
// call. A CTA that aborted (its ring may still receive page copies) writes
// NaN rows instead. Out of line: the code of the page loop does not depend
// on it.
template <int NT>
__device__ __noinline__ void merge_shared(const PartialParams& p, CtaShared<NT>& sh,
                                          uint8_t* stage, float v_scale) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int ncols = p.group * p.q_len;
  const int npend = sh.npend;
  const bool aborted = sh.abort_flag != 0;  // uniform: set only before the ticket barrier
  for (int n = 0; n < 2 * npend; ++n) {
    const int i = n % npend, rank = sh.pend_rank[i], s = sh.pend_seg[i];
    if (rank < 0 || (rank == 0) != (n < npend)) continue;
    const int e = s == sh.own_seg[0] ? 0 : 1;
    const int ilo = sh.own_ilo[e], ihi = sh.own_ihi[e], nh = sh.pend_nh[i];
    int32_t* written = p.tickets + kMaxCtas + ilo;
    if (tid == 0) sh.wait_word = wait_ticket_count(written, ihi - ilo + 1);
    __syncthreads();
    const int word = sh.wait_word;
    const bool seen = word >= 0;  // -1: the pieces were not all written in time
    int rel_old = 0;
    if (nh > 1 && seen && tid == 0) rel_old = atomicAdd(&p.tickets[ilo], kTicketRelease);
    if (!seen && tid == 0) record_status(&sh.cta_status, XQA_ERR_DEVICE_TIMEOUT);
    if (seen && (word & kTicketPoisonMask) == 0 && !aborted) {
      merge_staged<NT>(p, stage, s, ilo, ihi, rank, nh, v_scale);
    } else {
      for (int col = rank + nh * warp; col < ncols; col += nh * kWarps) {
        const float nan = __int_as_float(0x7fc00000);
        store_half4(p.out + col_row(p, s, col) * kHeadDim + (tid & 31) * 4, nan, nan, nan, nan);
      }
    }
    if (seen && tid == 0 && (nh == 1 || rel_old / kTicketRelease == nh - 1)) {
      p.tickets[ilo] = 0;
      *written = 0;
    }
    __syncthreads();  // the gathered rows and wait_word are read before they are written again
  }
}

// End of a CTA's range: the merges still buffered (the range's last kBufs
// segments, in order), then for each split piece (at most two: the range's
// first and last segment) its merge tickets, and the final merges this CTA
// takes part in (all pieces in slot order, exactly as the combine kernel
// would). The tickets are device-wide atomic round trips taken once per piece
// after the whole range, so no mid-range segment boundary stalls the CTA on
// them. Last, after an abort, the copies still in flight are waited for.
template <int NT>
__device__ __forceinline__ void finish_range(const PartialParams& p, CtaShared<NT>& sh,
                                             const CtaSmem<NT>& sm, const RangeView& rv,
                                             float v_scale, int issued, int kseg) {
  constexpr int kCols = PartialGeom<NT>::kCols;
  constexpr int kBufs = PartialGeom<NT>::kMergeBufs;
  constexpr int kAlone = NT == 1 ? kWidePieces : kFewPieces;  // pieces the last merges alone
  const int tid = threadIdx.x, warp = tid >> 5;
  const int ncols = p.group * p.q_len;
  consumer_bar();
  stamp(4);
  // In-kernel merge: the arrival tickets of the range's split segments (its
  // first and last; thread e takes segment e) that are merged by arrival
  // order (see below) are taken now, so that their round trip overlaps the
  // merges of the buffered segments.
  int arrived = -1;  // -1: merged by the piece written last (no arrival ticket)
  if (p.fused_merge && tid < 2 && (tid == 0 || sh.own_seg[1] != sh.own_seg[0]) &&
      sh.own_ilo[tid] != sh.own_ihi[tid]) {
    const int sg = sh.own_seg[tid], np = sh.own_ihi[tid] - sh.own_ilo[tid] + 1;
    if (np > kAlone ||
        (np <= kArriveFirstPieces && rv.segs[sg + 1] - rv.segs[sg] >= kArriveFirstPages))
      arrived = atomicAdd(&p.tickets[sh.own_ilo[tid]], 1);
  }
  for (int k = kseg > kBufs ? kseg - kBufs : 0; k < kseg; ++k)
    merge_buffer<NT>(p, sh, sm.merge_bufs, k % kBufs, ncols, v_scale);
  if (tid < 2) sh.arrived[tid] = arrived;
  consumer_bar();
  stamp(5);

  const int npend = sh.npend;
  if (npend > 0) {
    consumer_bar();  // all of this CTA's partial-slot writes precede the written counts
    if (tid < npend) {
      // A split segment's tickets are the words of the CTA holding its first
      // page (unique in a call). Each piece raises the written count by 1,
      // plus kTicketPoison if it met a bad page, with release order after its
      // slot. In-kernel merge, by the piece count:
      //  * at most kArriveFirstPieces, of a segment of at least
      //    kArriveFirstPages pages: the last piece to arrive (arrival rank 0)
      //    merges alone once
      //    every other piece is written (acquire through the written count;
      //    it does not raise it), then clears both words;
      //  * other segments of up to kAlone pieces: the piece that completes
      //    the written count (its atomic returns the count and the bad
      //    flags) merges alone and clears both words (their pieces finish
      //    close together: the last to arrive would often wait for another's
      //    slot);
      //  * more: merge_shared, by the last nh pieces to arrive.
      // Combine kernel: the first word takes the written counts; the combine
      // kernel reads and clears it.
      const int ps = sh.pend_seg[tid];
      const int e = ps == sh.own_seg[0] ? 0 : 1;  // a split piece is the range's first or last
      const int ilo = sh.own_ilo[e], ihi = sh.own_ihi[e], np = ihi - ilo + 1;
      const int add = 1 + (sh.pend_poison[tid] ? kTicketPoison : 0);
      int32_t* written = p.tickets + kMaxCtas + ilo;
      int last = 0, bad = 0, rank = -1;
      if (p.fused_merge) {
        const int r = np - 1 - (sh.arrived[e] & kTicketCountMask);
        if (np > kAlone) {
          const int nh = max(1, min(min(np / 2, ncols), p.merge_helpers));
          if (r < nh) rank = r;
          red_add_release_gpu(written, add);
          sh.pend_nh[tid] = nh;
        } else if (sh.arrived[e] < 0) {
          const int old = atom_add_acq_rel_gpu(written, add);
          if ((old & kTicketCountMask) == np - 1) {
            last = 1;
            bad = ((old & kTicketPoisonMask) != 0 || add > 1) ? 1 : 0;
            *written = 0;  // (the arrival word is not used for these segments)
          }
        } else if (r == 0) {
          const int w = wait_ticket_count(written, np - 1);  // the other pieces' slots
          last = 1;
          bad = (w < 0 || (w & kTicketPoisonMask) != 0 || add > 1) ? 1 : 0;
          if (w < 0) {
            record_status(&sh.cta_status, XQA_ERR_DEVICE_TIMEOUT);
          } else {
            p.tickets[ilo] = 0;
            *written = 0;
          }
        } else {
          red_add_release_gpu(written, add);
        }
      } else {
        red_add_release_gpu(&p.tickets[ilo], add);  // the combine kernel reads and clears it
      }
      sh.pend_last[tid] = last;
      sh.pend_bad[tid] = bad;
      sh.pend_rank[tid] = rank;
    }
    consumer_bar();
    stamp(6);
    int m0 = 0, m1 = 0, b0 = 0, b1 = 0, nm = 0;  // the segments this CTA completes alone
    for (int i = 0; i < npend; ++i) {
      if (!sh.pend_last[i]) continue;
      if (nm == 0) {
        m0 = sh.pend_seg[i];
        b0 = sh.pend_bad[i];
      } else {
        m1 = sh.pend_seg[i];
        b1 = sh.pend_bad[i];
      }
      ++nm;
    }
    const int ms[2] = {m0, m1}, mbad[2] = {b0, b1};
    const int e0 = m0 == sh.own_seg[0] ? 0 : 1, e1 = m1 == sh.own_seg[0] ? 0 : 1;
    const int milo[2] = {sh.own_ilo[e0], sh.own_ilo[e1]}, mihi[2] = {sh.own_ihi[e0], sh.own_ihi[e1]};
    if (nm > 0)
      for (int col = tid >> 5; col < kCols; col += kWarps)
        merge_segments<NT == 1>(p, ms, mbad, milo, mihi, nm, col, (tid & 31) * 4, v_scale);
    if (sh.pend_rank[0] >= 0 || (npend > 1 && sh.pend_rank[1] >= 0)) {
      __syncthreads();  // the merge buffers and every warp's last pages are read
      merge_shared<NT>(p, sh, sm.stages, v_scale);
    }
  }

  // Drain: after an abort some issued copies may not have been waited for.
  // Each is waited for once more, with the same time budget. A copy that
  // still has not landed after that may land in this SM's shared memory after
  // the CTA exits: the CTA then records XQA_ERR_DRAIN_TIMEOUT (in place of the
  // timeout), which says that the device state is not to be trusted.
  if (sh.abort_flag) {
    int never = 0;
    volatile int* no_abort = &never;
    // only the last kLookahead issued pages can still be in flight: every
    // earlier one was waited for before its slot was reissued
    const int first = issued > kLookahead ? issued - kLookahead : 0;
    for (int k = first; k < issued; ++k) {
      const int q = warp + kWarps * k;
      const bool ok = mbar_wait_bounded(&sh.full_bar[q % kStages], (q / kStages) & 1, no_abort);
      if (!__all_sync(kFull, ok)) {
        if ((threadIdx.x & 31) == 0) atomicExch(&sh.cta_status, XQA_ERR_DRAIN_TIMEOUT);
        break;
      }
    }
  }
}

// Every CTA of the launch writes its status word once, at exit (the words of
// one call need no reset: the next call overwrites all it reads).
template <int NT>
__device__ __forceinline__ void publish_status(const PartialParams& p, CtaShared<NT>& sh) {
  __syncthreads();
  stamp(7);
  if (threadIdx.x == 0) p.status[blockIdx.x] = sh.cta_status;
}

}  // namespace

template <int kFmt, int NT, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) CtaShared<NT> sh;
  griddep_launch_dependents();  // a dependent next kernel waits for this grid itself
  stamp(0);
  const CtaSmem<NT> sm = carve_smem<NT>(smem_raw);
  RangeView rv;
  if (!setup_range<NT>(p, &tm_k, &tm_v, sh, sm, rv)) {
    publish_status<NT>(p, sh);
    return;
  }
  // per-tensor scales: host values, or device scalars read when the kernel
  // runs (after the wait in setup_range, like every input)
  const float k_scale = p.k_scale_ptr ? __ldg(p.k_scale_ptr) : p.k_scale;
  const float v_scale = p.v_scale_ptr ? __ldg(p.v_scale_ptr) : p.v_scale;
  const float scale_log2 = static_cast<float>(p.qk_scale_base * static_cast<double>(k_scale));
  const uint64_t policy = l2_evict_first_policy();

  WarpState<NT> st;
  uint32_t qf[NT][16], qf_next[NT][16];
  int q_next_seg = -1;
  int issued = 0;  // this warp's pages whose loads have been issued
  int kseg = 0;    // segments of this range handed to the merge buffers
  cta_mode_range<kFmt, NT, kMulti>(p, &tm_k, &tm_v, sh, sm, rv, scale_log2, v_scale, policy, st, qf,
                                   qf_next, q_next_seg, issued, kseg);
  finish_range<NT>(p, sh, sm, rv, v_scale, issued, kseg);
  publish_status<NT>(p, sh);
}

// The same kernel with a second way to work a range (warp mode): when the
// range touches at least kWarpModeMinPieces segment pieces of at most
// kWarpModePages pages each, whole pieces go to single warps (round-robin over
// the range's segments, a static rule), each warp accumulates its piece alone
// and writes it from registers, with no merge across warps and no CTA barrier
// per segment; other ranges are worked in CTA mode as above. Launched only for
// shapes with many segments per CTA (batches of many short sequences): the
// mode test and the warp-mode code slow the page loop of CTA-mode ranges.
template <int kFmt, int NT, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1)
    partial_kernel_wm(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const PartialParams p) {
  static_assert(NT == 1, "warp mode holds one column tile");
  constexpr bool kPrefetchQ = true;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) CtaShared<NT> sh;
  griddep_launch_dependents();  // a dependent next kernel waits for this grid itself
  stamp(0);
  const int ncols = p.group * p.q_len;
  const CtaSmem<NT> sm = carve_smem<NT>(smem_raw);
  RangeView rv;
  if (!setup_range<NT>(p, &tm_k, &tm_v, sh, sm, rv)) {
    publish_status<NT>(p, sh);
    return;
  }
  const float k_scale = p.k_scale_ptr ? __ldg(p.k_scale_ptr) : p.k_scale;
  const float v_scale = p.v_scale_ptr ? __ldg(p.v_scale_ptr) : p.v_scale;
  const float scale_log2 = static_cast<float>(p.qk_scale_base * static_cast<double>(k_scale));
  const uint64_t policy = l2_evict_first_policy();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int cta = blockIdx.x;
  const int32_t* segs = rv.segs;
  const int cbeg = rv.cbeg, cend = rv.cend;
  const int s_first = rv.s_first;

  WarpState<NT> st;
  uint32_t qf[NT][16], qf_next[NT][16];
  int q_next_seg = -1;
  int issued = 0;  // this warp's pages whose loads have been issued
  int kseg = 0;    // pieces handed to the merge buffers

  // ---- mode: at least kWarpModeMinPieces pieces, none longer than
  // kWarpModePages pages -> warp mode; otherwise CTA mode ----
  const int nsr = find_segment(segs, s_first, rv.s_hi + 1, cend - 1) - s_first + 1;  // segments touched
  bool warp_mode = false;
  if (nsr >= kWarpModeMinPieces && nsr <= kThreads) {
    int len = 0;
    if (tid < nsr) len = min(segs[s_first + tid + 1], cend) - max(segs[s_first + tid], cbeg);
    const int pieces = __syncthreads_count(len > 0);
    const int too_long = __syncthreads_or(len > kWarpModePages);
    warp_mode = pieces >= kWarpModeMinPieces && !too_long;
  }

  if (!warp_mode) {
    cta_mode_range<kFmt, NT, kMulti>(p, &tm_k, &tm_v, sh, sm, rv, scale_log2, v_scale, policy, st,
                                     qf, qf_next, q_next_seg, issued, kseg);
  } else {
    // ---- warp mode: this warp's pieces are the range's segments j = warp,
    // warp + 8, ... (j counted from s_first; empty ones skipped). A piece's
    // block ids are fetched one per lane; the next piece's when the current
    // one starts issuing.
    auto piece = [&](int j, int& pb, int& len) {
      const int sg = s_first + j;
      pb = max(segs[sg], cbeg);
      len = min(segs[sg + 1], cend) - pb;
    };
    auto next_piece = [&](int j) {  // the first non-empty piece among j, j + 8, ...
      for (; j < nsr; j += kWarps) {
        int pb, len;
        piece(j, pb, len);
        if (len > 0) break;
      }
      return j;
    };
    auto fetch = [&](int j) {
      PageBatch r{0, 0, 0};
      if (j < nsr) {
        int pb, len;
        piece(j, pb, len);
        const int sg = s_first + j;
        r.seg = sg;
        if (lane < len) {
          const int bb = sg / p.num_kv_heads, kvh = sg - bb * p.num_kv_heads;
          const int id =
              __ldg(&p.block_tables[(size_t)bb * p.max_blocks_per_seq + (pb + lane - segs[sg])]);
          r.bad = (id < 0 || id >= p.num_blocks) ? 1 : 0;
          r.y = r.bad ? 0
                      : (p.kv_layout == XQA_LAYOUT_HND ? (id * p.num_kv_heads + kvh) : id) * kBlockSize;
        }
      }
      return r;
    };
    int ij = next_piece(warp), ioff = 0;  // the piece being issued, its next page
    int ij_next = next_piece(ij + kWarps);
    PageBatch wcur = fetch(ij), wnxt = fetch(ij_next);
    auto issue_next_w = [&]() {
      while (ij < nsr) {
        int pb, len;
        piece(ij, pb, len);
        if (ioff < len) {
          const int y = __shfl_sync(kFull, wcur.y, ioff);
          const int bad = __shfl_sync(kFull, wcur.bad, ioff);
          ++ioff;
          const int k = issued++;
          const int slot = (warp + kWarps * k) % kStages;
          __syncwarp();  // all lanes' reads of this slot's previous page are done
          if (lane == 0) issue_page<NT>(p, &tm_k, &tm_v, sh, sm.stages, slot, y, bad, wcur.seg, policy);
          __syncwarp();
          return;
        }
        ij = ij_next;
        ioff = 0;
        wcur = wnxt;
        ij_next = next_piece(ij + kWarps);
        wnxt = fetch(ij_next);
      }
    };
#pragma unroll 1
    for (int i = 0; i < kLookahead; ++i) issue_next_w();
    if (warp == kWarps - 1 && lane == 0) piece_owners<NT>(sh, rv);

    int k = 0;  // this warp's running page index (ring slot and phase)
    for (int j = next_piece(warp); j < nsr; j = next_piece(j + kWarps)) {
      const int s = s_first + j;
      int pb, len;
      piece(j, pb, len);
      const int sb = segs[s], se = segs[s + 1];
      const bool whole = (sb >= cbeg) && (se <= cend);
      const int ctx = rv.ctxs[s / p.num_kv_heads];
      if (kPrefetchQ && q_next_seg == s) {
#pragma unroll
        for (int i = 0; i < 16; ++i) qf[0][i] = qf_next[0][i];
      } else {
        load_q<NT>(p, s, g, c, qf);
      }
      if (kPrefetchQ) {  // Q of this warp's next piece
        const int jn = next_piece(j + kWarps);
        if (jn < nsr) {
          q_next_seg = s_first + jn;
          load_q<NT>(p, q_next_seg, g, c, qf_next);
        }
      }
      const SegLimits<NT> sl = seg_limits<NT>(p, ctx, ncols, c);
      reset_state<NT>(st);
      int poisoned = 0;
      for (int o = 0; o < len; o += 2) {
        const bool pair = o + 1 < len;
        const int t0 = (pb + o - sb) * kBlockSize;
        consume_pages<kFmt, NT, kMulti>(p, sh, sm.stages, (warp + kWarps * k) % kStages,
                                        (k / kLookahead) & 1, (warp + kWarps * (k + 1)) % kStages,
                                        ((k + 1) / kLookahead) & 1, pair, t0, t0 + kBlockSize, ctx,
                                        st, qf, sl, scale_log2, g, c, lane, poisoned, issue_next_w);
        k += pair ? 2 : 1;
      }
      // ---- the piece's (m, l, O) straight from this warp's registers: lane
      // (g, c) holds dims 16g + 2i (+1) of columns 2c, 2c + 1 ----
      const float nan = __int_as_float(0x7fc00000);
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int col = 2 * c + e2;
        if (col >= ncols) continue;
        if (whole) {
          __half* orow = p.out + col_row(p, s, col) * kHeadDim;
          const float l = st.l[0][e2];
          const float rr = poisoned ? nan : ((l > 0.f) ? v_scale / l : 0.f);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int d0 = 16 * g + 2 * i;
            *reinterpret_cast<uint32_t*>(orow + d0) =
                pack_half2(st.o[0][i][e2] * rr, st.o[0][i][e2 + 2] * rr);
          }
        } else {
          float* slotp = p.partials + (size_t)(cta + s) * kSlotFloats;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int d0 = 16 * g + 2 * i;
            *reinterpret_cast<float2*>(slotp + col * kHeadDim + d0) =
                make_float2(st.o[0][i][e2], st.o[0][i][e2 + 2]);
          }
          if (g == 0) {
            slotp[kSlotM + col] = st.m[0][e2];
            slotp[kSlotL + col] = st.l[0][e2];
          }
        }
      }
      if (!whole && lane == 0) {  // a split piece: its ticket is taken after all the work
        const int idx = atomicAdd(&sh.npend, 1);
        sh.pend_seg[idx] = s;
        sh.pend_poison[idx] = poisoned;
      }
    }
  }
  finish_range<NT>(p, sh, sm, rv, v_scale, issued, kseg);
  publish_status<NT>(p, sh);
}

cudaError_t launch_partial(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const PartialParams& p, int n_max, cudaStream_t stream) {
  // Programmatic dependent launch: CTAs may become resident while the previous
  // kernel on the stream (the planner, or whatever the caller ran before)
  // still runs; each waits for it with griddepcontrol.wait before reading its
  // inputs or writing global memory (before the wait it reads only its
  // first-page hints, to prefetch pages into L2).
  const int nt = (p.group * p.q_len + 7) / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_max);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = nt == 1 ? PartialGeom<1>::kSmem : PartialGeom<2>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // instances: (format) x (one tile, single token | one tile, several tokens |
  // two tiles); one-tile shapes with at least kWarpModeMinPieces segments per
  // CTA take the warp-capable kernel
  const bool multi = p.q_len > 1;
  const bool wm = nt == 1 && (long long)p.batch * p.num_kv_heads >= (long long)kWarpModeMinPieces * n_max;
  if (wm) {
    if (p.kv_dtype == XQA_KV_E4M3)
      return multi ? cudaLaunchKernelEx(&cfg, partial_kernel_wm<XQA_KV_E4M3, 1, true>, tm_k, tm_v, p)
                   : cudaLaunchKernelEx(&cfg, partial_kernel_wm<XQA_KV_E4M3, 1, false>, tm_k, tm_v, p);
    return multi ? cudaLaunchKernelEx(&cfg, partial_kernel_wm<XQA_KV_E5M2, 1, true>, tm_k, tm_v, p)
                 : cudaLaunchKernelEx(&cfg, partial_kernel_wm<XQA_KV_E5M2, 1, false>, tm_k, tm_v, p);
  }
  if (p.kv_dtype == XQA_KV_E4M3) {
    if (nt == 2) return cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E4M3, 2, true>, tm_k, tm_v, p);
    return multi ? cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E4M3, 1, true>, tm_k, tm_v, p)
                 : cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E4M3, 1, false>, tm_k, tm_v, p);
  }
  if (nt == 2) return cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E5M2, 2, true>, tm_k, tm_v, p);
  return multi ? cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E5M2, 1, true>, tm_k, tm_v, p)
               : cudaLaunchKernelEx(&cfg, partial_kernel<XQA_KV_E5M2, 1, false>, tm_k, tm_v, p);
}

cudaError_t set_partial_attributes() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const int s1 = PartialGeom<1>::kSmem, s2 = PartialGeom<2>::kSmem;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E5M2, 1, false>, a, s1)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E5M2, 1, true>, a, s1)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E5M2, 2, true>, a, s2)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E4M3, 1, false>, a, s1)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E4M3, 1, true>, a, s1)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel<XQA_KV_E4M3, 2, true>, a, s2)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel_wm<XQA_KV_E5M2, 1, false>, a, s1)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel_wm<XQA_KV_E5M2, 1, true>, a, s1)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(partial_kernel_wm<XQA_KV_E4M3, 1, false>, a, s1)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(partial_kernel_wm<XQA_KV_E4M3, 1, true>, a, s1);
}

}  // namespace xqa

#ifdef XQA_STAMPS
// Diagnostic builds: copies the phase stamps of the last launch (n_ctas rows
// of kStampsPerCta %globaltimer values, ns) to host memory, then clears them.
// Synchronises `stream`.
extern "C" int xqa_diag_read_stamps(unsigned long long* host, int n_ctas, void* stream) {
  if (!host || n_ctas < 1 || n_ctas > xqa::kMaxCtas) return XQA_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = (size_t)n_ctas * xqa::kStampsPerCta * sizeof(unsigned long long);
  void* dev = nullptr;
  if (cudaGetSymbolAddress(&dev, xqa::g_stamps) != cudaSuccess ||
      cudaMemcpyAsync(host, dev, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(dev, 0, bytes, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return XQA_ERR_LAUNCH;
  return XQA_OK;
}
#endif
