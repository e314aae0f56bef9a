// xqa_device.cuh — device-side building blocks shared by the libxqa kernels:
// inline-PTX wrappers (mbarrier, TMA, warp MMA, movmatrix), the exact E5M2 ->
// fp16 conversions, bounded pipeline waits and the workspace layout.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "xqa.h"

namespace xqa {

// ---------------------------------------------------------------------------
// fixed geometry of the tuned path
// ---------------------------------------------------------------------------
constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
// Columns (new token x q head) per kv head: G * q_len <= 16, in one or two
// 8-wide MMA tiles (so G <= 16: G = 16 takes both tiles for one new token).
constexpr int kMaxCols = 16;
constexpr int kPageBytes = kBlockSize * kHeadDim;             // one (page, kv head) slice: 2048 B
constexpr int kStageBytes = 2 * kPageBytes;                   // K slice + V slice
constexpr int kWarps = 8;                                     // every warp loads and computes
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 32;                                   // smem ring depth (multiple of kWarps)
constexpr int kLookahead = kStages / kWarps;                  // pages in flight per warp
constexpr int kScratchStride = kHeadDim + 4;                  // floats per (warp, head) merge row
constexpr int kSegCache = 2048;  // seg_start (and context length) entries kept in smem

// Per-instance geometry of the partial kernel with NT MMA column tiles
// (8 * NT columns = new token x head): merge buffers hold every warp's O rows,
// then m[warp][col], l[warp][col]. One-tile kernels keep two buffers (merges
// deferred), two-tile kernels one (their buffer is twice as large).
template <int NT>
struct PartialGeom {
  static constexpr int kCols = 8 * NT;
  static constexpr int kScratchFloats = kWarps * kCols * kScratchStride;
  static constexpr int kMergeBufFloats = kScratchFloats + 2 * kWarps * kCols;
  static constexpr int kMergeBufs = NT == 1 ? 2 : 1;
  static constexpr int kSmem = 1024 /* alignment slack for the 1024-B swizzle atom */ +
                               kStages * kStageBytes + kMergeBufs * kMergeBufFloats * 4 +
                               kSegCache * 4 /* segment starts */ + kSegCache * 4 /* lengths */ +
                               kSegCache * 4 /* cost prefix */;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};
constexpr int kDefaultMinPagesPerCta = 16;
// Split rule cost line: every non-empty segment costs kSegCost page units on
// top of its pages (a segment switch inside a CTA, and the split-piece merge
// work that falls on CTAs holding segment boundaries; the value minimises the
// step time of the B8, B16 and mixed-length workloads, swept over 0..48).
constexpr int kSegCost = 32;
// The final merge of a split segment by its last CTA alone, from registers:
// up to kFewPieces pieces (both segments a CTA completes in one round trip),
// or in one-tile kernels up to kWidePieces pieces (one round trip each).
// Larger segments are merged by several CTAs, gathered in shared memory.
constexpr int kFewPieces = 6;  // covers the 5-6 pieces of 16K-token segments on 152 SMs
constexpr int kWidePieces = 16;
// A split segment of at most kArriveFirstPieces pieces and at least
// kArriveFirstPages pages is merged by the last piece to arrive (its long
// pieces finish at spread-out times); other segments of up to kWidePieces by
// the piece written last (their pieces finish nearly together, and the last
// to arrive would wait for another's slot).
constexpr int kArriveFirstPieces = 4;
constexpr int kArriveFirstPages = 512;
// Warp mode of the partial kernel: a CTA range of at least this many segment
// pieces, none longer than kWarpModePages pages, gives whole pieces to warps.
constexpr int kWarpModeMinPieces = 4;
constexpr int kWarpModePages = 32;
// The planner is one CTA. Its registers do not fit beside a partial CTA (which
// takes 61,440 of the SM's 65,536), so the partial CTA bound for the
// planner's SM starts when the planner exits; the planner therefore does one
// scan and a single round of loads whatever the batch.
constexpr int kPlanThreads = 256;
constexpr int kCombineThreads = 256;  // 8 warps: a warp per column, 4 dims per lane

// Partial-result slot: O[col][128] unnormalised fp32, then M[col] (log2 domain),
// L[col], for up to kMaxCols columns.
constexpr int kSlotFloats = kMaxCols * kHeadDim + 2 * kMaxCols;
constexpr int kSlotM = kMaxCols * kHeadDim;
constexpr int kSlotL = kMaxCols * kHeadDim + kMaxCols;

// A pipeline wait that has not completed after this long is treated as a fault.
constexpr unsigned long long kWaitBudgetNs = 1000000000ull;  // 1 s

// ---------------------------------------------------------------------------
// workspace layout (int32 words, then 256-byte aligned fp32 partials)
// ---------------------------------------------------------------------------
// Upper bound on the CTAs of one partial launch (max_ctas is clamped to it).
// The merge-ticket and status regions below are sized by it, not by the
// shape, so they sit at the same offsets whatever shape uses the workspace.
constexpr int kMaxCtas = 1024;
// Each split segment has two ticket words, indexed by the CTA holding its
// first page: tickets[i] and tickets[kMaxCtas + i].
//  * In-kernel merge (merge_mode 0): the first word counts the pieces that
//    have arrived (bits 0-15; taken as soon as a CTA's pages are done, the
//    old count giving the piece's arrival order) and, in bits 27-30, the
//    merging CTAs that have seen every piece written (when several CTAs share
//    the final merge); the second counts the pieces written (bits 0-15,
//    added with release order after the piece's slot) and those that met a
//    bad page (bits 16-26).
//  * Combine kernel (merge_mode 1): the first word counts the pieces written
//    and the bad ones as above; the combine kernel reads and clears it.
constexpr int kTicketPoison = 1 << 16;
constexpr int kTicketRelease = 1 << 27;
constexpr int kTicketCountMask = kTicketPoison - 1;
constexpr int kTicketPoisonMask = kTicketRelease - kTicketPoison;
static_assert(kMaxCtas * (long long)kTicketPoison < kTicketRelease, "poison bits overflow");
// The final merge of a larger split segment is shared by up to this many of
// its last CTAs (output rows dealt round robin) when every CTA of the launch
// is resident at once.
constexpr int kMergeHelpers = 8;
static_assert(kMergeHelpers * (long long)kTicketRelease <= 0x7fffffffLL + 1, "release bits overflow");
constexpr int kHeaderWords = 16;
// Pages of a CTA's range (each warp's first pair) that the CTA records for the
// next call, as (block id * Hkv + kv head) * 16: that call's CTA of the same
// index prefetches them into L2 while it waits for the kernels before it (a
// hint: consecutive calls, e.g. the layers of one decode step, cut the same
// pages).
constexpr int kHintPages = 2 * 8;

struct WsLayout {
  // header[0] CTAs of the last partial launch (status words written),
  // [1] CTAs holding work, [2] total pages, [3] segments
  size_t ticket_off;     // int32 [2 * kMaxCtas]: merge tickets, zero between calls
  size_t status_off;     // int32 [kMaxCtas]: each CTA's status in the last call
  size_t hint_off;       // int32 [kMaxCtas * kHintPages]: first pages of each CTA's last range
  size_t seg_start_off;  // int32 [nseg + 1]
  size_t seg_bad_off;    // int32 [nseg]: 1 where the context length is invalid
  size_t seg_cc_off;     // int32 [nseg]: cost of segments 0..s (inclusive), see seg_cost
  size_t partials_off;   // float [(n_max + nseg) * kSlotFloats]
  size_t total;
};

__host__ __device__ inline WsLayout ws_layout(long long nseg, long long n_max) {
  WsLayout l;
  l.ticket_off = 4 * kHeaderWords;
  l.status_off = l.ticket_off + 8 * (size_t)kMaxCtas;
  l.hint_off = l.status_off + 4 * (size_t)kMaxCtas;
  l.seg_start_off = l.hint_off + 4 * (size_t)kMaxCtas * kHintPages;
  l.seg_bad_off = l.seg_start_off + 4 * (size_t)(nseg + 1);
  l.seg_cc_off = l.seg_bad_off + 4 * (size_t)nseg;
  size_t end = l.seg_cc_off + 4 * (size_t)nseg;
  l.partials_off = (end + 255) & ~(size_t)255;
  l.total = l.partials_off + (size_t)(n_max + nseg) * kSlotFloats * sizeof(float);
  return l;
}

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar`. Gives up (returns false) when *abort is
// set by another warp or after budget_ns; never spins without bound.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort,
                                                  uint64_t budget_ns = kWaitBudgetNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > budget_ns) return false;
  }
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 prefetch of one 2-D tensor tile (coordinates outside the tensor fetch
// nothing; no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// L2 prefetch of one 3-D tensor tile (as tma_prefetch_2d).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Device-scope relaxed load (a value another kernel may be writing).
__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* addr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load (NHD caches: x = dims, y = kv head, z = token row).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// exact E5M2 -> fp16: the fp16 pattern of an E5M2 code is the code in the high
// byte and zero in the low byte, so dequantisation is a byte permutation.
// ---------------------------------------------------------------------------

// Two codes of one 32-bit word that are adjacent along the contraction index:
// bytes {0,1} (lo) or {2,3} (hi) of `w` -> half2 {w.b0<<8, w.b1<<8} etc.
__device__ __forceinline__ uint32_t e5m2x2_lo(uint32_t w) { return prmt(w, 0u, 0x1404u); }
__device__ __forceinline__ uint32_t e5m2x2_hi(uint32_t w) { return prmt(w, 0u, 0x3424u); }

// Codes of two different words taken at the same byte position: interleave
// {x.b0, x.b1, y.b0, y.b1} (or bytes 2,3), then widen each pair.
__device__ __forceinline__ uint32_t interleave01(uint32_t x, uint32_t y) { return prmt(x, y, 0x5410u); }
__device__ __forceinline__ uint32_t interleave23(uint32_t x, uint32_t y) { return prmt(x, y, 0x7632u); }
// From an interleaved word {x_k, x_k+1, y_k, y_k+1}: half2 {x_k, y_k} / {x_k+1, y_k+1}.
__device__ __forceinline__ uint32_t pair_even(uint32_t iw) { return prmt(iw, 0u, 0x2404u); }
__device__ __forceinline__ uint32_t pair_odd(uint32_t iw) { return prmt(iw, 0u, 0x3414u); }

// Programmatic dependent launch: the planner lets the partial kernel start
// early; the partial kernel waits for the planner's writes only where it needs
// them (no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The planner's split rule (also evaluated inside the partial kernel):
// n = 0 if P == 0 else min(n_max, max(1, ceil(P / min_pages))).
__host__ __device__ inline int num_ctas_for(int total_pages, int n_max, int min_pages) {
  if (total_pages <= 0) return 0;
  int n = (total_pages + min_pages - 1) / min_pages;
  n = n < 1 ? 1 : n;
  return n < n_max ? n : n_max;
}

// The cost line. Segment s (pages segs[s] .. segs[s+1]) costs
// seg_cost(pages) units before its pages; cc[s] = sum of the costs of
// segments 0..s. Page p of segment s sits at position p + cc[s], the line is
// V = P + cc[nseg - 1] long, CTA i takes the positions [floor(iV/n),
// floor((i+1)V/n)) and so a contiguous (possibly empty) run of pages.
__host__ __device__ inline int seg_cost(int pages) { return pages <= 0 ? 0 : kSegCost; }

// CTA owning position v of a line of length V split over n CTAs.
__host__ __device__ inline int cta_of_vpos(long long v, long long line, long long n) {
  return (int)(((v + 1) * n - 1) / line);
}


// Device-scope load with acquire ordering.
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* addr) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Polls a merge ticket (acquire) until its count reaches n; returns the word,
// or -1 once kWaitBudgetNs have passed.
__device__ __forceinline__ int wait_ticket_count(const int32_t* ticket, int n) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    const int w = ld_acquire_gpu(ticket);
    if ((w & kTicketCountMask) == n) return w;
    if (global_timer_ns() - t0 > kWaitBudgetNs) return -1;
  }
}

// Device-scope fetch-and-add with acquire-release ordering.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v)
               : "memory");
  return old;
}

// Device-scope reduction (no result) with release ordering.
__device__ __forceinline__ void red_add_release_gpu(int32_t* addr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// exact E4M3 -> fp16: every E4M3 value (and NaN) is an fp16 value; the
// hardware conversion of a pair of codes is exact.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<unsigned short>(pair16)));
  return d;
}

// Per-format conversions in the two shapes the attention kernel needs:
//   k_lo / k_hi: the two codes at bytes {0,1} / {2,3} of a word -> half2;
//   v_pairs:     same-position codes of two words x, y -> half2
//                {x0,y0}, {x1,y1}, {x2,y2}, {x3,y3}.
template <int kFmt>
struct KvConv;

template <>
struct KvConv<XQA_KV_E5M2> {
  __device__ __forceinline__ static uint32_t k_lo(uint32_t w) { return e5m2x2_lo(w); }
  __device__ __forceinline__ static uint32_t k_hi(uint32_t w) { return e5m2x2_hi(w); }
  __device__ __forceinline__ static void v_pairs(uint32_t x, uint32_t y, uint32_t (&o)[4]) {
    const uint32_t i01 = interleave01(x, y), i23 = interleave23(x, y);
    o[0] = pair_even(i01);
    o[1] = pair_odd(i01);
    o[2] = pair_even(i23);
    o[3] = pair_odd(i23);
  }
};

template <>
struct KvConv<XQA_KV_E4M3> {
  __device__ __forceinline__ static uint32_t k_lo(uint32_t w) { return e4m3x2_to_f16x2(w & 0xffffu); }
  __device__ __forceinline__ static uint32_t k_hi(uint32_t w) { return e4m3x2_to_f16x2(w >> 16); }
  __device__ __forceinline__ static void v_pairs(uint32_t x, uint32_t y, uint32_t (&o)[4]) {
    const uint32_t a = prmt(x, y, 0x5140u);  // {x0, y0, x1, y1}
    const uint32_t b = prmt(x, y, 0x7362u);  // {x2, y2, x3, y3}
    o[0] = e4m3x2_to_f16x2(a & 0xffffu);
    o[1] = e4m3x2_to_f16x2(a >> 16);
    o[2] = e4m3x2_to_f16x2(b & 0xffffu);
    o[3] = e4m3x2_to_f16x2(b >> 16);
  }
};

// First error of a CTA wins (status lives in shared memory until the CTA exits).
__device__ __forceinline__ void record_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

}  // namespace xqa
