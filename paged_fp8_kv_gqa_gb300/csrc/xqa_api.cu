// xqa_api.cu — the C ABI of libxqa: argument validation, TMA descriptors and
// the planner -> partial -> combine launches. See include/xqa.h for the
// contract of every entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "xqa.h"
#include "xqa_device.cuh"
#include "xqa_launch.h"

namespace xqa {
cudaError_t set_partial_attributes();
}

namespace {

using xqa::kBlockSize;
using xqa::kHeadDim;

constexpr int kMaxDevices = 64;
std::atomic<int> g_attrs_set[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];  // SM count, set with the attributes
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

struct Resolved {
  int batch, hq, hkv, group, mbs, nb;
  int nseg, n_max, min_pages, merge_mode, kv_dtype, kv_layout, q_len;
  float sm_scale;
  xqa::WsLayout ws;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

xqa_status_t resolve(const xqa_shape_t* s, Resolved* r) {
  if (!s) return XQA_ERR_NULL;
  if (s->head_dim != kHeadDim || s->block_size != kBlockSize) return XQA_ERR_SHAPE;
  if (s->batch < 1 || s->num_kv_heads < 1 || s->num_q_heads < 1) return XQA_ERR_SHAPE;
  if (s->num_q_heads % s->num_kv_heads != 0) return XQA_ERR_SHAPE;
  const int group = s->num_q_heads / s->num_kv_heads;
  if (s->max_blocks_per_seq < 1 || s->num_blocks < 1) return XQA_ERR_SHAPE;
  if (s->max_ctas < 0 || s->min_pages_per_cta < 0) return XQA_ERR_SHAPE;
  if (s->merge_mode != 0 && s->merge_mode != 1) return XQA_ERR_SHAPE;
  if (s->kv_dtype != XQA_KV_E5M2 && s->kv_dtype != XQA_KV_E4M3) return XQA_ERR_SHAPE;
  if (s->kv_layout != XQA_LAYOUT_HND && s->kv_layout != XQA_LAYOUT_NHD) return XQA_ERR_SHAPE;
  const int q_len = s->q_len > 0 ? s->q_len : 1;
  if (s->q_len < 0 || group * q_len > xqa::kMaxCols) return XQA_ERR_SHAPE;
  // int32 index arithmetic on the device: pool rows, total pages, segments
  const long long pool_rows = (long long)s->num_blocks * s->num_kv_heads * kBlockSize;
  const long long max_pages = (long long)s->batch * s->num_kv_heads * s->max_blocks_per_seq;
  if (pool_rows >= (1ll << 31) || max_pages >= (1ll << 31)) return XQA_ERR_SHAPE;
  if ((long long)s->batch * q_len * s->num_q_heads >= (1ll << 31) / kHeadDim) return XQA_ERR_SHAPE;
  r->batch = s->batch;
  r->hq = s->num_q_heads;
  r->hkv = s->num_kv_heads;
  r->group = group;
  r->mbs = s->max_blocks_per_seq;
  r->nb = s->num_blocks;
  r->nseg = s->batch * s->num_kv_heads;
  r->sm_scale = s->sm_scale > 0.f ? s->sm_scale : (float)(1.0 / sqrt((double)kHeadDim));
  r->min_pages = s->min_pages_per_cta > 0 ? s->min_pages_per_cta : xqa::kDefaultMinPagesPerCta;
  r->merge_mode = s->merge_mode;
  r->kv_dtype = s->kv_dtype;
  r->kv_layout = s->kv_layout;
  r->q_len = q_len;
  if (s->max_ctas > 0) {
    r->n_max = s->max_ctas;
  } else {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XQA_ERR_DEVICE;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1)
      return XQA_ERR_DEVICE;
    r->n_max = sms;
  }
  if (r->n_max > xqa::kMaxCtas) r->n_max = xqa::kMaxCtas;
  r->ws = xqa::ws_layout(r->nseg, r->n_max);
  return XQA_OK;
}

xqa_status_t check_workspace(const Resolved& r, const void* ws, size_t bytes) {
  if (!ws) return XQA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return XQA_ERR_ALIGN;
  if (bytes < r.ws.total) return XQA_ERR_WORKSPACE;
  return XQA_OK;
}

// SM count of the current device (cached by ensure_device_setup; 0 if unknown).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return g_sms[dev].load(std::memory_order_acquire);
}

xqa_status_t ensure_device_setup() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return XQA_ERR_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return XQA_ERR_DEVICE;
  if (g_attrs_set[dev].load(std::memory_order_acquire) == 0) {
    if (xqa::set_partial_attributes() != cudaSuccess) return XQA_ERR_LAUNCH;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return XQA_ERR_DEVICE;
    g_sms[dev].store(sms, std::memory_order_release);
    g_attrs_set[dev].store(1, std::memory_order_release);
  }
  if (g_encode.load(std::memory_order_acquire) == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return XQA_ERR_DEVICE;
    g_encode.store(reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn),
                   std::memory_order_release);
  }
  return XQA_OK;
}

// HND pool [NB, Hkv, BS, D]: 2-D view x = D (128 B rows), y = NB*Hkv*BS; box =
// one (page, kv head) slice of BS x D bytes.
// NHD pool [NB, BS, Hkv, D]: 3-D view x = D, y = Hkv, z = NB*BS; box = (D, 1, BS),
// the same 16 rows of 128 B in shared memory. Both with the 128-byte swizzle.
xqa_status_t encode_pool_map(CUtensorMap* map, const uint8_t* pool, const Resolved& r) {
  CUresult res;
  cuuint32_t estr[3] = {1, 1, 1};
  if (r.kv_layout == XQA_LAYOUT_HND) {
    cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)r.nb * r.hkv * kBlockSize};
    cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
    cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)kBlockSize};
    res = g_encode.load(std::memory_order_acquire)(
        map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(pool), dims, strides, box,
        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)r.hkv, (cuuint64_t)r.nb * kBlockSize};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)r.hkv * kHeadDim};
    cuuint32_t box[3] = {(cuuint32_t)kHeadDim, 1, (cuuint32_t)kBlockSize};
    res = g_encode.load(std::memory_order_acquire)(
        map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(pool), dims, strides, box,
        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
        // no L2 promotion: an NHD row is 128 B and its neighbours belong to
        // other kv heads, read by other CTAs much later (256-B promotion
        // nearly doubled the DRAM traffic: 70.8 vs 57.1 us per B16 step)
        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return res == CUDA_SUCCESS ? XQA_OK : XQA_ERR_LAUNCH;
}

int32_t* ws_i32(void* ws) { return reinterpret_cast<int32_t*>(ws); }

// The partial kernel derives the plan itself when its segment table fits in
// shared memory; larger batches need the planner kernel first.
bool needs_planner(const Resolved& r) { return r.nseg + 1 > xqa::kSegCache; }

}  // namespace

extern "C" {

xqa_status_t xqa_workspace_size(const xqa_shape_t* shape, size_t* bytes) {
  if (!bytes) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  *bytes = r.ws.total;
  return XQA_OK;
}

xqa_status_t xqa_kernels_per_call(const xqa_shape_t* shape, int32_t* kernels) {
  if (!kernels) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  *kernels = (needs_planner(r) ? 1 : 0) + 1 + (r.merge_mode == 1 ? 1 : 0);
  return XQA_OK;
}

xqa_status_t xqa_plan(const int32_t* context_lens, const xqa_shape_t* shape, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!context_lens) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  if ((st = check_workspace(r, workspace, workspace_bytes)) != XQA_OK) return st;
  cudaError_t e = xqa::launch_plan(context_lens, r.batch, r.hkv, r.mbs, r.n_max, r.min_pages,
                                   ws_i32(workspace), (cudaStream_t)stream);
  return e == cudaSuccess ? XQA_OK : XQA_ERR_LAUNCH;
}

}  // extern "C"

namespace {

xqa_status_t attend_partial_impl(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 float k_scale, float v_scale, const float* k_scale_ptr,
                                 const float* v_scale_ptr, void* out, const xqa_shape_t* shape,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  if ((st = check_workspace(r, workspace, workspace_bytes)) != XQA_OK) return st;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return XQA_ERR_ALIGN;
  if ((st = ensure_device_setup()) != XQA_OK) return st;
  alignas(64) CUtensorMap tm_k, tm_v;
  if ((st = encode_pool_map(&tm_k, k_cache, r)) != XQA_OK) return st;
  if ((st = encode_pool_map(&tm_v, v_cache, r)) != XQA_OK) return st;
  uint8_t* base = reinterpret_cast<uint8_t*>(workspace);
  xqa::PartialParams p;
  p.q = reinterpret_cast<const __half*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = reinterpret_cast<__half*>(out);
  p.header = ws_i32(workspace);
  p.seg_start = reinterpret_cast<int32_t*>(base + r.ws.seg_start_off);
  p.seg_bad = reinterpret_cast<int32_t*>(base + r.ws.seg_bad_off);
  p.seg_cc = reinterpret_cast<int32_t*>(base + r.ws.seg_cc_off);
  p.tickets = reinterpret_cast<int32_t*>(base + r.ws.ticket_off);
  p.status = reinterpret_cast<int32_t*>(base + r.ws.status_off);
  p.partials = reinterpret_cast<float*>(base + r.ws.partials_off);
  p.hints = reinterpret_cast<int32_t*>(base + r.ws.hint_off);
  p.n_max = r.n_max;
  p.min_pages = r.min_pages;
  p.fused_merge = r.merge_mode == 0 ? 1 : 0;
  // CTAs that wait for one another's merge tickets need the whole grid
  // resident at once: one CTA per SM, so no more CTAs than SMs
  p.merge_helpers = r.n_max <= device_sms() ? xqa::kMergeHelpers : 1;
  p.batch = r.batch;
  p.num_q_heads = r.hq;
  p.num_kv_heads = r.hkv;
  p.group = r.group;
  p.max_blocks_per_seq = r.mbs;
  p.num_blocks = r.nb;
  p.kv_dtype = r.kv_dtype;
  p.kv_layout = r.kv_layout;
  p.q_len = r.q_len;
  p.qk_scale_base = (double)r.sm_scale * 1.4426950408889634;  // sm_scale * log2(e)
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.k_scale_ptr = k_scale_ptr;
  p.v_scale_ptr = v_scale_ptr;
  cudaError_t e = xqa::launch_partial(tm_k, tm_v, p, r.n_max, (cudaStream_t)stream);
  return e == cudaSuccess ? XQA_OK : XQA_ERR_LAUNCH;
}

xqa_status_t combine_impl(const int32_t* context_lens, float v_scale, const float* v_scale_ptr,
                          void* out, const xqa_shape_t* shape, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!context_lens || !out) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  if ((st = check_workspace(r, workspace, workspace_bytes)) != XQA_OK) return st;
  if (!aligned16(out)) return XQA_ERR_ALIGN;
  if (r.merge_mode == 0) return XQA_OK;  // merged inside the partial kernel
  uint8_t* base = reinterpret_cast<uint8_t*>(workspace);
  xqa::CombineParams p;
  p.out = reinterpret_cast<__half*>(out);
  p.header = ws_i32(workspace);
  p.seg_start = reinterpret_cast<const int32_t*>(base + r.ws.seg_start_off);
  p.seg_cc = reinterpret_cast<const int32_t*>(base + r.ws.seg_cc_off);
  p.tickets = reinterpret_cast<int32_t*>(base + r.ws.ticket_off);
  p.partials = reinterpret_cast<const float*>(base + r.ws.partials_off);
  p.num_q_heads = r.hq;
  p.num_kv_heads = r.hkv;
  p.group = r.group;
  p.q_len = r.q_len;
  p.v_scale = v_scale;
  p.v_scale_ptr = v_scale_ptr;
  cudaError_t e = xqa::launch_combine(p, r.nseg, (cudaStream_t)stream);
  return e == cudaSuccess ? XQA_OK : XQA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

xqa_status_t xqa_attend_partial(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float k_scale, float v_scale, void* out,
                                const xqa_shape_t* shape, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return attend_partial_impl(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale,
                             nullptr, nullptr, out, shape, workspace, workspace_bytes, stream);
}

xqa_status_t xqa_combine(const int32_t* context_lens, float v_scale, void* out,
                         const xqa_shape_t* shape, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return combine_impl(context_lens, v_scale, nullptr, out, shape, workspace, workspace_bytes,
                      stream);
}

xqa_status_t xqa_decode(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens,
                        float k_scale, float v_scale, void* out, const xqa_shape_t* shape,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  if ((st = check_workspace(r, workspace, workspace_bytes)) != XQA_OK) return st;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return XQA_ERR_ALIGN;
  if ((st = ensure_device_setup()) != XQA_OK) return st;
  if (needs_planner(r) &&
      (st = xqa_plan(context_lens, shape, workspace, workspace_bytes, stream)) != XQA_OK)
    return st;
  if ((st = xqa_attend_partial(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale,
                               out, shape, workspace, workspace_bytes, stream)) != XQA_OK)
    return st;
  return xqa_combine(context_lens, v_scale, out, shape, workspace, workspace_bytes, stream);
}

xqa_status_t xqa_decode_device_scales(const void* q, const uint8_t* k_cache,
                                      const uint8_t* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, const float* k_scale,
                                      const float* v_scale, void* out, const xqa_shape_t* shape,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !k_scale ||
      !v_scale)
    return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  if ((st = check_workspace(r, workspace, workspace_bytes)) != XQA_OK) return st;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return XQA_ERR_ALIGN;
  if ((st = ensure_device_setup()) != XQA_OK) return st;
  if (needs_planner(r) &&
      (st = xqa_plan(context_lens, shape, workspace, workspace_bytes, stream)) != XQA_OK)
    return st;
  if ((st = attend_partial_impl(q, k_cache, v_cache, block_tables, context_lens, 0.f, 0.f,
                                k_scale, v_scale, out, shape, workspace, workspace_bytes,
                                stream)) != XQA_OK)
    return st;
  return combine_impl(context_lens, 0.f, v_scale, out, shape, workspace, workspace_bytes, stream);
}

xqa_status_t xqa_dequant_e5m2(const uint8_t* in, size_t n, float scale, uint16_t* out_fp16_bits,
                              float* out_f32, void* stream) {
  if (n == 0) return XQA_OK;
  if (!in || !out_fp16_bits) return XQA_ERR_NULL;
  cudaError_t e = xqa::launch_dequant(XQA_KV_E5M2, in, n, scale, out_fp16_bits, out_f32,
                                      (cudaStream_t)stream);
  return e == cudaSuccess ? XQA_OK : XQA_ERR_LAUNCH;
}

xqa_status_t xqa_dequant_e4m3(const uint8_t* in, size_t n, float scale, uint16_t* out_fp16_bits,
                              float* out_f32, void* stream) {
  if (n == 0) return XQA_OK;
  if (!in || !out_fp16_bits) return XQA_ERR_NULL;
  cudaError_t e = xqa::launch_dequant(XQA_KV_E4M3, in, n, scale, out_fp16_bits, out_f32,
                                      (cudaStream_t)stream);
  return e == cudaSuccess ? XQA_OK : XQA_ERR_LAUNCH;
}

xqa_status_t xqa_selftest_wait_timeout(int32_t* device_status, uint64_t budget_ns,
                                       void* stream) {
  if (!device_status) return XQA_ERR_NULL;
  if (budget_ns == 0 || budget_ns > 2000000000ull) return XQA_ERR_SHAPE;
  cudaError_t e = xqa::launch_wait_timeout(device_status, budget_ns, (cudaStream_t)stream);
  return e == cudaSuccess ? XQA_OK : XQA_ERR_LAUNCH;
}

xqa_status_t xqa_read_status(const void* workspace, int32_t* device_status, void* stream) {
  if (!workspace || !device_status) return XQA_ERR_NULL;
  cudaStream_t s = (cudaStream_t)stream;
  // header, tickets and status words: one copy of a fixed-size region
  const xqa::WsLayout lay = xqa::ws_layout(0, 0);
  static_assert(xqa::kMaxCtas <= 1024, "status region copied through the stack");
  int32_t words[xqa::kHeaderWords + 3 * xqa::kMaxCtas];
  if (cudaMemcpyAsync(words, workspace, lay.hint_off, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return XQA_ERR_LAUNCH;
  const int32_t launched = words[0];
  const int32_t* status = words + lay.status_off / 4;
  *device_status = XQA_OK;
  if (launched < 0 || launched > xqa::kMaxCtas) return XQA_ERR_WORKSPACE;  // never written
  for (int i = 0; i < launched; ++i)
    if (status[i] != XQA_OK) {
      *device_status = status[i];
      break;
    }
  return XQA_OK;
}

xqa_status_t xqa_read_plan(const void* workspace, const xqa_shape_t* shape, int32_t* header,
                           int32_t* seg_start, int32_t* seg_bad, int32_t* seg_cost,
                           void* stream) {
  if (!workspace || !header || !seg_start) return XQA_ERR_NULL;
  Resolved r;
  xqa_status_t st = resolve(shape, &r);
  if (st != XQA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const uint8_t* base = reinterpret_cast<const uint8_t*>(workspace);
  if (cudaMemcpyAsync(header, base, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(seg_start, base + r.ws.seg_start_off, (size_t)(r.nseg + 1) * 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return XQA_ERR_LAUNCH;
  if (seg_bad && cudaMemcpyAsync(seg_bad, base + r.ws.seg_bad_off, (size_t)r.nseg * 4,
                                 cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return XQA_ERR_LAUNCH;
  if (seg_cost && cudaMemcpyAsync(seg_cost, base + r.ws.seg_cc_off, (size_t)r.nseg * 4,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return XQA_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return XQA_ERR_LAUNCH;
  return XQA_OK;
}

const char* xqa_status_string(xqa_status_t status) {
  switch (status) {
    case XQA_OK: return "ok";
    case XQA_ERR_NULL: return "a required pointer is NULL";
    case XQA_ERR_SHAPE: return "unsupported or inconsistent dimensions";
    case XQA_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case XQA_ERR_WORKSPACE: return "workspace smaller than xqa_workspace_size";
    case XQA_ERR_LAUNCH: return "a CUDA call or kernel launch failed";
    case XQA_ERR_DEVICE: return "no usable CUDA device";
    case XQA_ERR_BAD_BLOCK_ID: return "device: block table entry outside [0, num_blocks)";
    case XQA_ERR_CTX_TOO_LONG: return "device: context length < 0 or > max_blocks_per_seq*16";
    case XQA_ERR_DEVICE_TIMEOUT: return "device: pipeline wait exceeded its time budget";
    case XQA_ERR_DRAIN_TIMEOUT:
      return "device: a copy was still in flight when its CTA gave up; device state not trusted";
  }
  return "unknown status";
}

}  // extern "C"
