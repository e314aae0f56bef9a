/*
 * xqa.h — C ABI of the paged E5M2-KV grouped-query decode-attention library
 * (libxqa.so, sm_103a).
 *
 * One decode step: every sequence b contributes one query token with Hq heads;
 * its keys and values live in a paged FP8 E5M2 cache; q head h attends over the
 * ctx_b cached tokens of kv head h / G (G = Hq / Hkv). This is the operation
 * the page "[Kernel][SM70] Pipeline batched E5M2 XQA decode" optimises: one
 * step for many long sequences at once, keys and values stored as E5M2
 * (sections "Purpose" and "Starting bottleneck"). The partial kernel below is built from the phases that page
 * times separately (section "Pending work and gates"): fetching and decoding
 * K, sharing it through shared memory, QK, fetching and decoding V, PV, and
 * the synchronisation between them. The split-KV
 * planner -> forward -> merge structure follows the page "[Kernel][WIP] Follow
 * up FlashNext batch HC fusion and QSA route audit" (section "Test Result").
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers (or managed memory)
 *     owned by the caller; the library never frees or retains them.
 *   - The library allocates no memory and reads no environment variables,
 *     never calls abort/exit and never synchronises except in the xqa_read_*
 *     helpers, which say so. Host state it keeps: a per-device "kernel
 *     attributes set" flag and SM count, and the cached cuTensorMapEncodeTiled
 *     entry point.
 *     Device state it keeps: the XQA_STATIC_WORKSPACE_BYTES array of
 *     xqa_decode_static_workspace (one per device, shared by every call of
 *     that entry point). Between calls, a caller's workspace keeps the merge
 *     tickets (all zero after every completed call) and the last call's
 *     status words.
 *   - Work is enqueued on `stream` (a cudaStream_t; 0 = legacy default stream)
 *     on the current device. A non-OK return means nothing was enqueued unless
 *     the code is XQA_ERR_LAUNCH.
 *   - Problems only the device can see (a block id outside [0, NB), a context
 *     length outside [0, MBS*BS], a pipeline wait that ran out of time) are
 *     recorded in the status words inside the workspace (read them with
 *     xqa_read_status); the affected (sequence, kv head) output rows are
 *     written as NaN, and no out-of-bounds address is ever read.
 */
#ifndef XQA_H_
#define XQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum xqa_status {
  XQA_OK = 0,
  XQA_ERR_NULL = 1,        /* a required pointer is NULL */
  XQA_ERR_SHAPE = 2,       /* unsupported or inconsistent dimensions */
  XQA_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  XQA_ERR_WORKSPACE = 4,   /* workspace smaller than xqa_workspace_size */
  XQA_ERR_LAUNCH = 5,      /* a CUDA call or kernel launch failed */
  XQA_ERR_DEVICE = 6,      /* no usable CUDA device / attribute query failed */
  /* written by the device into the workspace status word: */
  XQA_ERR_BAD_BLOCK_ID = 16,    /* block_tables entry outside [0, num_blocks) */
  XQA_ERR_CTX_TOO_LONG = 17,    /* context length < 0 or > MBS * block_size */
  XQA_ERR_DEVICE_TIMEOUT = 18,  /* a pipeline or merge-ticket wait exceeded its time budget */
  XQA_ERR_DRAIN_TIMEOUT = 19    /* after a timeout, a copy was still in flight when its
                                   CTA exited: the device state is not to be trusted */
} xqa_status_t;

/* KV cache code formats (xqa_shape_t.kv_dtype). */
#define XQA_KV_E5M2 0 /* 1 sign, 5 exponent (bias 15), 2 mantissa bits */
#define XQA_KV_E4M3 1 /* 1 sign, 4 exponent (bias 7), 3 mantissa bits, no inf */

/* KV cache layouts (xqa_shape_t.kv_layout). */
#define XQA_LAYOUT_HND 0 /* [NB, Hkv, BS, D]: one (page, kv head) slice is contiguous */
#define XQA_LAYOUT_NHD 1 /* [NB, BS, Hkv, D]: token-major pages */

/* Problem dimensions. head_dim must be 128 and block_size 16; Hq must be a
 * multiple of Hkv, and G * q_len <= 16 with G = Hq / Hkv (so G <= 16). */
typedef struct xqa_shape {
  int32_t batch;              /* B: sequences (one query token each), >= 1 */
  int32_t num_q_heads;        /* Hq */
  int32_t num_kv_heads;       /* Hkv */
  int32_t head_dim;           /* D = 128 */
  int32_t block_size;         /* BS = 16 tokens per page */
  int32_t max_blocks_per_seq; /* MBS: row length of block_tables */
  int32_t num_blocks;         /* NB: pages in the K (and V) pool */
  float sm_scale;             /* softmax scale; <= 0 selects 1/sqrt(D) */
  int32_t max_ctas;           /* upper bound on split-KV CTAs; 0 = SM count;
                                 values above 1024 are taken as 1024 */
  int32_t min_pages_per_cta;  /* planner lower bound on pages per CTA; 0 = 16 */
  int32_t merge_mode;         /* how segments split over several CTAs are merged:
                                 0 = inside the partial kernel (default), by the
                                 last CTA to finish one, or for a segment of
                                 more than 16 pieces (6 when G * q_len > 8) by
                                 its last CTAs to finish, each taking some of
                                 the rows (when max_ctas <= SM count, so that
                                 every CTA is resident at once);
                                 1 = by the separate combine kernel (xqa_combine) */
  int32_t kv_dtype;           /* XQA_KV_E5M2 (0, default) or XQA_KV_E4M3 */
  int32_t kv_layout;          /* XQA_LAYOUT_HND (0, default) or XQA_LAYOUT_NHD */
  int32_t q_len;              /* T: new tokens per sequence; 0 or 1 = single-token
                                 decode. With T > 1, q and out are [B, T, Hq, D],
                                 context_lens count the T new tokens (their K/V
                                 already in the cache) and new token i attends
                                 causally to tokens 0 .. ctx_b - T + i (none if
                                 negative: a zero row) */
} xqa_shape_t;

/* Bytes of device workspace xqa_decode needs for `shape` on the current
 * device (depends on the SM count when max_ctas == 0). Host only. */
xqa_status_t xqa_workspace_size(const xqa_shape_t* shape, size_t* bytes);

/* Number of kernels one xqa_decode call enqueues for `shape` (so a caller can
 * size CUDA graphs or count launches). Host only; *kernels receives 1, 2 or 3. */
xqa_status_t xqa_kernels_per_call(const xqa_shape_t* shape, int32_t* kernels);

/* One decode step of paged GQA attention.
 *
 *   q             device, fp16 [B, Hq, D] ([B, T, Hq, D] with q_len T > 1),
 *                 contiguous, 16-byte aligned
 *   k_cache       device, FP8 codes (shape->kv_dtype) in the shape->kv_layout
 *                 layout: [NB, Hkv, BS, D] (HND: one (page, kv head) slice is
 *                 BS*D = 2048 contiguous bytes) or [NB, BS, Hkv, D] (NHD),
 *                 16-byte aligned
 *   v_cache       device, same layout as k_cache
 *   block_tables  device, int32 [B, MBS]; entry j of row b is the physical page
 *                 of tokens [16j, 16j+16) of sequence b; entries at or past
 *                 ceil(ctx_b / 16) are never read
 *   context_lens  device, int32 [B]; 0 <= ctx_b <= MBS*BS (0 gives a zero row)
 *   k_scale       per-tensor K scale (the key value is k_scale * FP8(code))
 *   v_scale       per-tensor V scale
 *   out           device, fp16, same shape as q, contiguous, 16-byte aligned
 *   workspace     device, >= xqa_workspace_size bytes, 256-byte aligned; holds
 *                 the plan, the split partials, the merge tickets, the
 *                 status words and each CTA's first pages of the last call
 *                 (a prefetch hint for the next call: any content is safe,
 *                 results never depend on it). Zero-fill it once before its
 *                 first use (e.g.
 *                 cudaMemsetAsync(workspace, 0, bytes)): every call leaves the
 *                 tickets at zero for the next. The tickets and status words
 *                 sit at fixed offsets, so one workspace may serve calls of
 *                 different shapes (sized for the largest). A call that is
 *                 not run to completion, or that reports
 *                 XQA_ERR_DEVICE_TIMEOUT or XQA_ERR_DRAIN_TIMEOUT (or
 *                 xqa_attend_partial with merge_mode 1 not followed by
 *                 xqa_combine) leaves it needing a fresh zero fill
 *
 * out[b, h, :] = sum_t softmax_t(sm_scale * <q[b,h], k_t>) * v_t over the
 * ctx_b tokens of kv head h / G, rounded to fp16 (round to nearest even).
 * Kernels enqueued: the split-KV partial kernel, which derives the split plan
 * itself and merges split segments when merge_mode is 0; before it the planner
 * when the batch is too large for the partial kernel to hold the segment table
 * (B * Hkv + 1 > 2048); with merge_mode 1 the log-sum-exp combine after it.
 * The first kernel becomes resident while the previous kernel on the stream
 * still runs and waits for it to complete before reading any input. No host
 * synchronisation; the call may be captured into a CUDA graph. Concurrent
 * calls must not share a workspace. */
xqa_status_t xqa_decode(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens,
                        float k_scale, float v_scale, void* out, const xqa_shape_t* shape,
                        void* workspace, size_t workspace_bytes, void* stream);

/* xqa_decode with the per-tensor scales read from device memory when the
 * kernels run (so a captured CUDA graph picks up new scales on replay):
 * k_scale and v_scale are device pointers to one float each. Results are
 * bitwise equal to xqa_decode called with the same values. */
xqa_status_t xqa_decode_device_scales(const void* q, const uint8_t* k_cache,
                                      const uint8_t* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, const float* k_scale,
                                      const float* v_scale, void* out, const xqa_shape_t* shape,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* The three stages of xqa_decode, exposed separately so they can be timed one
 * by one. Called in this order with the same arguments they give exactly the
 * results of xqa_decode. xqa_plan always launches the planner kernel (which
 * publishes the plan in the workspace, see xqa_read_plan); xqa_decode
 * launches it only when the batch needs it (see xqa_kernels_per_call), and
 * xqa_attend_partial must then follow it on the same workspace. With
 * merge_mode 0 the partial kernel merges split segments itself and
 * xqa_combine enqueues nothing. */
xqa_status_t xqa_plan(const int32_t* context_lens, const xqa_shape_t* shape, void* workspace,
                      size_t workspace_bytes, void* stream);
xqa_status_t xqa_attend_partial(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float k_scale, float v_scale, void* out,
                                const xqa_shape_t* shape, void* workspace,
                                size_t workspace_bytes, void* stream);
xqa_status_t xqa_combine(const int32_t* context_lens, float v_scale, void* out,
                         const xqa_shape_t* shape, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Exact E5M2 dequantisation (the "E5M2 conversion" phase on its own):
 *   out_fp16_bits[i] = (uint16_t)in[i] << 8        (the fp16 pattern, exact)
 *   out_f32[i]       = (float)fp16(in[i]) * scale  (optional; NULL to skip)
 * in, out_fp16_bits, out_f32: device pointers, n elements each; any
 * alignment. */
xqa_status_t xqa_dequant_e5m2(const uint8_t* in, size_t n, float scale, uint16_t* out_fp16_bits,
                              float* out_f32, void* stream);

/* Exact E4M3 dequantisation with the conversion routes the attention kernel
 * uses for E4M3 caches (every E4M3 value is an fp16 value):
 *   out_fp16_bits[i] = fp16 pattern of E4M3(in[i])      (exact; NaN codes -> NaN)
 *   out_f32[i]       = (float)fp16 * scale              (optional; NULL to skip)
 * Same argument conventions as xqa_dequant_e5m2. */
xqa_status_t xqa_dequant_e4m3(const uint8_t* in, size_t n, float scale, uint16_t* out_fp16_bits,
                              float* out_f32, void* stream);

/* Self-check of the device-side failure detection: launches one CTA whose
 * threads wait, through the same bounded mbarrier wait the attention kernel
 * uses, on a barrier that nothing ever arrives at. After budget_ns
 * (1 .. 2e9 ns) the wait gives up and the kernel writes XQA_ERR_DEVICE_TIMEOUT
 * to *device_status (a device int32) and returns; the context stays usable.
 * The attention kernel's budget is 1 s. Test use only. */
xqa_status_t xqa_selftest_wait_timeout(int32_t* device_status, uint64_t budget_ns, void* stream);

/* The device-reported status of the last call that used `workspace`:
 * *device_status receives XQA_OK or the first device-reported code in CTA
 * order (each CTA of the partial kernel writes its own status word as it
 * exits). Copies the fixed-size header/ticket/status region (12352 bytes) to
 * the host and synchronises `stream`. Returns XQA_ERR_WORKSPACE if the
 * workspace holds no status (neither zero-filled nor written by a call). */
xqa_status_t xqa_read_status(const void* workspace, int32_t* device_status, void* stream);

/* Copies the planner's output to host memory. Synchronises `stream`.
 *   header[4]          = {CTAs of the last partial launch, CTAs holding work,
 *                         total_pages, num_segments}
 *   seg_start[B*Hkv+1] = exclusive prefix sum of pages per (sequence, kv head)
 *   seg_bad[B*Hkv]     = 1 where the segment's context length is invalid,
 *                        else 0 (may be NULL)
 * The plan is published by the planner kernel when it runs, else by the
 * partial kernel's first CTA.
 *   seg_cost[B*Hkv]    = inclusive prefix sum of the segments' switch costs on
 *                        the cost line the CTAs are cut on: 32 page units per
 *                        non-empty segment, 0 for an empty one (may be NULL) */
xqa_status_t xqa_read_plan(const void* workspace, const xqa_shape_t* shape, int32_t* header,
                           int32_t* seg_start, int32_t* seg_bad, int32_t* seg_cost,
                           void* stream);

/* Size of the device array behind xqa_decode_static_workspace (per device). */
#define XQA_STATIC_WORKSPACE_BYTES ((size_t)8 << 20)

/* xqa_decode for callers that cannot allocate device memory.
 *
 * None of the pages describes this entry point. It exists for callers that
 * are not allowed to call cudaMalloc: a plugin inside a host runtime that owns
 * all device memory through its own pool, a latency-critical path where an
 * allocation (which may synchronise the device) is forbidden, or an operator
 * interface that passes only inputs and outputs and has no workspace hook.
 *
 * Arguments and results are those of xqa_decode, minus the workspace: the
 * split-KV scratch comes from a fixed XQA_STATIC_WORKSPACE_BYTES array in the
 * library's device image, which every device that loads the library holds
 * until the process exits. Nothing is allocated. The array is zero-filled when
 * the library's module loads on a device, and every completed call leaves it
 * ready for the next, so nothing needs clearing.
 *
 *   - Shapes whose xqa_workspace_size exceeds XQA_STATIC_WORKSPACE_BYTES are
 *     rejected with XQA_ERR_WORKSPACE before anything is enqueued (for 152
 *     SMs: B * Hkv up to about 850 segments).
 *   - Every call looks up the array's device address with
 *     cudaGetSymbolAddress, with the caller's device current (a host-side
 *     lookup; nothing is cached, so a device reset that reloads the module
 *     is followed). The first call on a device may load the library's module
 *     there: make it before any stream capture.
 *   - All calls on a device share the one array: calls that may overlap on the
 *     GPU (different streams without ordering, or threads racing on one device)
 *     race on it and corrupt each other. Order them, e.g. on one stream.
 *   - The device status words live in the shared array and are not exposed;
 *     rows affected by a bad block id or context length still come back NaN. */
xqa_status_t xqa_decode_static_workspace(const void* q, const uint8_t* k_cache,
                                         const uint8_t* v_cache, const int32_t* block_tables,
                                         const int32_t* context_lens, float k_scale,
                                         float v_scale, void* out, const xqa_shape_t* shape,
                                         void* stream);

/* Static, NUL-terminated description of a status code. */
const char* xqa_status_string(xqa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* XQA_H_ */
