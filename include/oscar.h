/*
 * oscar.h -- C ABI of the GB300 three-segment INT2 KV cache (OSCAR hot path).
 *
 * Sources (web pages about OSCAR, "Offline Spectral Covariance-Aware Rotation"):
 *   [MTP] "Together AI Open-Sources OSCAR: An Attention-Aware 2-Bit KV Cache
 *         Quantization System for Long-Context LLM Serving" (MarkTechPost)
 *   [MS]  "TogetherAI开源OSCAR：超越 TurboQuant! 面向真实 Serving 的 2-bit KV
 *         Cache量化" (ModelScope community)
 *
 * The cache keeps, per request and layer, a BF16 sink of the first 64 tokens,
 * INT2 history, and a BF16 window of the most recent (up to) 256 tokens
 * ([MTP] section "The Serving System: Mixed-Precision Cache Layout"; [MS]
 * section "OSCAR的设计").  History tokens are rotated by the per-layer,
 * per-kv-head R_K / R_V, clipped to tau_K / tau_V, quantised to 2-bit codes
 * with an fp16 scale and zero point per 128-channel token-head group, and
 * packed four codes per byte into 64-token pages.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses of the current device; host
 *     pointers are ordinary process memory.  "stream" is a cudaStream_t (NULL
 *     = legacy default stream) passed as void*.
 *   - Tensors are dense row-major; bf16 values are passed as uint16_t bit
 *     patterns.  head_dim is 128 everywhere.  Device tensors (k, v, q, out)
 *     must start on a 16-byte boundary.
 *   - Every call returns an oscar_status.  Argument and state errors are
 *     detected on the host before any side effect and leave the cache
 *     unchanged.  Kernels are enqueued asynchronously on "stream"; device-side
 *     consistency failures (a page id out of range) set a sticky error word
 *     that oscar_cache_check() reports.  Nothing aborts or traps.
 *   - The caller owns every buffer it passes (q, k, v, out, workspace, the
 *     cache's device memory); the cache owns its host metadata.  A cache is
 *     not thread-safe; calls on one cache must come from one host thread at
 *     a time, and its kernels must run in stream order (one stream, or
 *     streams the caller orders).
 *   - A cache created with device_mem == NULL is a metadata-only "dry run":
 *     page allocation, page tables and lengths behave exactly as on a GPU,
 *     but no CUDA call is made and compute calls return OSCAR_ERR_DRY_RUN
 *     after validating and applying their metadata effects.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,   /* bad pointer, size, id or configuration       */
  OSCAR_ERR_OUT_OF_PAGES = 2,  /* page pool or request slots exhausted         */
  OSCAR_ERR_STATE = 3,         /* call not valid in the request's state        */
  OSCAR_ERR_CUDA = 4,          /* a CUDA runtime call failed                   */
  OSCAR_ERR_TIMEOUT = 5,       /* a bounded device wait gave up                */
  OSCAR_ERR_DEVICE_CHECK = 6,  /* a kernel found inconsistent metadata         */
  OSCAR_ERR_DRY_RUN = 7        /* compute requested on a metadata-only cache   */
} oscar_status;

typedef struct oscar_cache oscar_cache;

/* Geometry of a cache.  The fixed fields follow the pages: head_dim 128,
 * sink 64 and recent 256 tokens ([MTP] section "The Serving System"), group
 * size 128 ([MS] section "快速实践", --kv-cache-quant-group-size 128) or 64
 * ([MTP] section "What OSCAR Does Differently": G_K = 64 by default), and
 * 64-token pages (a reading: the pages name no page size).  With group size 64
 * each token-head has two {fp16 s, fp16 z} pairs (channels 0..63, 64..127)
 * and a record is 5120 bytes: K codes [0, 2048), V codes [2048, 4096), K meta
 * [4096, 4608) with token slot r at 4096 + 8 r (group 0's s, z, then group
 * 1's), V meta [4608, 5120) the same way. */
typedef struct {
  int32_t num_layers;
  int32_t num_q_heads;             /* multiple of num_kv_heads, G = q/kv <= 8   */
  int32_t num_kv_heads;
  int32_t head_dim;                /* must be 128                               */
  int32_t sink_tokens;             /* must be 64                                */
  int32_t recent_tokens;           /* must be 256                               */
  int32_t page_tokens;             /* must be 64                                */
  int32_t group_size;              /* 128, or 64 (two groups per token-head)    */
  int32_t max_requests;            /* request slots                             */
  int32_t max_pages_per_request;   /* INT2 pages one request may hold           */
  int64_t num_int2_pages;          /* physical INT2 pages (shared by layers)   */
  int64_t num_bf16_pages;          /* physical BF16 pages; 0 -> 5*max_requests  */
  float softmax_scale;             /* 0 -> 1/sqrt(head_dim)                     */
  uint64_t page_perm_seed;         /* 0 -> identity page order                  */
} oscar_cache_config;

/* Where each region lives inside the cache's device memory (byte offsets from
 * device_mem).  INT2 pool: [layer][page][kv_head][4608 bytes], each record
 * = K codes [64][32] | V codes [64][32] | K meta [64]{fp16 s, fp16 z} |
 * V meta [64]{s, z}; codes in rotated channel order, channel 4j+i in bits
 * 2i..2i+1 of byte j ([MS] section "OSCAR的设计": four 2-bit values per byte).
 * BF16 pool: [layer][page][kv_head][2][64][128] bf16 (K rows, then V rows).
 * Page tables: int32 hist_pt[max_requests][max_pages_per_request],
 * int32 bf16_pt[max_requests][5] (sink page, then four ring pages).  Ring
 * slot of position p >= 64: (p - 64) mod 256 -> page slot/64, row slot%64. */
typedef struct {
  size_t total_bytes;
  size_t int2_pool_offset, int2_layer_stride, int2_page_stride, int2_record_bytes;
  size_t bf16_pool_offset, bf16_layer_stride, bf16_page_stride, bf16_record_bytes;
  size_t rot_k_offset, rot_v_offset, rot_kt_offset, rot_vt_offset; /* fp32 [L][Hkv][128][128] */
  size_t rot_colnorm_offset;                                       /* fp32 [2][L][Hkv] */
  size_t tau_k_offset, tau_v_offset;                               /* fp32 [L][Hkv] */
  size_t hist_pt_offset, bf16_pt_offset, error_word_offset;
  size_t decode_count_offset;      /* int32 [max_requests][Hkv], zero between decode launches */
  size_t decode_flag_offset;       /* uint32 [max_requests][Hkv], step epochs (see oscar_decode_step) */
} oscar_cache_layout;

/* Bytes of device memory oscar_cache_create() needs for cfg (0 if invalid). */
size_t oscar_cache_device_bytes(const oscar_cache_config* cfg);

/* Create a cache in caller-owned device memory.
 *   device_mem  device buffer of >= oscar_cache_device_bytes(cfg) bytes,
 *               256-byte aligned; NULL -> metadata-only dry run.
 *   rot_k/rot_v device fp32 [L][Hkv][128][128]: R_K = U_Q H_Had P_br and
 *               R_V = U_S H_Had P_br of each layer and kv head ([MTP] section
 *               "What OSCAR Does Differently"), row-major, x_rot = x R.
 *               Copied in (and transposed copies made); ignored in dry run.
 *   tau_k/tau_v host fp32 [L][Hkv]: clip thresholds, each in (0, 65504].
 * The pools' contents start undefined; every byte that decode reads is
 * written by prefill / append before it is read. */
oscar_status oscar_cache_create(const oscar_cache_config* cfg, void* device_mem, size_t device_bytes,
                                const float* rot_k, const float* rot_v,
                                const float* tau_k, const float* tau_v,
                                void* stream, oscar_cache** out);
oscar_status oscar_cache_destroy(oscar_cache* cache);
oscar_status oscar_cache_get_layout(const oscar_cache* cache, oscar_cache_layout* out);

/* Open an empty request (takes one sink and four ring BF16 pages). */
oscar_status oscar_request_open(oscar_cache* cache, void* stream, int32_t* req_out);

/* Fork a request sharing the parent's first prefix_tokens positions: the sink
 * page and the history pages of positions 64..prefix_tokens-1 (prefix caching,
 * [MTP] Visual Explainer step 5; [MS] section "评估结果").  Requires
 * prefix_tokens >= 64, (prefix_tokens - 64) % 64 == 0, and that the parent has
 * demoted every position below prefix_tokens in every layer.  The child
 * starts with T = prefix_tokens and an empty recent window. */
oscar_status oscar_request_fork(oscar_cache* cache, int32_t parent, int64_t prefix_tokens, void* stream,
                                int32_t* req_out);

/* Close a request; pages whose reference count drops to zero are freed. */
oscar_status oscar_request_close(oscar_cache* cache, int32_t req);

/* Tokens cached and end of INT2 history of (req, layer): history is
 * [64, hist_end), the recent window [hist_end, T). */
oscar_status oscar_request_length(const oscar_cache* cache, int32_t req, int32_t layer,
                                  int64_t* tokens, int64_t* hist_end);

/* Host copy of a request's page tables.  hist_pt_out receives up to cap
 * entries; *num_pages the number allocated; bf16_pt_out (5 entries) the sink
 * page and the four ring pages. */
oscar_status oscar_request_pages(const oscar_cache* cache, int32_t req, int32_t* hist_pt_out, int32_t cap,
                                 int32_t* num_pages, int32_t* bf16_pt_out);

/* Free INT2 and BF16 pages. */
oscar_status oscar_cache_free_pages(const oscar_cache* cache, int64_t* int2_free, int64_t* bf16_free);

/* Prefill-quantize: append n_tokens tokens of one layer in bulk.
 *   k, v  device bf16 [n_tokens][Hkv][128]: positions T..T+n_tokens-1.
 * Positions < 64 go to the sink, the last min(256, ...) to the recent ring,
 * the rest are rotated, clipped, quantised and packed into history ([MTP]
 * section "The Serving System", write path).  Allowed on an empty request or
 * one whose recent window is empty (e.g. a fresh fork).  The result is
 * byte-identical to n_tokens calls of oscar_append. */
oscar_status oscar_prefill_quantize(oscar_cache* cache, int32_t req, int32_t layer,
                                    const uint16_t* k, const uint16_t* v, int64_t n_tokens, void* stream);

/* Append one token per request to one layer, demoting first when the recent
 * window is full: the oldest recent token is rotated, clipped, quantised and
 * packed into INT2 history, then the new token takes its ring slot ([MS]
 * section "OSCAR的设计": new tokens enter the recent window, the oldest recent
 * token is demoted by the fused write kernel).
 *   reqs  host int32 [n], distinct request ids.
 *   k, v  device bf16 [n][Hkv][128]. */
oscar_status oscar_append(oscar_cache* cache, int32_t layer, int32_t n, const int32_t* reqs,
                          const uint16_t* k, const uint16_t* v, void* stream);

/* Demote the oldest recent token of each request to INT2 (the recent window
 * shrinks by one).  reqs: host int32 [n], distinct. */
oscar_status oscar_demote(oscar_cache* cache, int32_t layer, int32_t n, const int32_t* reqs, void* stream);

/* Multi-layer demote: oscar_demote(l, n, reqs) for every layer l in
 * [layer_begin, layer_end), with the same state changes and cache bytes, as one
 * launch per 96 (layer, request) pairs.  The token leaving the recent window at
 * a step is the same position in every layer and already sits in each layer's
 * ring, so its demotion in all layers can run at the start of the step; the
 * per-layer appends (or oscar_decode_step calls) that follow find room in the
 * window and only write the new token ([MTP] section "The Serving System":
 * write path; [MS] section "OSCAR的设计": the oldest recent token is demoted).
 *   reqs  host int32 [n], distinct request ids.
 * Errors: a bad layer range or batch is OSCAR_ERR_INVALID_ARG; a layer whose
 * recent window is empty is OSCAR_ERR_STATE; too few free INT2 pages is
 * OSCAR_ERR_OUT_OF_PAGES.  Every layer is checked before any change, so an
 * error leaves the cache as it was. */
oscar_status oscar_demote_layers(oscar_cache* cache, int32_t layer_begin, int32_t layer_end, int32_t n,
                                 const int32_t* reqs, void* stream);

/* Workspace bytes oscar_decode_attention needs for this batch. */
oscar_status oscar_decode_workspace_bytes(const oscar_cache* cache, int32_t n, const int32_t* reqs,
                                          size_t* bytes);

/* Decode attention of one layer over every cached token of each request:
 * rotate q by R_K, scan the INT2 history (split over pages), attend to the
 * BF16 sink and recent window with the unrotated q, merge all partials with
 * an online-softmax (max / sum) reduction and apply R_V^T to the history part
 * ([MS] section "OSCAR的设计": unpack, scale/zero dequantise, float
 * accumulate, online-softmax merge; [MTP] section "The Serving System").
 *   reqs       host int32 [n] distinct request ids (each with T >= 1);
 *              a repeated id is OSCAR_ERR_INVALID_ARG.
 *   q          device bf16 [n][Hq][128].
 *   out        device fp32 [n][Hq][128].
 *   workspace  device, >= oscar_decode_workspace_bytes(), 256-byte aligned;
 *              no initial contents are needed.  Calls that share a workspace
 *              must not overlap on the GPU.
 * The decode is one kernel per launch of up to 64 requests: one CTA per SM
 * streams an equal share of the pages, and the CTAs that finish a (request, kv
 * head) are counted in the cache's per-(request, kv head) counters (layout
 * decode_count_offset); the last one merges it, or, when each (request, kv head)
 * of the launch has a CTA of its own for the BF16 pages, that CTA waits for the
 * count and merges.  The kernel waits for everything before it on
 * "stream", as any launch does; decodes of the same request must not overlap
 * on the GPU (on one stream they never do). */
oscar_status oscar_decode_attention(oscar_cache* cache, int32_t layer, int32_t n, const int32_t* reqs,
                                    const uint16_t* q, float* out, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* oscar_decode_attention without a workspace argument: the library allocates
 * nothing.  The pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory around a decode step (a serving engine
 * that gives all free HBM to its KV pools at start-up and owns no per-step
 * allocator, or a plain C host with no allocator to pass).  The decode's
 * scratch (its partial records) lives in one fixed static device array
 * of 8 MiB per device inside the library.
 *   Arguments, layouts and results are those of oscar_decode_attention.
 *   Size limit: a batch whose partial records (per launch of up to 64
 *     requests: two per request and kv head plus one per SM, G x 528
 *     bytes each) need more than 8 MiB is rejected with OSCAR_ERR_INVALID_ARG
 *     before any work; use oscar_decode_attention with a caller workspace.
 *   Set-up: every call takes the array's address on the current device
 *     (cudaGetSymbolAddress, so a module reloaded after a device reset is
 *     found afresh); the first call on each device also zeroes it on "stream"
 *     (an error there is OSCAR_ERR_CUDA).  Make that first call before
 *     capturing any stream.  No part of the array needs particular contents
 *     when a call starts.
 *   Overlap: the array is shared by every cache on the device; two calls
 *     that overlap on the GPU (other streams, other caches) race. */
oscar_status oscar_decode_attention_noalloc(oscar_cache* cache, int32_t layer, int32_t n, const int32_t* reqs,
                                            const uint16_t* q, float* out, void* stream);

/* One decode step of one layer: oscar_append(layer, n, reqs, k, v) followed by
 * oscar_decode_attention(layer, n, reqs, q, out, workspace), with identical
 * results, as one kernel per launch of up to 48 requests: its BF16 CTAs first
 * append the new token of each (request, kv head) -- the demotion of the oldest
 * recent token into INT2 history included -- and mark it done in the cache's
 * step flags (layout decode_flag_offset); the CTA that streams the history page
 * a demotion fills waits for that mark (bounded) before copying it, and the new
 * token itself is read from k / v ([MTP] section "The Serving System": the write
 * path and decode attention of a step).
 *   k, v       device bf16 [n][Hkv][128], the new token of each request.
 *   q, out     as oscar_decode_attention.
 *   workspace  device, >= oscar_decode_workspace_bytes() taken before the step
 *              (it covers the page the append may add), 256-byte aligned.
 * Every argument and state check (those of both calls, and a workspace too
 * small for the decode after the append) is made before any change. */
oscar_status oscar_decode_step(oscar_cache* cache, int32_t layer, int32_t n, const int32_t* reqs,
                               const uint16_t* k, const uint16_t* v, const uint16_t* q, float* out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Failure-detection hooks of the decode launches of this cache (test use; the
 * pages have no counterpart).  wait_limit: rounds (up to 20 us each) a bounded
 * device wait on a page copy makes before it gives up and reports
 * OSCAR_ERR_TIMEOUT through oscar_cache_check (default 100000, from 1 to
 * 2^24; the other bounded waits of a decode launch scale with it).
 * hold_copy: the page copy (numbered in issue order, from 0, across the segments
 * of the CTA) of warp 0 of every decode CTA that streams history pages that is
 * never issued, so that its wait runs out (-1, the default, holds none).  A warp whose wait ran out issues no
 * further copy, waits (with the default limit) for the copies it has in flight
 * and skips its remaining pages; the launch's output is then undefined but the
 * device stays usable and the next launch starts clean.  OSCAR_ERR_INVALID_ARG
 * for values out of range. */
oscar_status oscar_debug_decode_hooks(oscar_cache* cache, uint32_t wait_limit, int32_t hold_copy);

/* Synchronise "stream" and report the sticky device error word (then clear it). */
oscar_status oscar_cache_check(oscar_cache* cache, void* stream);

/* Text of the last error on this cache ("" if none); valid until the next call. */
const char* oscar_last_error(const oscar_cache* cache);

/* Library version string. */
const char* oscar_version(void);

/* ---- Uncompressed BF16 baseline -------------------------------------------
 * Plain softmax attention over a paged BF16 KV cache, the comparison point of
 * the pages' decode-speed results ([MTP] section "Results": the 2-bit cache
 * against a BF16 cache of the same context):
 *   out[i][h] = softmax(q[i][h] K_i^T * scale) V_i   over all lens[i] tokens,
 * K_i, V_i the tokens of request i in the kv head h / (Hq / Hkv).
 *   kv          device bf16 [num_pages][Hkv][2][64][128]: per page and kv head,
 *               64 K rows then 64 V rows; token t of request i sits in page
 *               page_table[i][t / 64], row t % 64.  Bytes of rows past lens[i]
 *               are never used.
 *   page_table  device int32 [n][max_pages].
 *   lens        host int32 [n], each >= 1 and <= 64 * max_pages.
 *   q           device bf16 [n][Hq][128]; out device fp32 [n][Hq][128].
 *   scale       softmax scale; <= 0 selects 1 / sqrt(128).
 *   workspace   device, >= oscar_bf16_decode_workspace_bytes(); its first 4
 *               bytes become nonzero if a page id was out of range (that page
 *               is then read as page 0).
 * 1 <= n <= 64, Hq / Hkv in {1, 2, 4, 8}; kv, q, out and workspace 16-byte
 * aligned.  Asynchronous on "stream"; argument errors are returned before any
 * launch.  The workspace size returned is 0 for arguments outside these limits. */
size_t oscar_bf16_decode_workspace_bytes(int32_t n, const int32_t* lens, int32_t num_q_heads, int32_t num_kv_heads);
oscar_status oscar_bf16_decode(const void* kv, int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                               const int32_t* lens, int32_t n, int32_t num_q_heads, int32_t num_kv_heads,
                               float scale, const void* q, float* out, void* workspace, size_t workspace_bytes,
                               void* stream);

#ifdef __cplusplus
}
#endif
#endif /* OSCAR_H */
