// Internal declarations shared by the host library and the CUDA kernels.
// Layout constants follow the record format documented in include/oscar.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace oscar {

constexpr int D = 128;            // head_dim = quantisation group = Hadamard order
constexpr int PAGE = 64;          // tokens per page
constexpr int SINK = 64;          // BF16 sink tokens
constexpr int RECENT = 256;       // BF16 recent window
constexpr int RING_PAGES = RECENT / PAGE;
constexpr int BF16_PAGES_PER_REQ = 1 + RING_PAGES;
constexpr int CODE_BYTES = D / 4;              // 32
constexpr int META_BYTES = 4;                  // fp16 s, fp16 z
constexpr int K_CODES_OFF = 0;
constexpr int V_CODES_OFF = PAGE * CODE_BYTES;             // 2048
constexpr int K_META_OFF = 2 * PAGE * CODE_BYTES;          // 4096
constexpr int V_META_OFF = K_META_OFF + PAGE * META_BYTES; // 4352
constexpr int RECORD = V_META_OFF + PAGE * META_BYTES;     // 4608
constexpr int BF16_RECORD_ELEMS = 2 * PAGE * D;            // K rows then V rows
// INT2 record of a quantisation group size gk (128: the layout above; 64: two
// {s, z} per token, K meta [4096, 4608), V meta [4608, 5120))
__host__ __device__ constexpr int meta_bytes_for(int gk) { return META_BYTES * (D / gk); }
__host__ __device__ constexpr int k_meta_off_for(int) { return 2 * PAGE * CODE_BYTES; }
__host__ __device__ constexpr int v_meta_off_for(int gk) { return k_meta_off_for(gk) + PAGE * meta_bytes_for(gk); }
__host__ __device__ constexpr int record_for(int gk) { return v_meta_off_for(gk) + PAGE * meta_bytes_for(gk); }
static_assert(record_for(128) == RECORD && record_for(64) == 5120, "record sizes");
constexpr int MAX_G = 8;
// decode partial per (work item, query head): o[128], m, l, 2 floats of padding
// (a multiple of 16 bytes so o can be moved with 16-byte vector accesses)
constexpr int PARTIAL_FLOATS = D + 4;
constexpr int PARTIAL_M = D;
constexpr int PARTIAL_L = D + 1;

// sticky device error bits
constexpr int ERR_INT2_PAGE = 1;
constexpr int ERR_BF16_PAGE = 2;
constexpr int ERR_LENGTH = 4;
constexpr int ERR_TIMEOUT = 8;     // a bounded wait gave up

// Plain pointers into the cache's device memory.
struct DevCache {
  uint8_t* int2;
  size_t int2_layer_stride;      // bytes
  uint16_t* bf16;
  size_t bf16_layer_stride;      // elements
  const float* rot_k;            // [L][Hkv][D][D], x_rot = x R
  const float* rot_v;
  const float* rot_kt;           // transposes
  const float* rot_vt;
  const float* rot_cn;           // [2][L][Hkv]: max column norm of R_K, then R_V (rounded up)
  const float* tau_k;            // [L][Hkv]
  const float* tau_v;
  int32_t* hist_pt;              // [max_requests][max_pages]
  int32_t* bf16_pt;              // [max_requests][5]
  int32_t* err;
  int32_t* dec_count;            // [max_requests][Hkv]: decode CTAs done with a segment (0 between launches)
  uint32_t* dec_flag;            // [max_requests][Hkv]: epoch of the last step launch whose append of
                                 // that (request, kv head) is complete
  int32_t L, Hq, Hkv, G, max_pages;
  int32_t gk;                    // quantisation group size: 128 or 64
  int32_t record;                // record_for(gk) bytes per (page, kv head)
  int64_t n_int2_pages, n_bf16_pages;
  float scale;
};

// ---- page-table updates ---------------------------------------------------
struct PtEntry {
  int32_t table;   // 0 = hist_pt, 1 = bf16_pt
  int32_t index;   // flat index into that table
  int32_t value;
};
constexpr int PT_ENTRIES_PER_LAUNCH = 300;

cudaError_t launch_pt_update(const DevCache& c, const PtEntry* entries, int n, cudaStream_t s);

// ---- rotation set-up --------------------------------------------------------
cudaError_t launch_rotation_setup(const DevCache& c, const float* rot_k_src, const float* rot_v_src,
                                  float* rot_k, float* rot_v, float* rot_kt, float* rot_vt, float* rot_cn,
                                  cudaStream_t s);

// ---- prefill ------------------------------------------------------------------
// Copy input rows of positions [p0, p1) that fall in the sink or the recent ring.
struct BF16Dest {
  int32_t sink_page;
  int32_t ring_page[RING_PAGES];
};
cudaError_t launch_prefill_bf16(const DevCache& c, int layer, const uint16_t* k, const uint16_t* v,
                                int64_t in_base, int64_t p0, int64_t p1, BF16Dest dst, cudaStream_t s);
// Rotate / clip / quantise / pack input positions [h0, h1) into history pages
// read from the device page table row of `slot`.
cudaError_t launch_prefill_hist(const DevCache& c, int layer, int slot, const uint16_t* k, const uint16_t* v,
                                int64_t in_base, int64_t h0, int64_t h1, cudaStream_t s);

// ---- append / demote ----------------------------------------------------------
struct AppendReq {
  int32_t slot;
  int32_t in_row;          // row of the batch's k / v input (-1: demote only)
  int32_t dst_page;        // BF16 page of the new token
  int32_t dst_row;         // row inside it
  int32_t demote_slot;     // history slot (0..63) of the demoted token, -1: none
  int32_t hist_page;       // physical INT2 page receiving it
  int32_t src_page;        // BF16 ring page holding the demoted token
  int32_t src_row;
  int32_t pt_index;        // >= 0: write hist_pt[slot][pt_index] = hist_page
};
constexpr int APPEND_PER_LAUNCH = 48;
cudaError_t launch_append(const DevCache& c, int layer, const AppendReq* reqs, int n, const uint16_t* k,
                          const uint16_t* v, cudaStream_t s);
// Demotion of one (layer, request) in a multi-layer demote launch.
struct DemoteEntry {
  int32_t layer;
  AppendReq r;              // in_row = -1: no new token
};
constexpr int DEMOTE_PER_LAUNCH = 96;   // kernel arguments stay under 4 KiB
cudaError_t launch_demote_layers(const DevCache& c, const DemoteEntry* e, int n, cudaStream_t s);

// ---- decode ---------------------------------------------------------------------
// One launch covers up to DECODE_PER_LAUNCH requests; its segments are the
// (request i, kv head h) pairs, s = i Hkv + h.  The first nbc CTAs attend to the
// segments' BF16 pages (the sink page and the four ring pages): CTA b takes the
// BF16 blocks of segments b, b + nbc, ...  The other CTAs share the INT2 history
// pages: the segments' pages in order (npages per segment, one cost unit each),
// cut into one contiguous equal range per CTA.
struct DecodeReq {
  int32_t slot;            // request slot (page-table row)
  int32_t batch_row;       // row of q / out
  int32_t tokens;          // T
  int32_t hist_end;
  int32_t sink_page;
  int32_t ring_page[RING_PAGES];
  int32_t hot_page;        // history page index the step's append demotes into (-1: none)
  int32_t hot_new;         // physical INT2 page that demotion opens (page-table entry written by the
                           // step), -1: the page is already in the table
  int32_t npages;          // INT2 history pages of each kv head
  int32_t cost_start;      // first INT2 cost unit of (this request, kv head 0); each kv head
                           // takes DECODE_SEGMENT_SETUP_COST + npages units (none if npages is 0)
};
constexpr int DECODE_PER_LAUNCH = 64;
// A BF16 block (up to 20 sub-pages of 16 rows) counted as this many INT2 pages
// when the BF16 CTAs are sized: about the time it takes one CTA.
constexpr int DECODE_BF16_BLOCK_COST = 60;
// The append of one (request, kv head) in a decode step (K and V), likewise.
constexpr int DECODE_APPEND_COST = 30;
// Cost units in front of each segment's pages on the INT2 line: the set-up a CTA
// pays on entering a segment (q rotation, first-page latency), in INT2 pages.
constexpr int DECODE_SEGMENT_SETUP_COST = 40;
constexpr int DECODE_MAX_INT2 = 256;            // INT2 CTAs of a decode launch (at most one per SM)
constexpr int DECODE_BF16_ITEMS = 1 + RING_PAGES;   // BF16 pages per (request, kv head)
struct DecodePlan {
  int n;
  int ncta;                // persistent CTAs (at most one per SM): nbc BF16 CTAs, then the INT2 CTAs
  int nbc;
  int64_t total_cost;      // INT2 pages of the launch
  int64_t segments;        // n Hkv
  size_t partial_bytes;    // workspace: INT2 records (segments + ncta), then BF16 records (segments)
};
// Partial record of one (segment, CTA) or of a segment's BF16 pages: per query head
// of the group o[128], m (log2 domain), l.
inline size_t decode_record_bytes(int g) { return (size_t)g * PARTIAL_FLOATS * sizeof(float); }
// Failure-detection hooks of a launch: mbarrier wait rounds before a wait gives up
// (ERR_TIMEOUT), and the page copy (issue order) that warp 0 of every INT2 CTA
// never issues (-1: none), so that a test can make a wait run out.
struct DecodeDebug {
  uint32_t wait_limit;
  int32_t hold_copy;
};
constexpr uint32_t DECODE_WAIT_LIMIT = 100000;   // rounds of up to 20 us each
// One launch: the CTAs stream their cost ranges, and the last CTA to finish a
// segment (counted in dec_count) merges it into out.  With k_new / v_new (the
// step's new token rows [n][Hkv][128] bf16, batch rows) the launch is a whole
// decode step: its BF16 CTAs first append the new token of each (request, kv
// head) -- demoting into reqs[i].hot_page where it is set -- and release
// dec_flag = epoch; the CTA that streams the hot page waits for that flag.
// prefetch: the kernel launched just before on the stream is a decode of this
// cache, so the older history pages may be copied before the launch waits for it.
cudaError_t launch_decode(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& plan,
                          const uint16_t* q, float* out, void* workspace, const uint16_t* k_new,
                          const uint16_t* v_new, uint32_t epoch, bool prefetch, DecodeDebug dbg, cudaStream_t s);

// Fixed decode scratch (one static device array per device) for callers that
// cannot allocate.  The first call on a device, with that device current,
// takes the array's address and zeroes it on stream s.
constexpr size_t DECODE_SCRATCH_BYTES = size_t(8) << 20;
cudaError_t decode_scratch_address(void** ptr, cudaStream_t s);

}  // namespace oscar
