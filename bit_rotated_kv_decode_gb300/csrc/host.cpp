// Host side of the C ABI: configuration checks, device-memory layout, the
// seeded page allocator, request state (lengths and page tables) and kernel
// launches.  Nothing here touches the GPU in a metadata-only (dry-run) cache.
//
// Request state follows the three-segment layout of "Together AI Open-Sources
// OSCAR" (MarkTechPost), section "The Serving System: Mixed-Precision Cache
// Layout": sink [0, 64), INT2 history [64, hist_end), BF16 recent window
// [hist_end, T) of at most 256 tokens.  Page sharing for forks follows the
// prefix-cache compatibility the pages claim (same page, Visual Explainer step
// 5; "TogetherAI开源OSCAR" (ModelScope), section "评估结果").
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "oscar.h"

using namespace oscar;

namespace {


size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// SplitMix64 (Steele, Lea, Flood 2014).
struct SplitMix64 {
  uint64_t state;
  uint64_t next() {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
};

// Stack of free page ids; the first pops follow a seeded Fisher-Yates
// permutation of 0..n-1 (identity for seed 0).  Freed pages are pushed on top.
struct PagePool {
  std::vector<int32_t> stack;
  std::vector<int32_t> refs;
  void init(int64_t n, uint64_t seed) {
    std::vector<int32_t> order(n);
    for (int64_t i = 0; i < n; ++i) order[i] = static_cast<int32_t>(i);
    if (seed != 0) {
      SplitMix64 g{seed};
      for (int64_t i = n - 1; i >= 1; --i) {
        const uint64_t j = g.next() % static_cast<uint64_t>(i + 1);
        std::swap(order[i], order[j]);
      }
    }
    stack.assign(order.rbegin(), order.rend());
    refs.assign(n, 0);
  }
  int64_t free_count() const { return static_cast<int64_t>(stack.size()); }
  int32_t alloc() {
    const int32_t p = stack.back();
    stack.pop_back();
    refs[p] = 1;
    return p;
  }
  void share(int32_t p) { ++refs[p]; }
  void release(int32_t p) {
    if (--refs[p] == 0) stack.push_back(p);
  }
};

struct Request {
  bool used = false;
  std::vector<int32_t> hist_pt;
  int32_t bf16_pt[BF16_PAGES_PER_REQ] = {-1, -1, -1, -1, -1};
  std::vector<int64_t> T;
  std::vector<int64_t> he;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int64_t pages_for(int64_t hist_end) { return hist_end > SINK ? (hist_end - SINK + PAGE - 1) / PAGE : 0; }

}  // namespace

struct oscar_cache {
  oscar_cache_config cfg{};
  bool dry = true;
  char* dev = nullptr;
  oscar_cache_layout lay{};
  DevCache dc{};
  PagePool int2, bf16;
  std::vector<Request> reqs;
  std::string err;
  int num_sms = 152;
  DecodeDebug dbg{DECODE_WAIT_LIMIT, -1};   // failure-detection hooks of decode launches
  uint32_t epoch = 0;                       // decode-step launches so far (never 0 once launched)
  bool last_decode = false;                 // the last kernel this cache launched is a decode

  oscar_status fail(oscar_status s, const std::string& msg) {
    err = msg;
    return s;
  }
  oscar_status cuda_fail(cudaError_t e, const char* what) {
    err = std::string(what) + ": " + cudaGetErrorString(e);
    return OSCAR_ERR_CUDA;
  }
  bool valid_req(int32_t r) const { return r >= 0 && r < cfg.max_requests && reqs[r].used; }
  bool valid_layer(int32_t l) const { return l >= 0 && l < cfg.num_layers; }
  int G() const { return cfg.num_q_heads / cfg.num_kv_heads; }
};

namespace {

bool config_ok(const oscar_cache_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!c) return bad("null config");
  if (c->head_dim != D) return bad("head_dim must be 128");
  if (c->sink_tokens != SINK) return bad("sink_tokens must be 64");
  if (c->recent_tokens != RECENT) return bad("recent_tokens must be 256");
  if (c->page_tokens != PAGE) return bad("page_tokens must be 64");
  if (c->group_size != D && c->group_size != 64) return bad("group_size must be 128 or 64");
  if (c->num_layers < 1 || c->num_kv_heads < 1 || c->num_q_heads < 1) return bad("layer / head counts must be >= 1");
  if (c->num_q_heads % c->num_kv_heads != 0) return bad("num_q_heads must be a multiple of num_kv_heads");
  const int g = c->num_q_heads / c->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return bad("GQA group size must be 1, 2, 4 or 8");
  if (c->max_requests < 1 || c->max_pages_per_request < 1) return bad("max_requests / max_pages_per_request must be >= 1");
  if (c->num_int2_pages < 1 || c->num_int2_pages > INT32_MAX) return bad("num_int2_pages out of range");
  const int64_t nb = c->num_bf16_pages == 0 ? (int64_t)BF16_PAGES_PER_REQ * c->max_requests : c->num_bf16_pages;
  if (nb < BF16_PAGES_PER_REQ || nb > INT32_MAX) return bad("num_bf16_pages out of range");
  if (!(c->softmax_scale >= 0.0f) || !std::isfinite(c->softmax_scale)) return bad("softmax_scale must be finite and >= 0");
  return true;
}

oscar_cache_layout make_layout(const oscar_cache_config& c) {
  oscar_cache_layout l{};
  const size_t L = c.num_layers, H = c.num_kv_heads;
  const size_t nb = c.num_bf16_pages == 0 ? (size_t)BF16_PAGES_PER_REQ * c.max_requests : (size_t)c.num_bf16_pages;
  size_t off = 0;
  l.int2_record_bytes = record_for(c.group_size);
  l.int2_page_stride = H * l.int2_record_bytes;
  l.int2_layer_stride = align256((size_t)c.num_int2_pages * l.int2_page_stride);
  l.int2_pool_offset = off;
  off += L * l.int2_layer_stride;
  l.bf16_record_bytes = (size_t)BF16_RECORD_ELEMS * 2;
  l.bf16_page_stride = H * l.bf16_record_bytes;
  l.bf16_layer_stride = align256(nb * l.bf16_page_stride);
  l.bf16_pool_offset = off;
  off += L * l.bf16_layer_stride;
  const size_t rot = align256(L * H * D * D * sizeof(float));
  l.rot_k_offset = off;
  off += rot;
  l.rot_v_offset = off;
  off += rot;
  l.rot_kt_offset = off;
  off += rot;
  l.rot_vt_offset = off;
  off += rot;
  l.rot_colnorm_offset = off;
  off += align256(2 * L * H * sizeof(float));
  const size_t tau = align256(L * H * sizeof(float));
  l.tau_k_offset = off;
  off += tau;
  l.tau_v_offset = off;
  off += tau;
  l.hist_pt_offset = off;
  off += align256((size_t)c.max_requests * c.max_pages_per_request * sizeof(int32_t));
  l.bf16_pt_offset = off;
  off += align256((size_t)c.max_requests * BF16_PAGES_PER_REQ * sizeof(int32_t));
  l.error_word_offset = off;
  off += 256;
  l.decode_count_offset = off;
  off += align256((size_t)c.max_requests * H * sizeof(int32_t));
  l.decode_flag_offset = off;
  off += align256((size_t)c.max_requests * H * sizeof(uint32_t));
  l.total_bytes = off;
  return l;
}

}  // namespace

extern "C" {

const char* oscar_version(void) { return "oscar-gb300 0.1 (sm_103a)"; }

size_t oscar_cache_device_bytes(const oscar_cache_config* cfg) {
  if (!config_ok(cfg, nullptr)) return 0;
  return make_layout(*cfg).total_bytes;
}

oscar_status oscar_cache_create(const oscar_cache_config* cfg, void* device_mem, size_t device_bytes,
                                const float* rot_k, const float* rot_v, const float* tau_k, const float* tau_v,
                                void* stream, oscar_cache** out) {
  if (!out) return OSCAR_ERR_INVALID_ARG;
  *out = nullptr;
  std::string why;
  if (!config_ok(cfg, &why)) return OSCAR_ERR_INVALID_ARG;
  if (!tau_k || !tau_v) return OSCAR_ERR_INVALID_ARG;
  const size_t LH = (size_t)cfg->num_layers * cfg->num_kv_heads;
  for (size_t i = 0; i < LH; ++i) {
    for (float t : {tau_k[i], tau_v[i]}) {
      if (!(t > 0.0f) || !(t <= 65504.0f)) return OSCAR_ERR_INVALID_ARG;
    }
  }
  oscar_cache* c = new oscar_cache();
  c->cfg = *cfg;
  if (c->cfg.num_bf16_pages == 0) c->cfg.num_bf16_pages = (int64_t)BF16_PAGES_PER_REQ * cfg->max_requests;
  if (c->cfg.softmax_scale == 0.0f) c->cfg.softmax_scale = 1.0f / std::sqrt(static_cast<float>(D));
  c->lay = make_layout(c->cfg);
  c->dry = device_mem == nullptr;
  c->int2.init(c->cfg.num_int2_pages, c->cfg.page_perm_seed);
  c->bf16.init(c->cfg.num_bf16_pages, 0);
  c->reqs.resize(c->cfg.max_requests);

  DevCache& d = c->dc;
  d.L = c->cfg.num_layers;
  d.Hq = c->cfg.num_q_heads;
  d.Hkv = c->cfg.num_kv_heads;
  d.G = c->G();
  d.max_pages = c->cfg.max_pages_per_request;
  d.n_int2_pages = c->cfg.num_int2_pages;
  d.n_bf16_pages = c->cfg.num_bf16_pages;
  d.scale = c->cfg.softmax_scale;
  d.gk = c->cfg.group_size;
  d.record = record_for(c->cfg.group_size);
  if (c->dry) {
    *out = c;
    return OSCAR_OK;
  }
  if (device_bytes < c->lay.total_bytes || (reinterpret_cast<uintptr_t>(device_mem) & 255) != 0 || !rot_k || !rot_v) {
    delete c;
    return OSCAR_ERR_INVALID_ARG;
  }
  char* base = static_cast<char*>(device_mem);
  c->dev = base;
  d.int2 = reinterpret_cast<uint8_t*>(base + c->lay.int2_pool_offset);
  d.int2_layer_stride = c->lay.int2_layer_stride;
  d.bf16 = reinterpret_cast<uint16_t*>(base + c->lay.bf16_pool_offset);
  d.bf16_layer_stride = c->lay.bf16_layer_stride / 2;
  float* rk = reinterpret_cast<float*>(base + c->lay.rot_k_offset);
  float* rv = reinterpret_cast<float*>(base + c->lay.rot_v_offset);
  float* rkt = reinterpret_cast<float*>(base + c->lay.rot_kt_offset);
  float* rvt = reinterpret_cast<float*>(base + c->lay.rot_vt_offset);
  d.rot_k = rk;
  d.rot_v = rv;
  d.rot_kt = rkt;
  d.rot_vt = rvt;
  float* rcn = reinterpret_cast<float*>(base + c->lay.rot_colnorm_offset);
  d.rot_cn = rcn;
  d.tau_k = reinterpret_cast<float*>(base + c->lay.tau_k_offset);
  d.tau_v = reinterpret_cast<float*>(base + c->lay.tau_v_offset);
  d.hist_pt = reinterpret_cast<int32_t*>(base + c->lay.hist_pt_offset);
  d.bf16_pt = reinterpret_cast<int32_t*>(base + c->lay.bf16_pt_offset);
  d.err = reinterpret_cast<int32_t*>(base + c->lay.error_word_offset);
  d.dec_count = reinterpret_cast<int32_t*>(base + c->lay.decode_count_offset);
  d.dec_flag = reinterpret_cast<uint32_t*>(base + c->lay.decode_flag_offset);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(const_cast<float*>(d.tau_k), tau_k, LH * sizeof(float), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(const_cast<float*>(d.tau_v), tau_v, LH * sizeof(float), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(d.hist_pt, 0xff, (size_t)c->cfg.max_requests * c->cfg.max_pages_per_request * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d.bf16_pt, 0xff, (size_t)c->cfg.max_requests * BF16_PAGES_PER_REQ * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d.err, 0, 4, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(d.dec_count, 0, (size_t)c->cfg.max_requests * c->cfg.num_kv_heads * sizeof(int32_t), s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(d.dec_flag, 0, (size_t)c->cfg.max_requests * c->cfg.num_kv_heads * sizeof(uint32_t), s);
  if (e == cudaSuccess) e = launch_rotation_setup(d, rot_k, rot_v, rk, rv, rkt, rvt, rcn, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    delete c;
    return OSCAR_ERR_CUDA;
  }
  *out = c;
  return OSCAR_OK;
}

oscar_status oscar_cache_destroy(oscar_cache* cache) {
  delete cache;
  return OSCAR_OK;
}

oscar_status oscar_cache_get_layout(const oscar_cache* c, oscar_cache_layout* out) {
  if (!c || !out) return OSCAR_ERR_INVALID_ARG;
  *out = c->lay;
  return OSCAR_OK;
}

const char* oscar_last_error(const oscar_cache* c) { return c ? c->err.c_str() : "null cache"; }

oscar_status oscar_cache_free_pages(const oscar_cache* c, int64_t* int2_free, int64_t* bf16_free) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (int2_free) *int2_free = c->int2.free_count();
  if (bf16_free) *bf16_free = c->bf16.free_count();
  return OSCAR_OK;
}

oscar_status oscar_request_open(oscar_cache* c, void* stream, int32_t* req_out) {
  if (!c || !req_out) return OSCAR_ERR_INVALID_ARG;
  int32_t slot = -1;
  for (int32_t i = 0; i < c->cfg.max_requests; ++i)
    if (!c->reqs[i].used) {
      slot = i;
      break;
    }
  if (slot < 0) return c->fail(OSCAR_ERR_OUT_OF_PAGES, "no free request slot");
  if (c->bf16.free_count() < BF16_PAGES_PER_REQ) return c->fail(OSCAR_ERR_OUT_OF_PAGES, "out of BF16 pages");
  Request& r = c->reqs[slot];
  r = Request();
  r.used = true;
  for (int i = 0; i < BF16_PAGES_PER_REQ; ++i) r.bf16_pt[i] = c->bf16.alloc();
  r.T.assign(c->cfg.num_layers, 0);
  r.he.assign(c->cfg.num_layers, SINK);
  *req_out = slot;
  if (c->dry) return OSCAR_OK;
  PtEntry e[BF16_PAGES_PER_REQ];
  for (int i = 0; i < BF16_PAGES_PER_REQ; ++i) e[i] = PtEntry{1, slot * BF16_PAGES_PER_REQ + i, r.bf16_pt[i]};
  c->last_decode = false;
  cudaError_t err = launch_pt_update(c->dc, e, BF16_PAGES_PER_REQ, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OSCAR_OK : c->cuda_fail(err, "page-table update");
}

oscar_status oscar_request_fork(oscar_cache* c, int32_t parent, int64_t prefix, void* stream, int32_t* req_out) {
  if (!c || !req_out) return OSCAR_ERR_INVALID_ARG;
  if (!c->valid_req(parent)) return c->fail(OSCAR_ERR_INVALID_ARG, "bad parent request");
  if (prefix < SINK || (prefix - SINK) % PAGE != 0)
    return c->fail(OSCAR_ERR_INVALID_ARG, "prefix must be 64 plus a multiple of 64");
  const Request& par = c->reqs[parent];
  for (int l = 0; l < c->cfg.num_layers; ++l)
    if (par.he[l] < prefix) return c->fail(OSCAR_ERR_STATE, "parent has not demoted the whole prefix");
  int32_t slot = -1;
  for (int32_t i = 0; i < c->cfg.max_requests; ++i)
    if (!c->reqs[i].used) {
      slot = i;
      break;
    }
  if (slot < 0) return c->fail(OSCAR_ERR_OUT_OF_PAGES, "no free request slot");
  if (c->bf16.free_count() < RING_PAGES) return c->fail(OSCAR_ERR_OUT_OF_PAGES, "out of BF16 pages");
  const int64_t npages = (prefix - SINK) / PAGE;
  Request& r = c->reqs[slot];
  r = Request();
  r.used = true;
  c->bf16.share(par.bf16_pt[0]);
  r.bf16_pt[0] = par.bf16_pt[0];
  for (int i = 1; i < BF16_PAGES_PER_REQ; ++i) r.bf16_pt[i] = c->bf16.alloc();
  for (int64_t i = 0; i < npages; ++i) {
    c->int2.share(par.hist_pt[i]);
    r.hist_pt.push_back(par.hist_pt[i]);
  }
  r.T.assign(c->cfg.num_layers, prefix);
  r.he.assign(c->cfg.num_layers, prefix);
  *req_out = slot;
  if (c->dry) return OSCAR_OK;
  std::vector<PtEntry> e;
  for (int i = 0; i < BF16_PAGES_PER_REQ; ++i) e.push_back(PtEntry{1, slot * BF16_PAGES_PER_REQ + i, r.bf16_pt[i]});
  for (int64_t i = 0; i < npages; ++i)
    e.push_back(PtEntry{0, static_cast<int32_t>((int64_t)slot * c->cfg.max_pages_per_request + i), r.hist_pt[i]});
  c->last_decode = false;
  cudaError_t err = launch_pt_update(c->dc, e.data(), static_cast<int>(e.size()), static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OSCAR_OK : c->cuda_fail(err, "page-table update");
}

oscar_status oscar_request_close(oscar_cache* c, int32_t req) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (!c->valid_req(req)) return c->fail(OSCAR_ERR_INVALID_ARG, "bad request");
  Request& r = c->reqs[req];
  for (int32_t p : r.hist_pt) c->int2.release(p);
  for (int i = 0; i < BF16_PAGES_PER_REQ; ++i) c->bf16.release(r.bf16_pt[i]);
  r = Request();
  return OSCAR_OK;
}

oscar_status oscar_request_length(const oscar_cache* c, int32_t req, int32_t layer, int64_t* tokens,
                                  int64_t* hist_end) {
  if (!c || !c->valid_req(req) || !c->valid_layer(layer)) return OSCAR_ERR_INVALID_ARG;
  if (tokens) *tokens = c->reqs[req].T[layer];
  if (hist_end) *hist_end = c->reqs[req].he[layer];
  return OSCAR_OK;
}

oscar_status oscar_request_pages(const oscar_cache* c, int32_t req, int32_t* hist_pt_out, int32_t cap,
                                 int32_t* num_pages, int32_t* bf16_pt_out) {
  if (!c || !c->valid_req(req)) return OSCAR_ERR_INVALID_ARG;
  const Request& r = c->reqs[req];
  if (num_pages) *num_pages = static_cast<int32_t>(r.hist_pt.size());
  if (hist_pt_out)
    for (int32_t i = 0; i < cap && i < (int32_t)r.hist_pt.size(); ++i) hist_pt_out[i] = r.hist_pt[i];
  if (bf16_pt_out)
    for (int i = 0; i < BF16_PAGES_PER_REQ; ++i) bf16_pt_out[i] = r.bf16_pt[i];
  return OSCAR_OK;
}

oscar_status oscar_prefill_quantize(oscar_cache* c, int32_t req, int32_t layer, const uint16_t* k, const uint16_t* v,
                                    int64_t n, void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (!c->valid_req(req) || !c->valid_layer(layer) || n < 1) return c->fail(OSCAR_ERR_INVALID_ARG, "bad request, layer or length");
  if (!c->dry && (!k || !v || !aligned16(k) || !aligned16(v)))
    return c->fail(OSCAR_ERR_INVALID_ARG, "null or misaligned k / v");
  Request& r = c->reqs[req];
  const int64_t t0 = r.T[layer], he0 = r.he[layer];
  if (!(t0 == 0 || (t0 >= SINK && he0 == t0))) return c->fail(OSCAR_ERR_STATE, "prefill needs an empty recent window");
  const int64_t total = t0 + n;
  const int64_t he1 = std::max<int64_t>({he0, total - RECENT, (int64_t)SINK});
  const int64_t need = pages_for(he1);
  if (need > c->cfg.max_pages_per_request) return c->fail(OSCAR_ERR_INVALID_ARG, "request exceeds its page table");
  const int64_t fresh = std::max<int64_t>(0, need - (int64_t)r.hist_pt.size());
  if (fresh > c->int2.free_count()) return c->fail(OSCAR_ERR_OUT_OF_PAGES, "out of INT2 pages");
  std::vector<PtEntry> e;
  while ((int64_t)r.hist_pt.size() < need) {
    const int32_t p = c->int2.alloc();
    e.push_back(PtEntry{0, static_cast<int32_t>((int64_t)req * c->cfg.max_pages_per_request + r.hist_pt.size()), p});
    r.hist_pt.push_back(p);
  }
  r.T[layer] = total;
  r.he[layer] = he1;
  if (c->dry) return OSCAR_ERR_DRY_RUN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  BF16Dest dst;
  dst.sink_page = r.bf16_pt[0];
  for (int i = 0; i < RING_PAGES; ++i) dst.ring_page[i] = r.bf16_pt[1 + i];
  c->last_decode = false;
  cudaError_t err = launch_pt_update(c->dc, e.data(), static_cast<int>(e.size()), s);
  if (err == cudaSuccess && t0 < SINK) err = launch_prefill_bf16(c->dc, layer, k, v, t0, t0, std::min<int64_t>(total, SINK), dst, s);
  const int64_t r0 = std::max<int64_t>(he1, SINK);
  if (err == cudaSuccess && total > r0) err = launch_prefill_bf16(c->dc, layer, k, v, t0, r0, total, dst, s);
  const int64_t h0 = std::max<int64_t>(t0, SINK);
  if (err == cudaSuccess && he1 > h0) err = launch_prefill_hist(c->dc, layer, req, k, v, t0, h0, he1, s);
  return err == cudaSuccess ? OSCAR_OK : c->cuda_fail(err, "prefill launch");
}

namespace {

// Shared by append and demote: validate a batch, then apply it.
// Append / demote of a batch in two halves: every check first (no side effect),
// then the page allocation and state update, which cannot fail.
oscar_status validate_write(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, const uint16_t* k,
                            const uint16_t* v, bool append) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (!c->valid_layer(layer) || n < 1 || !reqs) return c->fail(OSCAR_ERR_INVALID_ARG, "bad layer or batch");
  if (append && !c->dry && (!k || !v || !aligned16(k) || !aligned16(v)))
    return c->fail(OSCAR_ERR_INVALID_ARG, "null or misaligned k / v");
  std::vector<char> seen(c->cfg.max_requests, 0);
  int64_t fresh = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t q = reqs[i];
    if (!c->valid_req(q)) return c->fail(OSCAR_ERR_INVALID_ARG, "bad request id");
    if (seen[q]) return c->fail(OSCAR_ERR_INVALID_ARG, "duplicate request id");
    seen[q] = 1;
    const Request& r = c->reqs[q];
    const int64_t T = r.T[layer], he = r.he[layer];
    bool demote;
    if (append) {
      demote = T >= SINK && T - he == RECENT;
    } else {
      if (T <= SINK || he >= T) return c->fail(OSCAR_ERR_STATE, "recent window is empty");
      demote = true;
    }
    if (demote) {
      const int64_t need = pages_for(he + 1);
      if (need > c->cfg.max_pages_per_request) return c->fail(OSCAR_ERR_INVALID_ARG, "request exceeds its page table");
      fresh += std::max<int64_t>(0, need - (int64_t)r.hist_pt.size());
    }
  }
  if (fresh > c->int2.free_count()) return c->fail(OSCAR_ERR_OUT_OF_PAGES, "out of INT2 pages");
  return OSCAR_OK;
}

std::vector<AppendReq> apply_write(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, bool append) {
  std::vector<AppendReq> work(n);
  for (int32_t i = 0; i < n; ++i) {
    Request& r = c->reqs[reqs[i]];
    const int64_t T = r.T[layer], he = r.he[layer];
    AppendReq& a = work[i];
    a.slot = reqs[i];
    a.in_row = append ? i : -1;
    a.dst_page = a.dst_row = -1;
    a.demote_slot = a.hist_page = a.src_page = a.src_row = a.pt_index = -1;
    const bool demote = append ? (T >= SINK && T - he == RECENT) : true;
    if (demote) {
      const int64_t h = he - SINK;
      const int64_t idx = h / PAGE;
      if ((int64_t)r.hist_pt.size() <= idx) {
        r.hist_pt.push_back(c->int2.alloc());
        a.pt_index = static_cast<int32_t>(idx);
      }
      a.hist_page = r.hist_pt[idx];
      a.demote_slot = static_cast<int32_t>(h % PAGE);
      const int64_t slot = (he - SINK) % RECENT;
      a.src_page = r.bf16_pt[1 + slot / PAGE];
      a.src_row = static_cast<int32_t>(slot % PAGE);
      r.he[layer] = he + 1;
    }
    if (append) {
      if (T < SINK) {
        a.dst_page = r.bf16_pt[0];
        a.dst_row = static_cast<int32_t>(T);
      } else {
        const int64_t slot = (T - SINK) % RECENT;
        a.dst_page = r.bf16_pt[1 + slot / PAGE];
        a.dst_row = static_cast<int32_t>(slot % PAGE);
      }
      r.T[layer] = T + 1;
    }
  }
  return work;
}

oscar_status write_batch(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, const uint16_t* k,
                         const uint16_t* v, bool append, void* stream) {
  const oscar_status st = validate_write(c, layer, n, reqs, k, v, append);
  if (st != OSCAR_OK) return st;
  const std::vector<AppendReq> work = apply_write(c, layer, n, reqs, append);
  if (c->dry) return OSCAR_ERR_DRY_RUN;
  c->last_decode = false;
  cudaError_t err = launch_append(c->dc, layer, work.data(), n, k, v, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OSCAR_OK : c->cuda_fail(err, append ? "append launch" : "demote launch");
}

// Work split of one decode launch over reqs[0..n), n <= DECODE_PER_LAUNCH: nbc
// CTAs for the segments' BF16 blocks (and, in a decode step, their appends),
// sized so that this work takes about one CTA's share of the INT2 cost each
// (DECODE_BF16_BLOCK_COST, DECODE_APPEND_COST), at least one and at most one per
// segment; the other CTAs (one per SM in all, at most one per INT2 cost unit)
// split the INT2 line into contiguous equal ranges.
DecodePlan plan_decode(const oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, int32_t first_row,
                       DecodeReq* out, bool step = false) {
  const int64_t H = c->cfg.num_kv_heads;
  int64_t cost = 0;
  for (int32_t i = 0; i < n; ++i) {
    const Request& r = c->reqs[reqs[i]];
    const int64_t T = r.T[layer], he = r.he[layer];
    const int64_t np = pages_for(he);
    if (out) {
      DecodeReq& d = out[i];
      d.slot = reqs[i];
      d.batch_row = first_row + i;
      d.tokens = static_cast<int32_t>(T);
      d.hist_end = static_cast<int32_t>(he);
      d.sink_page = r.bf16_pt[0];
      for (int k = 0; k < RING_PAGES; ++k) d.ring_page[k] = r.bf16_pt[1 + k];
      d.hot_page = -1;
      d.hot_new = -1;
      d.npages = static_cast<int32_t>(np);
      d.cost_start = static_cast<int32_t>(cost);
    }
    cost += H * (np > 0 ? np + DECODE_SEGMENT_SETUP_COST : 0);
  }
  DecodePlan p{};
  p.n = n;
  p.total_cost = cost;
  p.segments = (int64_t)n * H;
  const int64_t sms = std::max(2, c->num_sms);
  const int64_t share = cost / sms + 1;   // INT2 cost per CTA were every CTA on INT2 pages
  // a decode step's BF16 CTAs also append the new token of each segment first
  const int64_t per_seg = DECODE_BF16_BLOCK_COST + (step ? DECODE_APPEND_COST : 0);
  int64_t nbc = (p.segments * per_seg + share - 1) / share;
  // few segments: one BF16 CTA each, which then also merges its segment (the
  // INT2 CTAs only count), however short its BF16 work
  if (p.segments * 8 <= sms) nbc = std::max(nbc, p.segments);
  nbc = std::max<int64_t>(1, std::min<int64_t>({nbc, p.segments, cost > 0 ? sms / 2 : sms}));
  const int64_t n_int2 = std::min<int64_t>({sms - nbc, cost, (int64_t)DECODE_MAX_INT2});
  p.nbc = static_cast<int>(nbc);
  p.ncta = static_cast<int>(nbc + n_int2);
  p.partial_bytes = align256((size_t)(2 * p.segments + p.ncta) * decode_record_bytes(c->G()));
  return p;
}

// Requests per decode launch.
int32_t decode_launch_size(const oscar_cache*, int32_t, int32_t n, const int32_t*) {
  return std::min<int32_t>(n, DECODE_PER_LAUNCH);
}

// Workspace of a decode of n requests, whatever their lengths: per launch an INT2
// and a BF16 record per (request, kv head), and one INT2 record per CTA (one per SM).
size_t decode_bytes_bound(const oscar_cache* c, int32_t n) {
  const int64_t segs = (int64_t)std::min<int32_t>(n, DECODE_PER_LAUNCH) * c->cfg.num_kv_heads;
  return align256((size_t)(2 * segs + (int64_t)c->num_sms) * decode_record_bytes(c->G()));
}

size_t decode_bytes_needed(const oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs) {
  size_t need = 0;
  const int32_t per = decode_launch_size(c, layer, n, reqs);
  for (int32_t b = 0; b < n; b += per) {
    const int32_t m = std::min<int32_t>(per, n - b);
    need = std::max(need, plan_decode(c, layer, m, reqs + b, b, nullptr).partial_bytes);
  }
  return need;
}

oscar_status check_decode_batch(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs) {
  if (!c->valid_layer(layer) || n < 1 || !reqs) return c->fail(OSCAR_ERR_INVALID_ARG, "bad layer or batch");
  std::vector<char> seen(c->cfg.max_requests, 0);
  for (int32_t i = 0; i < n; ++i) {
    if (!c->valid_req(reqs[i])) return c->fail(OSCAR_ERR_INVALID_ARG, "bad request id");
    // each (request, kv head) of a launch owns one merge counter
    if (seen[reqs[i]]) return c->fail(OSCAR_ERR_INVALID_ARG, "duplicate request id");
    seen[reqs[i]] = 1;
    if (c->reqs[reqs[i]].T[layer] < 1) return c->fail(OSCAR_ERR_STATE, "request has no cached tokens");
    if (c->reqs[reqs[i]].T[layer] > INT32_MAX) return c->fail(OSCAR_ERR_INVALID_ARG, "request too long");
  }
  return OSCAR_OK;
}

}  // namespace

oscar_status oscar_append(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, const uint16_t* k,
                          const uint16_t* v, void* stream) {
  return write_batch(c, layer, n, reqs, k, v, true, stream);
}

oscar_status oscar_demote(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, void* stream) {
  return write_batch(c, layer, n, reqs, nullptr, nullptr, false, stream);
}

// Every layer's checks first (a page opened by one layer is reused by the
// others, so checking each layer against the current free count is enough),
// then each layer's state change in order, then the launches.
oscar_status oscar_demote_layers(oscar_cache* c, int32_t layer_begin, int32_t layer_end, int32_t n,
                                 const int32_t* reqs, void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (layer_begin < 0 || layer_end > c->cfg.num_layers || layer_begin >= layer_end)
    return c->fail(OSCAR_ERR_INVALID_ARG, "bad layer range");
  for (int32_t l = layer_begin; l < layer_end; ++l) {
    const oscar_status st = validate_write(c, l, n, reqs, nullptr, nullptr, false);
    if (st != OSCAR_OK) return st;
  }
  std::vector<DemoteEntry> work;
  work.reserve((size_t)n * (size_t)(layer_end - layer_begin));
  for (int32_t l = layer_begin; l < layer_end; ++l)
    for (const AppendReq& a : apply_write(c, l, n, reqs, false)) work.push_back(DemoteEntry{l, a});
  if (c->dry) return OSCAR_ERR_DRY_RUN;
  c->last_decode = false;
  const cudaError_t err =
      launch_demote_layers(c->dc, work.data(), static_cast<int>(work.size()), static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OSCAR_OK : c->cuda_fail(err, "demote launch");
}

oscar_status oscar_decode_workspace_bytes(const oscar_cache* c, int32_t n, const int32_t* reqs, size_t* bytes) {
  if (!c || !bytes) return OSCAR_ERR_INVALID_ARG;
  oscar_cache* mc = const_cast<oscar_cache*>(c);
  for (int32_t l = 0; l < c->cfg.num_layers; ++l) {
    const oscar_status st = check_decode_batch(mc, l, n, reqs);
    if (st != OSCAR_OK && st != OSCAR_ERR_STATE) return st;
  }
  // the records depend only on the batch and the CTA count, not on the lengths:
  // this size holds after any number of appends
  *bytes = decode_bytes_bound(c, n);
  return OSCAR_OK;
}

oscar_status oscar_decode_attention(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, const uint16_t* q,
                                    float* out, void* workspace, size_t ws_bytes, void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  oscar_status st = check_decode_batch(c, layer, n, reqs);
  if (st != OSCAR_OK) return st;
  if (c->dry) return OSCAR_ERR_DRY_RUN;
  if (!q || !out || !workspace || !aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return c->fail(OSCAR_ERR_INVALID_ARG, "null or misaligned q / out / workspace");
  if (decode_bytes_needed(c, layer, n, reqs) > ws_bytes) return c->fail(OSCAR_ERR_INVALID_ARG, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DecodeReq dr[DECODE_PER_LAUNCH];
  const int32_t per = decode_launch_size(c, layer, n, reqs);
  for (int32_t b = 0; b < n; b += per) {
    const int32_t m = std::min<int32_t>(per, n - b);
    const DecodePlan p = plan_decode(c, layer, m, reqs + b, b, dr);
    const cudaError_t err =
        launch_decode(c->dc, layer, dr, p, q, out, workspace, nullptr, nullptr, 0u, c->last_decode, c->dbg, s);
    c->last_decode = err == cudaSuccess;
    if (err != cudaSuccess) return c->cuda_fail(err, "decode launch");
  }
  return OSCAR_OK;
}

// Same decode, with the partial records in the library's fixed static scratch
// (decode_scratch.cu) instead of a caller workspace, for callers that cannot
// allocate device memory around a step.
oscar_status oscar_decode_attention_noalloc(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs,
                                            const uint16_t* q, float* out, void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  const oscar_status st = check_decode_batch(c, layer, n, reqs);
  if (st != OSCAR_OK) return st;
  const size_t need = decode_bytes_needed(c, layer, n, reqs);
  if (need > DECODE_SCRATCH_BYTES) {
    char msg[192];
    std::snprintf(msg, sizeof msg,
                  "batch needs %zu bytes of decode scratch, above the fixed %zu; "
                  "use oscar_decode_attention with a caller workspace",
                  need, DECODE_SCRATCH_BYTES);
    return c->fail(OSCAR_ERR_INVALID_ARG, msg);
  }
  if (c->dry) return OSCAR_ERR_DRY_RUN;
  void* scratch = nullptr;
  const cudaError_t e = decode_scratch_address(&scratch, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return c->cuda_fail(e, "decode scratch set-up");
  return oscar_decode_attention(c, layer, n, reqs, q, out, scratch, DECODE_SCRATCH_BYTES, stream);
}

oscar_status oscar_decode_step(oscar_cache* c, int32_t layer, int32_t n, const int32_t* reqs, const uint16_t* k,
                               const uint16_t* v, const uint16_t* q, float* out, void* workspace, size_t ws_bytes,
                               void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (!c->dry && (!q || !out || !workspace || !aligned16(q) || !aligned16(out) ||
                  (reinterpret_cast<uintptr_t>(workspace) & 255) != 0))
    return c->fail(OSCAR_ERR_INVALID_ARG, "null or misaligned q / out / workspace");
  oscar_status st = validate_write(c, layer, n, reqs, k, v, true);
  if (st != OSCAR_OK) return st;
  // the decode after the append needs one record per (segment, CTA) and the BF16
  // records: the same count before and after the append, checked before any change
  for (int32_t i = 0; i < n; ++i)
    if (c->reqs[reqs[i]].T[layer] + 1 > INT32_MAX) return c->fail(OSCAR_ERR_INVALID_ARG, "request too long");
  if (!c->dry && decode_bytes_bound(c, std::min<int32_t>(n, APPEND_PER_LAUNCH)) > ws_bytes)
    return c->fail(OSCAR_ERR_INVALID_ARG, "workspace too small");
  const std::vector<AppendReq> work = apply_write(c, layer, n, reqs, true);
  if (c->dry) return OSCAR_ERR_DRY_RUN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DecodeReq dr[DECODE_PER_LAUNCH];
  const int32_t per = std::min<int32_t>(APPEND_PER_LAUNCH, decode_launch_size(c, layer, n, reqs));
  for (int32_t b = 0; b < n; b += per) {
    const int32_t m = std::min<int32_t>(per, n - b);
    const DecodePlan p = plan_decode(c, layer, m, reqs + b, b, dr, true);
    for (int32_t i = 0; i < m; ++i) {
      const AppendReq& a = work[b + i];
      if (a.demote_slot >= 0) {
        dr[i].hot_page = static_cast<int32_t>((c->reqs[reqs[b + i]].he[layer] - 1 - SINK) / PAGE);
        dr[i].hot_new = a.pt_index >= 0 ? a.hist_page : -1;
      }
    }
    if (++c->epoch == 0) c->epoch = 1;
    const cudaError_t err =
        launch_decode(c->dc, layer, dr, p, q, out, workspace, k, v, c->epoch, c->last_decode, c->dbg, s);
    c->last_decode = err == cudaSuccess;
    if (err != cudaSuccess) return c->cuda_fail(err, "decode step launch");
  }
  return OSCAR_OK;
}

oscar_status oscar_debug_decode_hooks(oscar_cache* c, uint32_t wait_limit, int32_t hold_copy) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  // the device's other bounded waits take multiples of wait_limit in 32 bits
  if (wait_limit < 1 || wait_limit > (1u << 24) || hold_copy < -1)
    return c->fail(OSCAR_ERR_INVALID_ARG, "bad hook values");
  c->dbg.wait_limit = wait_limit;
  c->dbg.hold_copy = hold_copy;
  return OSCAR_OK;
}

oscar_status oscar_cache_check(oscar_cache* c, void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (c->dry) return OSCAR_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return c->cuda_fail(e, "stream synchronize");
  int32_t word = 0;
  e = cudaMemcpy(&word, c->dc.err, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return c->cuda_fail(e, "error word read");
  if (word != 0) {
    const int32_t zero = 0;
    cudaMemcpy(c->dc.err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    // a launch that reported an error still counts every segment to the end, but
    // the merge counters are cleared as well so that no count can carry over
    cudaMemset(c->dc.dec_count, 0, (size_t)c->cfg.max_requests * c->cfg.num_kv_heads * sizeof(int32_t));
    char msg[160];
    std::snprintf(msg, sizeof msg,
                  "device check failed: error bits 0x%x (1 INT2 page, 2 BF16 page, 4 length, 8 wait timed out)",
                  word);
    return c->fail((word & ERR_TIMEOUT) ? OSCAR_ERR_TIMEOUT : OSCAR_ERR_DEVICE_CHECK, msg);
  }
  return OSCAR_OK;
}

}  // extern "C"
