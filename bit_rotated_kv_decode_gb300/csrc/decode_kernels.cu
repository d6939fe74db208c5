// Three-segment decode attention.
//
// "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计": at decode time the
// INT2 history is unpacked, dequantised with its scale / zero point and
// accumulated in floating point; the BF16 sink and recent window are handled
// separately; the partials are merged with an online softmax (max / sum).
// "Together AI Open-Sources OSCAR" (MarkTechPost), section "The Serving
// System": the value path is inverse-rotated.
//
// One launch per layer.  Work items, per (request, kv head):
//   item 0      the BF16 sink + recent tokens, with the unrotated q;
//   items 1..C  chunks of INT2 history pages, in the rotated basis: q is
//               rotated by R_K, and for token j with codes c_j, scale s_j,
//               zero z_j the logit is scale * (s_j (q_rot . c_j) + z_j sum(q_rot))
//               and the value contribution is p_j (s_j c_j + z_j 1).
// Every item writes an (m, l, o[128]) partial per query head of the GQA group
// (log2-domain max m).  The last item of a (request, kv head) to finish --
// decided by an atomic ticket, no waiting -- merges the partials, applies R_V^T
// to the history part and writes out = (O_bf16 + O_hist R_V^T) / L.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int PART = PARTIAL_FLOATS;

struct DecodeArgs {
  int n;
  int pages_per_chunk;
  DecodeReq r[DECODE_PER_LAUNCH];
};

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

struct Online {
  float m;          // running max (log2 domain)
  float l;          // this lane's part of the running sum
  float o[4];       // this lane's 4 output channels
  float u;          // running sum of p_j z_j (INT2 items only)
};

// Rescale the running state to a new maximum; returns the new max.
__device__ __forceinline__ float online_rescale(Online& st, float page_max) {
  const float m_new = fmaxf(st.m, page_max);
  const float corr = (st.m == -INFINITY) ? 0.0f : exp2f(st.m - m_new);
  st.l *= corr;
  st.u *= corr;
#pragma unroll
  for (int i = 0; i < 4; ++i) st.o[i] *= corr;
  st.m = m_new;
  return m_new;
}

template <int G>
struct Smem {
  float q[G][D];
  float qsum[G];
  float w[G][PAGE];
  float u[G][PAGE];
  float oh[G][D];
  int ticket;
  union {
    __align__(16) uint8_t rec[RECORD];
    struct {
      __align__(16) uint16_t k[PAGE][D];
      __align__(16) uint16_t v[PAGE][D];
    } bf;
  } buf;
};

template <int G>
__global__ void __launch_bounds__(32 * G) decode_kernel(DevCache c, int layer, DecodeArgs a,
                                                        const uint16_t* __restrict__ q, float* __restrict__ out,
                                                        int32_t* counters, float* partials) {
  __shared__ Smem<G> sm;
  const int item = blockIdx.x;
  int ri = 0;
  while (ri + 1 < a.n && a.r[ri + 1].item_start <= item) ++ri;
  const DecodeReq R = a.r[ri];
  const int local = item - R.item_start;
  const int per_head = 1 + R.chunks;
  const int head = local / per_head;
  const int sub = local % per_head;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qh = head * G + warp;
  const size_t lh = (size_t)layer * c.Hkv + head;
  const float scale2 = c.scale * LOG2E;

  // q of this warp's head (bf16 -> fp32)
  const uint16_t* qrow = q + ((size_t)R.batch_row * c.Hq + qh) * D;
  for (int i = lane; i < D; i += 32) sm.q[warp][i] = bf16f(qrow[i]);
  __syncwarp();

  Online st;
  st.m = -INFINITY;
  st.l = 0.0f;
  st.u = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) st.o[i] = 0.0f;

  if (sub == 0) {
    // ---- BF16 sink + recent window, unrotated basis ------------------------
    const int T = R.tokens;
    const int nsink = T < SINK ? T : SINK;
    const int rec_lo = T > SINK ? R.hist_end : T;   // recent = [hist_end, T)
    const int nrec = T - rec_lo;
    const int ntot = nsink + nrec;
    for (int base = 0; base < ntot; base += PAGE) {
      const int cnt = min(PAGE, ntot - base);
      __syncthreads();
      for (int idx = threadIdx.x; idx < cnt * (D / 8); idx += blockDim.x) {
        const int j = idx / (D / 8);
        const int part = idx % (D / 8);
        const int t = base + j;
        int page, row;
        if (t < nsink) {
          page = R.sink_page;
          row = t;
        } else {
          const int p = rec_lo + (t - nsink);
          const int slot = (p - SINK) % RECENT;
          page = R.ring_page[slot / PAGE];
          row = slot % PAGE;
        }
        if (page < 0 || page >= c.n_bf16_pages) {
          atomicOr(c.err, ERR_BF16_PAGE);
          page = 0;
        }
        const uint16_t* src = c.bf16 + layer * c.bf16_layer_stride + ((size_t)page * c.Hkv + head) * BF16_RECORD_ELEMS;
        const uint4 kk = reinterpret_cast<const uint4*>(src + (size_t)row * D)[part];
        const uint4 vv = reinterpret_cast<const uint4*>(src + (size_t)(PAGE + row) * D)[part];
        // K rows are stored with their 16-byte chunks XOR-swizzled by the row
        reinterpret_cast<uint4*>(&sm.buf.bf.k[j][0])[part ^ (j & 15)] = kk;
        reinterpret_cast<uint4*>(&sm.buf.bf.v[j][0])[part] = vv;
      }
      __syncthreads();
      float lg[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int j = lane + 32 * h2;
        float dot = 0.0f;
        if (j < cnt) {
          const uint4* kr = reinterpret_cast<const uint4*>(&sm.buf.bf.k[j][0]);
#pragma unroll
          for (int b = 0; b < D / 8; ++b) {
            const uint4 w = kr[b ^ (j & 15)];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              dot = fmaf(sm.q[warp][8 * b + 2 * e], __uint_as_float(ww[e] << 16), dot);
              dot = fmaf(sm.q[warp][8 * b + 2 * e + 1], __uint_as_float(ww[e] & 0xffff0000u), dot);
            }
          }
          lg[h2] = dot * scale2;
        } else {
          lg[h2] = -INFINITY;
        }
      }
      const float m_new = online_rescale(st, warp_max(fmaxf(lg[0], lg[1])));
      const float p0 = exp2f(lg[0] - m_new);
      const float p1 = exp2f(lg[1] - m_new);
      st.l += p0 + p1;
      sm.w[warp][lane] = p0;
      sm.w[warp][lane + 32] = p1;
      __syncwarp();
      for (int j = 0; j < cnt; ++j) {
        const float p = sm.w[warp][j];
        const uint2 vv = reinterpret_cast<const uint2*>(&sm.buf.bf.v[j][0])[lane];
        st.o[0] = fmaf(p, __uint_as_float(vv.x << 16), st.o[0]);
        st.o[1] = fmaf(p, __uint_as_float(vv.x & 0xffff0000u), st.o[1]);
        st.o[2] = fmaf(p, __uint_as_float(vv.y << 16), st.o[2]);
        st.o[3] = fmaf(p, __uint_as_float(vv.y & 0xffff0000u), st.o[3]);
      }
      __syncwarp();
    }
  } else {
    // ---- INT2 history chunk, rotated basis ----------------------------------
    // q_rot = q R_K: lane computes channels 4 lane .. 4 lane + 3
    const float* __restrict__ RK = c.rot_k + lh * D * D;
    float qr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int i = 0; i < D; ++i) {
      const float qi = sm.q[warp][i];
      const float4 r = __ldg(reinterpret_cast<const float4*>(RK + (size_t)i * D) + lane);
      qr[0] = fmaf(qi, r.x, qr[0]);
      qr[1] = fmaf(qi, r.y, qr[1]);
      qr[2] = fmaf(qi, r.z, qr[2]);
      qr[3] = fmaf(qi, r.w, qr[3]);
    }
    const float qs = warp_sum(qr[0] + qr[1] + qr[2] + qr[3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) sm.q[warp][4 * lane + i] = qr[i];
    __syncwarp();

    const int nhist = R.hist_end - SINK;
    const int npages = (nhist + PAGE - 1) / PAGE;
    const int pc0 = (sub - 1) * a.pages_per_chunk;
    const int pc1 = min(npages, pc0 + a.pages_per_chunk);
    const int32_t* pt = c.hist_pt + (size_t)R.slot * c.max_pages;
    for (int pi = pc0; pi < pc1; ++pi) {
      const int valid = min(PAGE, nhist - pi * PAGE);
      int32_t page = pt[pi];
      __syncthreads();
      if (page < 0 || page >= c.n_int2_pages) {
        if (threadIdx.x == 0) atomicOr(c.err, ERR_INT2_PAGE);
        page = 0;
      }
      const uint4* src = reinterpret_cast<const uint4*>(c.int2 + layer * c.int2_layer_stride +
                                                        ((size_t)page * c.Hkv + head) * RECORD);
      for (int idx = threadIdx.x; idx < RECORD / 16; idx += blockDim.x)
        reinterpret_cast<uint4*>(sm.buf.rec)[idx] = src[idx];
      __syncthreads();

      float lg[2];
      float sv[2], zv[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int j = lane + 32 * h2;
        const uint32_t km = *reinterpret_cast<const uint32_t*>(sm.buf.rec + K_META_OFF + j * META_BYTES);
        const uint32_t vm = *reinterpret_cast<const uint32_t*>(sm.buf.rec + V_META_OFF + j * META_BYTES);
        sv[h2] = 0.0f;
        zv[h2] = 0.0f;
        if (j < valid) {
          // slots past the last demoted token hold stale bytes: never read them
          sv[h2] = __half2float(__ushort_as_half(static_cast<uint16_t>(vm & 0xffff)));
          zv[h2] = __half2float(__ushort_as_half(static_cast<uint16_t>(vm >> 16)));
          const float sk = __half2float(__ushort_as_half(static_cast<uint16_t>(km & 0xffff)));
          const float zk = __half2float(__ushort_as_half(static_cast<uint16_t>(km >> 16)));
          const uint4* cr = reinterpret_cast<const uint4*>(sm.buf.rec + K_CODES_OFF + j * CODE_BYTES);
          float dot = 0.0f;
#pragma unroll
          for (int half16 = 0; half16 < 2; ++half16) {
            const uint4 w = cr[half16];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
#pragma unroll
              for (int bit = 0; bit < 16; ++bit) {
                const int ch = 64 * half16 + 16 * e + bit;
                dot = fmaf(sm.q[warp][ch], static_cast<float>((ww[e] >> (2 * bit)) & 3u), dot);
              }
            }
          }
          lg[h2] = scale2 * fmaf(sk, dot, zk * qs);
        } else {
          lg[h2] = -INFINITY;
        }
      }
      const float m_new = online_rescale(st, warp_max(fmaxf(lg[0], lg[1])));
      const float p0 = exp2f(lg[0] - m_new);
      const float p1 = exp2f(lg[1] - m_new);
      st.l += p0 + p1;
      sm.w[warp][lane] = p0 * sv[0];
      sm.w[warp][lane + 32] = p1 * sv[1];
      st.u += p0 * zv[0] + p1 * zv[1];     // summed over lanes at the end
      __syncwarp();
      for (int j = 0; j < valid; ++j) {
        const float w = sm.w[warp][j];
        const uint32_t byte = sm.buf.rec[V_CODES_OFF + j * CODE_BYTES + lane];
        st.o[0] = fmaf(w, static_cast<float>(byte & 3u), st.o[0]);
        st.o[1] = fmaf(w, static_cast<float>((byte >> 2) & 3u), st.o[1]);
        st.o[2] = fmaf(w, static_cast<float>((byte >> 4) & 3u), st.o[2]);
        st.o[3] = fmaf(w, static_cast<float>((byte >> 6) & 3u), st.o[3]);
      }
      __syncwarp();
    }
    const float usum = warp_sum(st.u);
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[i] += usum;
  }

  // ---- write this item's partial for the warp's query head ----------------------
  const float lsum = warp_sum(st.l);
  float* part = partials + ((size_t)item * G + warp) * PART;
  if (lane == 0) {
    part[PARTIAL_M] = st.m;
    part[PARTIAL_L] = lsum;
  }
  reinterpret_cast<float4*>(part)[lane] = make_float4(st.o[0], st.o[1], st.o[2], st.o[3]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sm.ticket = atomicAdd(counters + ri * c.Hkv + head, 1);
  __syncthreads();
  if (sm.ticket != per_head - 1) return;
  __threadfence();

  // ---- last item of this (request, kv head): merge --------------------------------
  const int first = R.item_start + head * per_head;
  float M = -INFINITY;
  for (int k = 0; k < per_head; ++k) M = fmaxf(M, __ldcg(partials + ((size_t)(first + k) * G + warp) * PART + PARTIAL_M));
  float L = 0.0f;
  float ob[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float ohist[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int k = 0; k < per_head; ++k) {
    const float* pk = partials + ((size_t)(first + k) * G + warp) * PART;
    const float mk = __ldcg(pk + PARTIAL_M);
    if (mk == -INFINITY) continue;
    const float f = exp2f(mk - M);
    L = fmaf(__ldcg(pk + PARTIAL_L), f, L);
    const float4 ok = __ldcg(reinterpret_cast<const float4*>(pk) + lane);
    float* dst = (k == 0) ? ob : ohist;
    dst[0] = fmaf(ok.x, f, dst[0]);
    dst[1] = fmaf(ok.y, f, dst[1]);
    dst[2] = fmaf(ok.z, f, dst[2]);
    dst[3] = fmaf(ok.w, f, dst[3]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) sm.oh[warp][4 * lane + i] = ohist[i];
  __syncwarp();
  // out_c = O_bf16_c + sum_j O_hist_j R_V[c][j]; rot_vt[j][c] = R_V[c][j]
  const float* __restrict__ RVt = c.rot_vt + lh * D * D;
  for (int j = 0; j < D; ++j) {
    const float oj = sm.oh[warp][j];
    const float4 r = __ldg(reinterpret_cast<const float4*>(RVt + (size_t)j * D) + lane);
    ob[0] = fmaf(oj, r.x, ob[0]);
    ob[1] = fmaf(oj, r.y, ob[1]);
    ob[2] = fmaf(oj, r.z, ob[2]);
    ob[3] = fmaf(oj, r.w, ob[3]);
  }
  const float inv = 1.0f / L;
  float* orow = out + ((size_t)R.batch_row * c.Hq + qh) * D;
  reinterpret_cast<float4*>(orow)[lane] = make_float4(ob[0] * inv, ob[1] * inv, ob[2] * inv, ob[3] * inv);
  if (threadIdx.x == 0) counters[ri * c.Hkv + head] = 0;
}

}  // namespace

cudaError_t launch_decode(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& plan,
                          const uint16_t* q, float* out, void* workspace, cudaStream_t s) {
  DecodeArgs a;
  a.n = plan.n;
  a.pages_per_chunk = plan.pages_per_chunk;
  for (int i = 0; i < plan.n; ++i) a.r[i] = reqs[i];
  int32_t* counters = static_cast<int32_t*>(workspace);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.counter_bytes);
  switch (c.G) {
    case 1: decode_kernel<1><<<plan.total_items, 32, 0, s>>>(c, layer, a, q, out, counters, partials); break;
    case 2: decode_kernel<2><<<plan.total_items, 64, 0, s>>>(c, layer, a, q, out, counters, partials); break;
    case 4: decode_kernel<4><<<plan.total_items, 128, 0, s>>>(c, layer, a, q, out, counters, partials); break;
    case 8: decode_kernel<8><<<plan.total_items, 256, 0, s>>>(c, layer, a, q, out, counters, partials); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace oscar
