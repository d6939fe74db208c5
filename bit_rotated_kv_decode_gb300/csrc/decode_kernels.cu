// Three-segment decode attention.
//
// "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计": at decode time the
// INT2 history is unpacked, dequantised with its scale / zero point and
// accumulated in floating point; the BF16 sink and recent window are handled
// separately; the partials are merged with an online softmax (max / sum).
// "Together AI Open-Sources OSCAR" (MarkTechPost), section "The Serving
// System": the value path is inverse-rotated.
//
// One launch per layer.  Work items per (request, kv head):
//   items 0..4   BF16 sink page and the four recent-ring pages, unrotated q;
//   items 5..    chunks of INT2 history pages in the rotated basis.
// For an INT2 token j with codes c_j and fp16 scale / zero (s_j, z_j):
//   logit_j = scale * (s_j (q_rot . c_j) + z_j sum(q_rot)),
//   value   = s_j c_j + z_j 1   (accumulated as p_j s_j c_j plus sum p_j z_j).
// The two contractions over a 64-token page -- q_rot . c (64 tokens x G heads x
// 128 channels) and sum_j (p_j s_j) c_j (128 channels x G heads x 64 tokens) --
// run on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulate):
//   * a 2-bit field masked out of a packed byte word, with every other bit
//     zero, is the fp16 subnormal code * 2^(2e-24) -- exact, one LOP3 per two
//     codes; the factor 4^e of its bit position is folded into the other operand;
//   * q_rot and p s are split into fp16 hi + lo parts (22 significant bits),
//     occupying the N columns as (head, part) pairs;
//   * every product is exact in fp32; accumulation is fp32.
// Pages are staged HBM -> shared memory by TMA bulk copies (cp.async.bulk, one
// 4608-byte record per page and kv head) into a per-warp ring, completion on
// mbarriers; every wait is bounded and reports ERR_TIMEOUT instead of hanging.
// Each item writes an (o[128], m, l) partial per query head (log2-domain max m).
// The last item of a (request, kv head) to finish -- an atomic ticket, no
// waiting -- merges the partials, applies R_V^T to the history part and writes
// out = (O_bf16 + O_hist R_V^T) / L.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int PART = PARTIAL_FLOATS;
constexpr int WARPS = 4;                 // warps per CTA
constexpr int THREADS = 32 * WARPS;
// TMA ring depth per warp and resident CTAs per SM: GQA <= 4 trades a stage for
// a fourth resident CTA (16 warps per SM); GQA 8 keeps three stages
template <int G> struct Tune {
  static constexpr int STAGES = G <= 4 ? 2 : 3;
  static constexpr int CTAS = G <= 4 ? 4 : 3;
};
constexpr int BF16_ITEMS = DECODE_BF16_ITEMS;
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr int ERR_TIMEOUT_BIT = 8;

struct DecodeArgs {
  int n;
  int pages_per_chunk;
  int int2_items;            // INT2 CTAs, before the BF16 CTAs
  int group_stride;          // group partial slots per (request, kv head)
  DecodeReq r[DECODE_PER_LAUNCH];
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// 1-D TMA bulk copy global -> shared; completion counted on bar.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait for the phase with the given parity; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < WAIT_LIMIT; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Pair of 2-bit codes m of each 16-bit half of w (m = 0..7) as an fp16x2 of
// subnormals code * 2^(2 e(m) - 24), e(m) = m for m <= 4, m - 5 otherwise.
template <int M>
__device__ __forceinline__ uint32_t code_pair(uint32_t w) {
  if constexpr (M <= 4) {
    return w & (0x00030003u << (2 * M));
  } else {
    return (w >> 10) & (0x00030003u << (2 * (M - 5)));
  }
}
__device__ __forceinline__ uint32_t code_pair_rt(uint32_t w, int m) {
  return m <= 4 ? (w & (0x00030003u << (2 * m))) : ((w >> 10) & (0x00030003u << (2 * (m - 5))));
}
__host__ __device__ constexpr int code_exp(int m) { return m <= 4 ? m : m - 5; }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 hi / lo split of x: hi = fp16_rn(x), lo = fp16_rn(x - hi).
__device__ __forceinline__ void split_half(float x, float& hi, float& lo) {
  hi = __half2float(__float2half_rn(x));
  lo = x - hi;
}

template <int G>
struct Smem {
  // INT2: per-warp TMA rings; BF16 items: the page's K rows (16-byte chunks
  // XOR-swizzled by row) and V rows; after the page loop: per-warp states.
  union {
    __align__(128) uint8_t ring[WARPS][Tune<G>::STAGES][RECORD];
    struct {
      __align__(16) uint16_t k[PAGE][D];
      __align__(16) uint16_t v[PAGE][D];
    } bf;
    float state[WARPS][G][PART];
  } buf;
  __align__(8) uint64_t bar[WARPS][Tune<G>::STAGES];
  float qin[G][D];           // q of the group's query heads (unrotated)
  float q[G][D];             // q_rot (INT2 chunks); merge scratch
  float qsum[G];             // sum of q_rot over channels
  float qscale[G];           // power-of-two prescale of q_rot into fp16 range
  __align__(16) float pw[WARPS][G][PAGE];  // p * s_v of the current page, per warp
  float red[WARPS][G];
  float cred[DECODE_CLUSTER][G][2];   // per-CTA partial sums / maxima of q_rot
  int ticket;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Store to the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Execution-only cluster barrier: every CTA of the cluster has started (no
// memory ordering, so outstanding loads are not waited for).
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// q_rot = q R_K for the G query heads, computed by the DECODE_CLUSTER CTAs of
// one (request, kv head) together: CTA r of the cluster computes channels
// 32 r .. 32 r + 31 (thread (group g, lane l): rows 32 g .. 32 g + 31 of column
// 32 r + l, 32 independent loads of R_K) and stores them into every CTA's
// sm.q through distributed shared memory, with its partial per-head sums and
// maxima; a cluster barrier publishes them.  Leaves sm.q, sm.qsum and the
// power-of-two prescale sm.qscale (|q_rot| 2^24 prescale <= 2^15).
// q of the group (G x 128 bf16) into sm.qin, every load in flight at once.
template <int G>
__device__ __forceinline__ void load_q(const uint16_t* qrow, Smem<G>& sm) {
  const int t = threadIdx.x;
  uint16_t qv[G * D / THREADS];
#pragma unroll
  for (int u = 0; u < G * D / THREADS; ++u) qv[u] = qrow[u * THREADS + t];
#pragma unroll
  for (int u = 0; u < G * D / THREADS; ++u) {
    const int i = u * THREADS + t;
    sm.qin[i / D][i % D] = __uint_as_float(static_cast<uint32_t>(qv[u]) << 16);
  }
}

// This CTA's slab of R_K (column 32 rank + lane, rows 32 grp .. 32 grp + 31), loaded
// before the page copies are queued so it is not served behind them.
__device__ __forceinline__ void load_rk_slab(const DevCache& c, size_t lh, float (&r)[32]) {
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const float* __restrict__ RK = c.rot_k + lh * D * D + 32 * cluster_rank() + lane;
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __ldg(RK + (size_t)(32 * grp + i) * D);
}

template <int G>
__device__ __forceinline__ void cluster_rotate_q(const float (&r)[32], Smem<G>& sm) {
  static_assert(DECODE_CLUSTER * 32 == D, "one 32-channel slab per cluster CTA");
  const int t = threadIdx.x, lane = t & 31, grp = t >> 5;
  const uint32_t rank = cluster_rank();
  cluster_sync_relaxed();   // every CTA of the cluster runs before any remote store
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    acc[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[h] = fmaf(sm.qin[h][32 * grp + i], r[i], acc[h]);
    sm.pw[grp][h][lane] = acc[h];
  }
  __syncthreads();
  for (int idx = t; idx < G * 32; idx += THREADS) {
    const int h = idx >> 5, l = idx & 31;
    float v = 0.0f;
#pragma unroll
    for (int g2 = 0; g2 < WARPS; ++g2) v += sm.pw[g2][h][l];
#pragma unroll
    for (uint32_t dst = 0; dst < DECODE_CLUSTER; ++dst) st_cluster(&sm.q[h][32 * rank + l], dst, v);
    float sum = v, mx = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (l == 0) {
#pragma unroll
      for (uint32_t dst = 0; dst < DECODE_CLUSTER; ++dst) {
        st_cluster(&sm.cred[rank][h][0], dst, sum);
        st_cluster(&sm.cred[rank][h][1], dst, mx);
      }
    }
  }
  cluster_sync();
  if (t < G) {
    float sum = 0.0f, mx = 0.0f;
#pragma unroll
    for (int k = 0; k < DECODE_CLUSTER; ++k) {
      sum += sm.cred[k][t][0];
      mx = fmaxf(mx, sm.cred[k][t][1]);
    }
    int e = 0;
    if (mx > 0.0f) e = static_cast<int>(floorf(log2f(32768.0f / mx))) - 24;
    e = max(-60, min(e, 60));
    sm.qsum[t] = sum;
    sm.qscale[t] = ldexpf(1.0f, e);
  }
  __syncthreads();
}

// One chunk of INT2 history pages of one (request, kv head); leaves the CTA's
// partial (rotated basis) for every query head of the group in part_out.
template <int G>
__device__ __forceinline__ void int2_chunk(const DevCache& c, int layer, const DecodeReq& R, int head, int chunk,
                                           int ppc, const uint16_t* qrow, Smem<G>& sm, float* part_out) {
  constexpr int NT = (G + 3) / 4;       // n-tiles of 8 columns = 4 heads x (hi, lo)
  constexpr int STAGES = Tune<G>::STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid = lane & 3;
  const float scale2 = c.scale * LOG2E;
  const int nhist = R.hist_end - SINK;
  const int npages = (nhist + PAGE - 1) / PAGE;
  const int pc0 = chunk * ppc;
  const int pc1 = min(npages, pc0 + ppc);
  const int my_n = (pc1 - pc0 > warp) ? (pc1 - pc0 - warp + WARPS - 1) / WARPS : 0;
  const int32_t* pt = c.hist_pt + (size_t)R.slot * c.max_pages;
  const uint8_t* base = c.int2 + layer * c.int2_layer_stride + (size_t)head * RECORD;
  const size_t pstride = (size_t)c.Hkv * RECORD;
  bool timed_out = false;
  int issued = 0;
  float rk_slab[32];   // copies issued by this warp (lane 0's count)

  // page ids of this warp's pages, read 32 at a time (lane l holds page 32 b + l of
  // batch b); page_src is called by the whole warp with increasing j
  int32_t batch_pages = 0;
  int batch_idx = -1;
  auto page_src = [&](int j) -> const uint8_t* {
    const int b = j >> 5;
    if (b != batch_idx) {
      batch_idx = b;
      const int jj = 32 * b + lane;
      int32_t page = 0;
      if (jj < my_n) {
        page = pt[pc0 + warp + WARPS * jj];
        if (page < 0 || page >= c.n_int2_pages) {
          atomicOr(c.err, ERR_INT2_PAGE);
          page = 0;
        }
      }
      batch_pages = page;
    }
    return base + (size_t)__shfl_sync(0xffffffffu, batch_pages, j & 31) * pstride;
  };
  // every global load the prologue needs, issued together before any page copy:
  // the first batch of page ids, this CTA's R_K slab and q
  (void)page_src(0);
  load_rk_slab(c, (size_t)layer * c.Hkv + head, rk_slab);
  load_q<G>(qrow, sm);
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(&sm.bar[warp][st], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
#pragma unroll
  for (int j = 0; j < STAGES; ++j) {
    const uint8_t* src = page_src(j);
    if (lane == 0 && j < my_n) {
      mbar_expect_tx(&sm.bar[warp][j], RECORD);
      tma_load_1d(sm.buf.ring[warp][j], src, RECORD, &sm.bar[warp][j]);
      ++issued;
    }
  }
  // the copies are in flight while the cluster rotates q
  cluster_rotate_q<G>(rk_slab, sm);
  // weights p * s_v are prescaled by 2^ew so the smallest ones stay representable in
  // fp16: s_v <= fp16(2 tau_V / 3) and p <= 1, so p s_v 2^ew <= 2^15
  int ew;
  {
    const float smax = c.tau_v[(size_t)layer * c.Hkv + head] * (2.0f / 3.0f) * 1.002f;
    ew = max(-60, min(60, static_cast<int>(floorf(log2f(32768.0f / smax)))));
  }
  const float wscale = ldexpf(1.0f, ew);

  // B operands of q_rot . c: per n-tile, k-step s, two registers (hi or lo part)
  uint32_t bq[NT][8][2];
  float invp[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + (gid >> 1);
    const bool lo_part = gid & 1;
    const bool hv = h < G;
    const float p = hv ? sm.qscale[h] : 1.0f;
    invp[nt] = (4 * nt + tid < G) ? 1.0f / sm.qscale[4 * nt + tid] : 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int ch0 = 32 * tid + 16 * (s >> 2) + 2 * (s & 3);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int m = 2 * (s & 3) + r;
        const int cha = ch0 + r;
        const float f = ldexpf(p, 24 - 2 * code_exp(m));
        float va = hv ? sm.q[h][cha] * f : 0.0f;
        float vb = hv ? sm.q[h][cha + 8] * f : 0.0f;
        float ha, la, hb, lb;
        split_half(va, ha, la);
        split_half(vb, hb, lb);
        bq[nt][s][r] = lo_part ? pack_half2(la, lb) : pack_half2(ha, hb);
      }
    }
  }
  float qs[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) qs[nt] = (4 * nt + tid < G) ? sm.qsum[4 * nt + tid] : 0.0f;

  float o[NT][8][4];
  float m_run[NT], l_run[NT], u_run[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.0f;
    u_run[nt] = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][mt][e] = 0.0f;
  }

  for (int j = 0; j < my_n; ++j) {
    const int stg = j % STAGES;
    if (!timed_out && !mbar_wait(&sm.bar[warp][stg], (j / STAGES) & 1)) {
      timed_out = true;
      if (lane == 0) atomicOr(c.err, ERR_TIMEOUT_BIT);
    }
    if (timed_out) break;
    const uint8_t* rec = sm.buf.ring[warp][stg];
    const int pi = pc0 + warp + WARPS * j;
    const int valid = min(PAGE, nhist - pi * PAGE);

    // ---- logits: 4 m-tiles of 16 tokens x NT n-tiles, K = 128 channels
    float acc[NT][4][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const uint2 ka = *reinterpret_cast<const uint2*>(rec + K_CODES_OFF + (16 * mt + gid) * CODE_BYTES + 8 * tid);
      const uint2 kb = *reinterpret_cast<const uint2*>(rec + K_CODES_OFF + (16 * mt + gid + 8) * CODE_BYTES + 8 * tid);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t wa = s < 4 ? ka.x : ka.y;
        const uint32_t wb = s < 4 ? kb.x : kb.y;
        const int m0 = 2 * (s & 3);
        const uint32_t a0 = code_pair_rt(wa, m0), a1 = code_pair_rt(wb, m0);
        const uint32_t a2 = code_pair_rt(wa, m0 + 1), a3 = code_pair_rt(wb, m0 + 1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt][mt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
      }
    }
    // token meta of this lane's 8 tokens: 16 mt + gid + 8 rr
    float lg[NT][8], sv[8], zv[8];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int tok = 16 * mt + gid + 8 * rr;
        const __half2 km = *reinterpret_cast<const __half2*>(rec + K_META_OFF + tok * META_BYTES);
        const __half2 vm = *reinterpret_cast<const __half2*>(rec + V_META_OFF + tok * META_BYTES);
        const bool ok = tok < valid;
        sv[2 * mt + rr] = ok ? __low2float(vm) : 0.0f;
        zv[2 * mt + rr] = ok ? __high2float(vm) : 0.0f;
        const float sk = __low2float(km), zk = __high2float(km);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float d = (acc[nt][mt][2 * rr] + acc[nt][mt][2 * rr + 1]) * invp[nt];
          lg[nt][2 * mt + rr] = (ok && 4 * nt + tid < G) ? scale2 * fmaf(sk, d, zk * qs[nt]) : -INFINITY;
        }
      }
    // ---- online softmax per head (lanes with equal tid share a head)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pm = lg[nt][0];
#pragma unroll
      for (int i = 1; i < 8; ++i) pm = fmaxf(pm, lg[nt][i]);
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      const float m_new = fmaxf(m_run[nt], pm);
      if (m_new > m_run[nt]) {   // rescale only when the running max grows
        const float corr = (m_run[nt] == -INFINITY) ? 0.0f : exp2f(m_run[nt] - m_new);
        m_run[nt] = m_new;
        l_run[nt] *= corr;
        u_run[nt] *= corr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][mt][e] *= corr;
      }
      const int h = 4 * nt + tid;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = (lg[nt][i] == -INFINITY) ? 0.0f : exp2f(lg[nt][i] - m_new);
        l_run[nt] += p;
        u_run[nt] = fmaf(p, zv[i], u_run[nt]);
        if (h < G) sm.pw[warp][h][16 * (i >> 1) + gid + 8 * (i & 1)] = p * sv[i] * wscale;
      }
    }
    __syncwarp();
    // ---- values: 8 m-tiles of 16 channels x NT n-tiles, K = 64 tokens
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int ta = 16 * s + 2 * tid;
      uint32_t bw[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = 4 * nt + (gid >> 1);
        if (h < G) {
          const float2 w01 = *reinterpret_cast<const float2*>(&sm.pw[warp][h][ta]);
          const float2 w89 = *reinterpret_cast<const float2*>(&sm.pw[warp][h][ta + 8]);
          float h0, l0, h1, l1, h8, l8, h9, l9;
          split_half(w01.x, h0, l0);
          split_half(w01.y, h1, l1);
          split_half(w89.x, h8, l8);
          split_half(w89.y, h9, l9);
          bw[nt][0] = (gid & 1) ? pack_half2(l0, l1) : pack_half2(h0, h1);
          bw[nt][1] = (gid & 1) ? pack_half2(l8, l9) : pack_half2(h8, h9);
        } else {
          bw[nt][0] = bw[nt][1] = 0u;
        }
      }
      const uint32_t* vrow = reinterpret_cast<const uint32_t*>(rec + V_CODES_OFF) + gid;
      const uint32_t wa = vrow[ta * (CODE_BYTES / 4)], wb = vrow[(ta + 1) * (CODE_BYTES / 4)];
      const uint32_t wc = vrow[(ta + 8) * (CODE_BYTES / 4)], wd = vrow[(ta + 9) * (CODE_BYTES / 4)];
      const uint32_t x1 = __byte_perm(wa, wb, 0x5410), y1 = __byte_perm(wa, wb, 0x7632);
      const uint32_t x2 = __byte_perm(wc, wd, 0x5410), y2 = __byte_perm(wc, wd, 0x7632);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t a0 = code_pair_rt(x1, mt), a1 = code_pair_rt(y1, mt);
        const uint32_t a2 = code_pair_rt(x2, mt), a3 = code_pair_rt(y2, mt);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(o[nt][mt], a0, a1, a2, a3, bw[nt][0], bw[nt][1]);
      }
    }
    __syncwarp();
    {
      const uint8_t* src = page_src(j + STAGES);
      if (lane == 0 && j + STAGES < my_n) {
        mbar_expect_tx(&sm.bar[warp][stg], RECORD);
        tma_load_1d(sm.buf.ring[warp][stg], src, RECORD, &sm.bar[warp][stg]);
        ++issued;
      }
    }
  }
  if (timed_out && lane == 0) {
    // let every copy this warp issued land (bounded) before the buffers are reused:
    // stage st received ceil((issued - st) / STAGES) copies; wait for the last phase
    for (int st = 0; st < STAGES && st < issued; ++st) {
      const int count = (issued - st + STAGES - 1) / STAGES;
      mbar_wait(&sm.bar[warp][st], (count - 1) & 1);
    }
  }
  __syncthreads();   // every warp is done with every ring before states overwrite them

  // ---- this warp's state -> shared memory (rotated basis, unscaled, z term added)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float l = l_run[nt], u = u_run[nt];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, off);
      u += __shfl_xor_sync(0xffffffffu, u, off);
    }
    const int h = 4 * nt + tid;
    if (h < G) {
      float* st = sm.buf.state[warp][h];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float f = ldexpf(1.0f, 24 - 2 * code_exp(mt) - ew);
        st[16 * gid + mt] = fmaf(o[nt][mt][0] + o[nt][mt][1], f, u);
        st[16 * gid + 8 + mt] = fmaf(o[nt][mt][2] + o[nt][mt][3], f, u);
      }
      if (gid == 0) {
        st[PARTIAL_M] = m_run[nt];
        st[PARTIAL_L] = l;
      }
    }
  }
  __syncthreads();
  // ---- merge the warps: thread t owns channel t
  const int t = threadIdx.x;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sm.buf.state[w][h][PARTIAL_M]);
    float acc_o = 0.0f, acc_l = 0.0f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float mw = sm.buf.state[w][h][PARTIAL_M];
      if (mw == -INFINITY) continue;
      const float f = exp2f(mw - M);
      acc_o = fmaf(sm.buf.state[w][h][t], f, acc_o);
      acc_l = fmaf(sm.buf.state[w][h][PARTIAL_L], f, acc_l);
    }
    part_out[h * PART + t] = acc_o;
    if (t == 0) {
      part_out[h * PART + PARTIAL_M] = M;
      part_out[h * PART + PARTIAL_L] = acc_l;
    }
  }
}

// One BF16 page (the sink page, or one of the four recent-ring pages) of one
// (request, kv head), with the unrotated q; partial for every query head.
template <int G>
__device__ __forceinline__ void bf16_item(const DevCache& c, int layer, const DecodeReq& R, int head, int which,
                                          Smem<G>& sm, float* part_out) {
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const float scale2 = c.scale * LOG2E;
  const int T = R.tokens, he = R.hist_end;
  int page = which == 0 ? R.sink_page : R.ring_page[which - 1];
  if (page < 0 || page >= c.n_bf16_pages) {
    if (t == 0) atomicOr(c.err, ERR_BF16_PAGE);
    page = 0;
  }
  // validity of row r: sink rows [0, min(T, 64)); ring slot s = 64 (which-1) + r holds
  // position he + ((s - (he - 64)) mod 256), valid when below T
  auto row_valid = [&](int r) -> bool {
    if (which == 0) return r < min(T, SINK);
    if (T <= SINK) return false;
    const int s = PAGE * (which - 1) + r;
    const int p = he + ((s - (he - SINK)) % RECENT + RECENT) % RECENT;
    return p < T;
  };
  const uint16_t* src = c.bf16 + layer * c.bf16_layer_stride + ((size_t)page * c.Hkv + head) * BF16_RECORD_ELEMS;
  constexpr int LOADS = PAGE * (D / 8) / THREADS;
  uint4 kk[LOADS], vv[LOADS];
#pragma unroll
  for (int it = 0; it < LOADS; ++it) {
    const int idx = t + THREADS * it, r = idx / (D / 8), part = idx % (D / 8);
    kk[it] = reinterpret_cast<const uint4*>(src + (size_t)r * D)[part];
    vv[it] = reinterpret_cast<const uint4*>(src + (size_t)(PAGE + r) * D)[part];
  }
#pragma unroll
  for (int it = 0; it < LOADS; ++it) {
    const int idx = t + THREADS * it, r = idx / (D / 8), part = idx % (D / 8);
    reinterpret_cast<uint4*>(&sm.buf.bf.k[r][0])[part ^ (r & 15)] = kk[it];
    reinterpret_cast<uint4*>(&sm.buf.bf.v[r][0])[part] = vv[it];
  }
  __syncthreads();
  // logits: thread t -> token t/2, channel half t%2, all G heads
  {
    const int r = t >> 1, half = t & 1;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
    const uint4* kr = reinterpret_cast<const uint4*>(&sm.buf.bf.k[r][0]);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int chunk = 8 * half + b;
      const uint4 w = kr[chunk ^ (r & 15)];
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float k0 = bf16lo(ww[e]), k1 = bf16hi(ww[e]);
        const int ch = 8 * chunk + 2 * e;
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = fmaf(sm.qin[h][ch + 1], k1, fmaf(sm.qin[h][ch], k0, acc[h]));
      }
    }
    const bool ok = row_valid(r);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
      if (half == 0) sm.pw[0][h][r] = ok ? acc[h] * scale2 : -INFINITY;
    }
  }
  __syncthreads();
  // softmax and values: warp w handles heads w, w + 4; lane owns channels 4 lane .. 4 lane + 3
  for (int h = warp; h < G; h += WARPS) {
    const float x0 = sm.pw[0][h][lane], x1 = sm.pw[0][h][lane + 32];
    float m = fmaxf(x0, x1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p0 = (x0 == -INFINITY) ? 0.0f : exp2f(x0 - m);
    const float p1 = (x1 == -INFINITY) ? 0.0f : exp2f(x1 - m);
    float l = p0 + p1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    __syncwarp();
    sm.pw[0][h][lane] = p0;
    sm.pw[0][h][lane + 32] = p1;
    __syncwarp();
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (m != -INFINITY) {
      for (int r = 0; r < PAGE; ++r) {
        const float p = sm.pw[0][h][r];
        const uint2 vv = reinterpret_cast<const uint2*>(&sm.buf.bf.v[r][0])[lane];
        acc[0] = fmaf(p, bf16lo(vv.x), acc[0]);
        acc[1] = fmaf(p, bf16hi(vv.x), acc[1]);
        acc[2] = fmaf(p, bf16lo(vv.y), acc[2]);
        acc[3] = fmaf(p, bf16hi(vv.y), acc[3]);
      }
    }
    reinterpret_cast<float4*>(part_out + h * PART)[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (lane == 0) {
      part_out[h * PART + PARTIAL_M] = m;
      part_out[h * PART + PARTIAL_L] = l;
    }
  }
}

// Online-softmax merge of `count` (<= MERGE_GROUP) consecutive partials
// (stride G * PART floats) into one.  The (m, l) pairs are loaded by
// different threads at once; then thread t owns channel t of every head and
// issues all of its count * G loads before using them.
template <int G>
__device__ __forceinline__ void merge_partials(const float* src, int count, float* dst, Smem<G>& sm) {
  const int t = threadIdx.x;
  if (t < count * G) {
    const int k = t / G, h = t % G;
    sm.pw[0][h][k] = __ldcg(src + ((size_t)k * G + h) * PART + PARTIAL_M);
    sm.pw[0][h][MERGE_GROUP + k] = __ldcg(src + ((size_t)k * G + h) * PART + PARTIAL_L);
  }
  float ov[MERGE_GROUP][G];
#pragma unroll
  for (int k = 0; k < MERGE_GROUP; ++k)
#pragma unroll
    for (int h = 0; h < G; ++h) ov[k][h] = k < count ? __ldcg(src + ((size_t)k * G + h) * PART + t) : 0.0f;
  __syncthreads();
  if (t < G) {
    float M = -INFINITY;
    for (int k = 0; k < count; ++k) M = fmaxf(M, sm.pw[0][t][k]);
    float L = 0.0f;
    for (int k = 0; k < count; ++k) {
      const float mk = sm.pw[0][t][k];
      const float f = (mk == -INFINITY) ? 0.0f : exp2f(mk - M);
      sm.pw[0][t][2 * MERGE_GROUP + k] = f;
      L = fmaf(sm.pw[0][t][MERGE_GROUP + k], f, L);
    }
    dst[t * PART + PARTIAL_M] = M;
    dst[t * PART + PARTIAL_L] = L;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float o = 0.0f;
#pragma unroll
    for (int k = 0; k < MERGE_GROUP; ++k)
      if (k < count) o = fmaf(ov[k][h], sm.pw[0][h][2 * MERGE_GROUP + k], o);
    dst[h * PART + t] = o;
  }
}

template <int G>
__global__ void __launch_bounds__(THREADS, Tune<G>::CTAS) decode_kernel(DevCache c, int layer, DecodeArgs a,
                                                         const uint16_t* __restrict__ q, float* __restrict__ out,
                                                         int32_t* counters, float* partials, float* gpart) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<G>& sm = *reinterpret_cast<Smem<G>*>(smem_raw);
  const int item = blockIdx.x;
  int ri = 0, head, sub;
  if (item < a.int2_items) {
    // INT2 chunk: clusters of DECODE_CLUSTER consecutive CTAs share one (request, kv head)
    while (ri + 1 < a.n && a.r[ri + 1].int2_start <= item) ++ri;
    const int local = item - a.r[ri].int2_start;
    head = local / a.r[ri].chunks;
    sub = BF16_ITEMS + local % a.r[ri].chunks;
  } else {
    const int b = item - a.int2_items;
    if (b >= a.n * c.Hkv * BF16_ITEMS) return;   // cluster padding
    ri = b / (c.Hkv * BF16_ITEMS);
    head = (b / BF16_ITEMS) % c.Hkv;
    sub = b % BF16_ITEMS;
  }
  const DecodeReq R = a.r[ri];
  const int per_head = BF16_ITEMS + R.chunks;
  const int t = threadIdx.x;
  const size_t lh = (size_t)layer * c.Hkv + head;
  const float* __restrict__ RVt = c.rot_vt + lh * D * D;

  if (sub == 0) {
    // warm L2 with R_V^T for whichever item of this head merges last
    for (int line = t; line < D * D / 32; line += THREADS)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(RVt + (size_t)line * 32));
  }
  const uint16_t* qrow = q + ((size_t)R.batch_row * c.Hq + (size_t)head * G) * D;
  if (sub < BF16_ITEMS) {
    load_q<G>(qrow, sm);
    __syncthreads();
  }

  const size_t head_parts = (size_t)R.part_start + (size_t)head * per_head;
  float* part = partials + (head_parts + sub) * G * PART;
  if (sub < BF16_ITEMS) {
    bf16_item<G>(c, layer, R, head, sub, sm, part);
  } else {
    int2_chunk<G>(c, layer, R, head, sub - BF16_ITEMS, a.pages_per_chunk, qrow, sm, part);
  }

  // ---- two-level merge by atomic tickets (nobody waits) -----------------------------
  // group 0 = the BF16 items, group g >= 1 = INT2 chunks (g-1)*MERGE_GROUP .. +MERGE_GROUP-1.
  // Ticket protocol: block barrier, then one thread fences (cumulative over the
  // block's writes) and takes the ticket; the winner fences before reading.
  const int g = sub < BF16_ITEMS ? 0 : 1 + (sub - BF16_ITEMS) / MERGE_GROUP;
  const int gfirst = g == 0 ? 0 : BF16_ITEMS + (g - 1) * MERGE_GROUP;
  const int gcount = g == 0 ? BF16_ITEMS : min(MERGE_GROUP, R.chunks - (g - 1) * MERGE_GROUP);
  const int ngroups = 1 + (R.chunks + MERGE_GROUP - 1) / MERGE_GROUP;
  int32_t* cnt = counters + (size_t)(ri * c.Hkv + head) * MERGE_COUNTERS;
  float* gbase = gpart + (size_t)(ri * c.Hkv + head) * a.group_stride * G * PART;
  __syncthreads();
  if (t == 0) {
    __threadfence();
    sm.ticket = atomicAdd(cnt + 1 + g, 1);
    if (sm.ticket == gcount - 1) __threadfence();
  }
  __syncthreads();
  if (sm.ticket != gcount - 1) return;
  merge_partials<G>(partials + (head_parts + gfirst) * G * PART, gcount, gbase + (size_t)g * G * PART, sm);
  __syncthreads();
  if (t == 0) {
    cnt[1 + g] = 0;
    __threadfence();
    sm.ticket = atomicAdd(cnt, 1);
    if (sm.ticket == ngroups - 1) __threadfence();
  }
  __syncthreads();
  if (sm.ticket != ngroups - 1) return;

  // ---- last group of this (request, kv head): BF16 part + R_V^T (history part) ----
  // stage every group partial in shared memory with one round of 16-byte loads
  float* gs = &sm.buf.state[0][0][0];   // [ngroups][G][PART], staged in chunks of STAGE_GROUPS
  constexpr int STAGE_GROUPS = (WARPS * Tune<G>::STAGES * RECORD) / (G * PART * 4);
  float* oh = &sm.pw[0][0][0];           // [G][D] history part (rotated basis)
  float M[G], L[G], ob[G], ohist[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.0f;
    ob[h] = 0.0f;
    ohist[h] = 0.0f;
  }
  for (int k0 = 0; k0 < ngroups; k0 += STAGE_GROUPS) {
    const int kn = min(STAGE_GROUPS, ngroups - k0);
    const int n4 = kn * G * PART / 4;
    const float4* src4 = reinterpret_cast<const float4*>(gbase + (size_t)k0 * G * PART);
    for (int i0 = 0; i0 < n4; i0 += 8 * THREADS) {
      float4 v4[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * THREADS + t;
        if (i < n4) v4[u] = __ldcg(src4 + i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * THREADS + t;
        if (i < n4) reinterpret_cast<float4*>(gs)[i] = v4[u];
      }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float Mn = M[h];
      for (int k = 0; k < kn; ++k) Mn = fmaxf(Mn, gs[(k * G + h) * PART + PARTIAL_M]);
      const float fo = (M[h] == -INFINITY) ? 0.0f : exp2f(M[h] - Mn);
      L[h] *= fo;
      ob[h] *= fo;
      ohist[h] *= fo;
      M[h] = Mn;
      for (int k = 0; k < kn; ++k) {
        const float* pk = gs + (k * G + h) * PART;
        const float mk = pk[PARTIAL_M];
        const float f = (mk == -INFINITY) ? 0.0f : exp2f(mk - Mn);
        L[h] = fmaf(pk[PARTIAL_L], f, L[h]);
        if (k0 + k == 0)
          ob[h] = fmaf(pk[t], f, ob[h]);
        else
          ohist[h] = fmaf(pk[t], f, ohist[h]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    oh[h * D + t] = ohist[h];
    if (t == 0) sm.qsum[h] = L[h];
    sm.q[h][t] = ob[h];
  }
  __syncthreads();
  // out_c = (O_bf16_c + sum_j O_hist_j R_V[c][j]) / L with rot_vt[j][c] = R_V[c][j]:
  // thread (group gr, lane l) sums rows 32 gr .. 32 gr + 31 for channels 4l .. 4l+3
  {
    const int lane = t & 31, grp = t >> 5;
    float4 acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    constexpr int BATCH = G <= 4 ? 16 : 8;   // R_V rows in flight per thread
#pragma unroll
    for (int half = 0; half < 32 / BATCH; ++half) {
      float4 r[BATCH];
#pragma unroll
      for (int i = 0; i < BATCH; ++i)
        r[i] = __ldg(reinterpret_cast<const float4*>(RVt + (size_t)(32 * grp + BATCH * half + i) * D) + lane);
#pragma unroll
      for (int i = 0; i < BATCH; ++i) {
        const int j = 32 * grp + BATCH * half + i;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float oj = oh[h * D + j];
          acc[h].x = fmaf(oj, r[i].x, acc[h].x);
          acc[h].y = fmaf(oj, r[i].y, acc[h].y);
          acc[h].z = fmaf(oj, r[i].z, acc[h].z);
          acc[h].w = fmaf(oj, r[i].w, acc[h].w);
        }
      }
    }
    float* mp = &sm.buf.state[0][0][0];   // [4][G][D]
#pragma unroll
    for (int h = 0; h < G; ++h) reinterpret_cast<float4*>(mp + ((size_t)grp * G + h) * D)[lane] = acc[h];
  }
  __syncthreads();
  {
    const float* mp = &sm.buf.state[0][0][0];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = sm.q[h][t];
#pragma unroll
      for (int g2 = 0; g2 < WARPS; ++g2) v += mp[((size_t)g2 * G + h) * D + t];
      out[((size_t)R.batch_row * c.Hq + (size_t)head * G + h) * D + t] = v / sm.qsum[h];
    }
  }
  if (t == 0) cnt[0] = 0;
}

template <int G>
cudaError_t launch_g(const DevCache& c, int layer, const DecodeArgs& a, int items, const uint16_t* q, float* out,
                     int32_t* counters, float* partials, float* gpart, cudaStream_t s) {
  static bool attr = false;
  const size_t smem = sizeof(Smem<G>);
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(items));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = DECODE_CLUSTER;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<G>, c, layer, a, q, out, counters, partials, gpart);
}

}  // namespace

cudaError_t launch_decode(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& plan,
                          const uint16_t* q, float* out, void* workspace, cudaStream_t s) {
  DecodeArgs a;
  a.n = plan.n;
  a.pages_per_chunk = plan.pages_per_chunk;
  a.group_stride = plan.group_stride;
  a.int2_items = plan.int2_items;
  for (int i = 0; i < plan.n; ++i) a.r[i] = reqs[i];
  int32_t* counters = static_cast<int32_t*>(workspace);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.counter_bytes);
  float* gpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.counter_bytes + plan.partial_bytes);
  switch (c.G) {
    case 1: return launch_g<1>(c, layer, a, plan.total_items, q, out, counters, partials, gpart, s);
    case 2: return launch_g<2>(c, layer, a, plan.total_items, q, out, counters, partials, gpart, s);
    case 4: return launch_g<4>(c, layer, a, plan.total_items, q, out, counters, partials, gpart, s);
    case 8: return launch_g<8>(c, layer, a, plan.total_items, q, out, counters, partials, gpart, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oscar

namespace oscar {
int decode_ctas_per_sm(int g) { return g <= 4 ? Tune<4>::CTAS : Tune<8>::CTAS; }
}  // namespace oscar
