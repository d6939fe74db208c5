// Three-segment decode attention.
//
// "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计": at decode time the
// INT2 history is unpacked, dequantised with its scale / zero point and
// accumulated in floating point; the BF16 sink and recent window are handled
// separately; the partials are merged with an online softmax (max / sum).
// "Together AI Open-Sources OSCAR" (MarkTechPost), section "The Serving
// System": the value path is inverse-rotated.
//
// One launch per layer (and per batch of up to 64 requests): one persistent CTA
// per SM.  nbc of them (the last blocks) attend to the BF16 sink and recent pages of the
// (request, kv head) segments, a whole segment's BF16 pages at a time, with the
// unrotated q (one record per segment, plain basis).  The other CTAs share the
// INT2 history pages, cut into equal contiguous ranges that a CTA walks segment
// by segment:
//   * q_rot = q R_K into tensor-core operands in shared memory (R_K is read
//     before the launch waits for the preceding grid, q after);
//   * the segment's INT2 pages, each warp through its own TMA ring, the warps'
//     partials combined into one record (o, m, l; rotated basis).
// A per-(request, kv head) counter in the cache counts the CTAs done with a
// segment; the one that completes the count merges the segment's records with
// an online softmax and writes out = (O_bf16 + O_hist R_V^T) / L for its G query
// heads.
// For an INT2 token j with codes c_j and fp16 scale / zero (s_j, z_j):
//   logit_j = scale * (s_j (q_rot . c_j) + z_j sum(q_rot)),
//   value   = s_j c_j + z_j 1   (accumulated as p_j s_j c_j plus sum p_j z_j).
// The two contractions over a 64-token page -- q_rot . c (64 tokens x G heads x
// 128 channels) and sum_j (p_j s_j) c_j (128 channels x G heads x 64 tokens) --
// run on the tensor cores as warp-level mma.sync m16n8k16 (fp16 operands, fp32
// accumulate).  These are skinny products (the N side is G heads x two parts),
// which the warp-level MMA of every sub-partition serves at a lower cost per
// page than the single-thread-issued tcgen05 MMA, whose per-instruction cost does
// not shrink with N:
//   * a 2-bit field masked out of a packed byte word, with every other bit
//     zero, is the fp16 subnormal code * 2^(2e-24) -- exact, one LOP3 per two
//     codes; the factor 4^e of its bit position is folded into the other operand;
//   * q_rot and p s are split into fp16 hi + lo parts (22 significant bits),
//     occupying the N columns as (head, part) pairs;
//   * every product is exact in fp32; accumulation is fp32.
// Pages are staged HBM -> shared memory by TMA bulk copies (cp.async.bulk, one
// record per page and kv head: 4608 B at quantisation group 128 -- K codes
// [64][32] B, V codes [64][32] B, K and V {s, z} [64] x 4 B -- and 5120 B at
// group 64, with two {s, z} per token) into a per-warp ring, completion on mbarriers;
// every wait is bounded and reports ERR_TIMEOUT instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <type_traits>

#include "append_device.cuh"
#include "internal.h"

namespace oscar {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int PART = PARTIAL_FLOATS;
constexpr int STAGES = 2;                // TMA ring depth per warp
constexpr uint32_t SUSPEND_NS = 20000;   // a waiting warp sleeps until the phase completes
constexpr int LAZY_MAX_INT = 8;          // softmax reference max kept within 2^8 of the true one
constexpr float LAZY_MAX = static_cast<float>(LAZY_MAX_INT);
constexpr int SLABS = D / 32;
constexpr int BF16_ITEMS = DECODE_BF16_ITEMS;

// Warps per CTA: all sixteen when a warp fits in 128 registers, fewer where the
// second n-tile (G = 8) or the second quantisation group (G_K = 64) take more
// registers and shared memory.
template <int G, int GK>
struct Tune {
  static constexpr int NW = (G <= 4 && GK == 128) ? 16 : ((G == 8 && GK == 64) ? 8 : 12);
  static constexpr int THREADS = 32 * NW;
};

struct Seg {
  int valid;
  int ri, head;    // request index in the launch, kv head
  int p0, p1;      // INT2 pages [p0, p1) of this CTA
  int slot;        // INT2 record: segment + INT2 CTA
  int c_lo, c_hi;  // the INT2 CTAs whose ranges meet the segment
};

struct DecodeArgs {
  int n, ncta, nbc;                 // nbc: the first nbc CTAs take the BF16 blocks
  int prefetch;                     // the preceding launch is a decode of this cache (see decode_kernel)
  uint32_t epoch;                   // a decode step (append first) when non-zero
  int64_t total_cost;
  DecodeDebug dbg;
  int32_t cstart[DECODE_MAX_INT2 + 1];   // INT2 CTA c holds cost units [cstart[c], cstart[c + 1])
  const uint16_t* k_new;   // fused step: the appended token's K / V rows (batch rows), else null
  const uint16_t* v_new;
  DecodeReq r[DECODE_PER_LAUNCH];
};

// Programmatic dependent launch: wait for the preceding grid (complete, its
// writes visible); allow the next grid to be scheduled.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(SUSPEND_NS)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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
// subnormals code * 2^(2 e(m) - 24), e(m) = m for m <= 4, m - 5 otherwise; the
// caller supplies ws = w >> 10, so one shift serves three codes.
__host__ __device__ constexpr int code_exp(int m) { return m <= 4 ? m : m - 5; }
__device__ __forceinline__ uint32_t code_pair2(uint32_t w, uint32_t ws, int m) {
  return m <= 4 ? (w & (0x00030003u << (2 * m))) : (ws & (0x00030003u << (2 * (m - 5))));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 hi / lo split of x: hi = fp16_rn(x), lo = fp16_rn(x - hi).
__device__ __forceinline__ void split_half(float x, float& hi, float& lo) {
  hi = __half2float(__float2half_rn(x));
  lo = x - hi;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- q operands ----------------------------------------------------------------------
// Per segment the CTA holds QFrag<G>::WORDS 32-bit words in shared memory:
//   frag[lane][nt][s][r]  fp16x2 B operands of the q_rot . c contraction
//                         (n-tile nt of (head, hi / lo part) columns, k-step s,
//                         register r), prescaled by qscale(h) 2^(24 - 2 e(m)) so
//                         that the fp32 accumulator holds qscale(h) q_rot . c;
//   kscale[8]             fp32 per query head h: scale log2(e) / qscale(h);
//   qsum[4][8]            fp32 per 32-channel slab and head: sum of q_rot.
// The logit in the log2 domain is
//   kscale[h] s_k acc + (scale log2(e) sum_slab qsum[slab][h]) z_k.
// Register r of k-step s for lane (gid, tid) pairs channel 32 tid + 16 (s >> 2) + m
// (low half) with that channel + 8 (high half), m = 2 (s & 3) + r, as the code
// registers of the A operand do.  With G_K = 64 the k-steps are group-pure instead:
// channel 64 (s >> 2) + 16 tid + m (and + 8), so k-steps 0..3 hold group 0 and
// 4..7 group 1.  qscale(h) = 2^e with |q_rot| 2^(e + 24) <= 2^15 taken from
// |q|_2 >= max |q_rot| (R_K is orthogonal).
template <int G>
struct QFrag {
  static constexpr int NT = (G + 3) / 4;
  static constexpr int REGS = NT * 16;              // fragment registers per lane
  static constexpr int CONSTS = 32 * REGS;          // word offset of kscale[8], qsum[4][8]
  static constexpr int WORDS = CONSTS + 40;
};

constexpr int WH_STRIDE = PAGE + 8;   // halves per weight row (bank spread)
// Softmax weights of the page being processed, fp16 [G x groups][hi, lo][WH_STRIDE]
// per warp (row (D / GK) h + g: head h, quantisation group g).  When they fit (up
// to four heads with one group, two with two) they live in the page's K-code
// region, dead once the logits are formed; otherwise in rows of their own.
template <int G, int GK = 128>
constexpr bool kWeightsInRing = G * (D / GK) * 2 * WH_STRIDE * 2 <= PAGE * CODE_BYTES;
template <int G, int GK, int NW, bool InRing = kWeightsInRing<G, GK>>
struct WeightRows {
  __align__(16) uint16_t wh[NW][G * (D / GK)][2][WH_STRIDE];
};
template <int G, int GK, int NW>
struct WeightRows<G, GK, NW, true> {};

template <int G, int GK>
struct Smem {
  static constexpr int NW = Tune<G, GK>::NW;
  static constexpr int NPART = Tune<G, GK>::THREADS / D;   // row parts of the q rotation
  // per-warp TMA rings of INT2 page records; while no copy is in flight (the merge
  // of a segment) the staging of the merged records
  struct {
    __align__(128) uint8_t ring[NW][STAGES][record_for(GK)];
  } buf;
  __align__(16) float state[NW][G][PART];   // each warp's partial (o, m, l) before the CTA combine
  union {
    struct {
      __align__(16) float q[D][G];      // q as [channel][head]: one row holds the G heads
      float part[NPART][G][D];
      float norm[G];
      int qe[G];                        // q scale exponents
    } pro;                              // rotation of q
    struct {
      __align__(16) float hist[D][G];   // O_hist of the merged segment, [channel][head]
      float part[NPART][G][D];          // row parts of O_hist R_V^T
    } mrg;                              // merge of a segment (last CTA)
  } scr;
  __align__(16) uint32_t qf[QFrag<G>::WORDS];   // q operands of the current segment (read as uint4)
  __align__(8) uint64_t bar[NW][STAGES];
  uint64_t mbar_m;                       // staging of a merge's records
  uint64_t mbar_r;                       // staging of a merge's R_V^T
  __align__(16) float4 meta[NW][PAGE];   // INT2: per token {s_k, z_k, s_v 2^ew, z_v}; BF16: weights
  __align__(16) float4 meta2[NW][GK == 64 ? PAGE : 1];   // G_K = 64: the same for group 1
  WeightRows<G, GK, NW> w;
  float wf[NW][8];                       // combine: per (warp, head) factor 2^(m_w - M)
  float mh[8], lh[8];                    // combine: per head M and L
  Seg seg[2];                            // segment e in slot e & 1
  int64_t u_next;                        // last cost unit before the last planned segment
  uint32_t skip0[NW];                    // per warp: bit j, the first copy j of the segment skips its page
  int ew;                                // the current segment's value-weight exponent (see build_qfrag)
  int last;                              // this CTA merges the segment just finished
};

// Rows of R_K that thread (part p, column c) of the q rotation uses: rows
// [p RP, (p + 1) RP) of column c.  R_K is written once, when the cache is
// created, so it may be read before the launch waits for the preceding grid.
template <int G, int GK>
struct RkRows {
  static constexpr int NPART = Smem<G, GK>::NPART;
  static constexpr int RP = (D + NPART - 1) / NPART;
  float v[RP];
};
template <int G, int GK>
__device__ __forceinline__ void load_rk(const DevCache& c, int layer, int head, RkRows<G, GK>& rk) {
  constexpr int RP = RkRows<G, GK>::RP;
  const int t = threadIdx.x, ch = t % D, part = t / D;
  const int r0 = part * RP, r1 = min(D, r0 + RP);
  const float* __restrict__ RK = c.rot_k + ((size_t)layer * c.Hkv + head) * D * D;
#pragma unroll
  for (int i = 0; i < RP; ++i) rk.v[i] = (r0 + i < r1) ? __ldg(RK + (size_t)(r0 + i) * D + ch) : 0.0f;
}

// The G query rows of (request, kv head): element t + k NTH of the G x 128 block
// in qv[k] (loaded ahead of the rotation, so that the load overlaps others).
template <int G, int GK>
struct QRows {
  static constexpr int N = (G * D + Tune<G, GK>::THREADS - 1) / Tune<G, GK>::THREADS;
  uint16_t v[N];
  float tau_v;   // the segment's value clip threshold (one thread)
};
template <int G, int GK>
__device__ __forceinline__ void load_q(const DevCache& c, int layer, const DecodeReq& R, int head,
                                       const uint16_t* __restrict__ q, QRows<G, GK>& qv) {
  constexpr int NTH = Tune<G, GK>::THREADS;
  qv.tau_v = threadIdx.x == D + G ? c.tau_v[(size_t)layer * c.Hkv + head] : 0.0f;
  const uint16_t* qrow = q + ((size_t)R.batch_row * c.Hq + (size_t)head * G) * D;
#pragma unroll
  for (int k = 0; k < QRows<G, GK>::N; ++k) {
    const int i = threadIdx.x + k * NTH;
    qv.v[k] = i < G * D ? qrow[i] : 0;
  }
}

// q_rot = q R_K for the G query heads of (request, kv head), written as the q
// operands (layout above).  Every thread of the CTA takes part: thread (part p,
// column c) sums rows [p RP, (p + 1) RP) of column c of R_K (held in rk).
template <int G, int GK>
__device__ __forceinline__ void build_qfrag(const DevCache& c, const QRows<G, GK>& qv, const RkRows<G, GK>& rkr,
                                            Smem<G, GK>& sm) {
  constexpr int NTH = Tune<G, GK>::THREADS, NPART = Smem<G, GK>::NPART;
  constexpr int RP = RkRows<G, GK>::RP;
  constexpr int REGS = QFrag<G>::REGS;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int ch = t % D, part = t / D;
  const int r0 = part * RP, r1 = min(D, r0 + RP);
  const float* rk = rkr.v;
#pragma unroll
  for (int k = 0; k < QRows<G, GK>::N; ++k) {
    const int i = t + k * NTH;
    if (i < G * D) sm.scr.pro.q[i % D][i / D] = __uint_as_float(static_cast<uint32_t>(qv.v[k]) << 16);
  }
  __syncthreads();
  // the G heads of a row in one load, two heads per packed fma (each an fmaf)
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.0f;
#pragma unroll
  for (int i = 0; i < RP; ++i) {
    if (r0 + i < r1) {
      const float* qr = sm.scr.pro.q[r0 + i];
      const float2 r2 = make_float2(rk[i], rk[i]);
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4) {
          const float4 x = *reinterpret_cast<const float4*>(qr + h);
          const float2 a = __ffma2_rn(make_float2(x.x, x.y), r2, make_float2(acc[h], acc[h + 1]));
          const float2 b = __ffma2_rn(make_float2(x.z, x.w), r2, make_float2(acc[h + 2], acc[h + 3]));
          acc[h] = a.x;
          acc[h + 1] = a.y;
          acc[h + 2] = b.x;
          acc[h + 3] = b.y;
        }
      } else if constexpr (G == 2) {
        const float2 a = __ffma2_rn(*reinterpret_cast<const float2*>(qr), r2, make_float2(acc[0], acc[1]));
        acc[0] = a.x;
        acc[1] = a.y;
      } else {
        acc[0] = fmaf(qr[0], rk[i], acc[0]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) sm.scr.pro.part[part][h][ch] = acc[h];
  // |q_h|^2 by the warps of part 0 (warp h), rounded up
  if (w < G) {
    const float4 x = make_float4(sm.scr.pro.q[4 * lane][w], sm.scr.pro.q[4 * lane + 1][w],
                                 sm.scr.pro.q[4 * lane + 2][w], sm.scr.pro.q[4 * lane + 3][w]);
    float n2 = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, x.w * x.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    if (lane == 0) sm.scr.pro.norm[w] = n2;
  }
  __syncthreads();
  if (t < D) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = sm.scr.pro.part[0][h][t];
#pragma unroll
      for (int p = 1; p < NPART; ++p) v += sm.scr.pro.part[p][h][t];
      sm.scr.pro.part[0][h][t] = v;
    }
  } else if (t < D + G) {
    // qscale(h) = 2^e, e = 15 - 24 - ceil(log2(|q|_2 1.001)) (read off the exponent of
    // the rounded-up norm), so |q_rot| qscale 2^24 <= 2^15
    const int h = t - D;
    const float n2 = sm.scr.pro.norm[h];
    int e = 0;
    if (n2 > 0.0f) {
      const uint32_t b = __float_as_uint(__fmul_ru(__fsqrt_ru(n2), 1.001f));
      const int ceil_log2 = static_cast<int>((b >> 23) & 0xffu) - 127 + ((b & 0x7fffffu) != 0u ? 1 : 0);
      e = 15 - 24 - ceil_log2;
    }
    sm.scr.pro.qe[h] = max(-60, min(e, 60));
  } else if (t == D + G) {
    // value weights p s_v are prescaled by 2^ew so the smallest ones stay representable
    // in fp16: s_v <= fp16(2 tau_V / 3) and p <= 2^LAZY_MAX, so p s_v 2^ew <= 2^15
    const float smax = qv.tau_v * (2.0f / 3.0f) * 1.002f;
    sm.ew = max(-60, min(60, static_cast<int>(floorf(log2f(32768.0f / smax))) - LAZY_MAX_INT));
  }
  __syncthreads();
  // 2^e for the small exponents here (normal range): built from its bits
  auto pow2 = [](int e) { return __int_as_float((e + 127) << 23); };
  auto qexp = [&](int h) { return sm.scr.pro.qe[h]; };
  uint32_t* dst = sm.qf;
  for (int wi = t; wi < 32 * REGS; wi += NTH) {
    const int lane_w = wi / REGS, k = wi % REGS;
    const int gid = lane_w >> 2, tid = lane_w & 3;
    const int nt = k >> 4, s = (k >> 1) & 7, rr = k & 1;
    const int h = 4 * nt + (gid >> 1);
    uint32_t word = 0u;
    if (h < G) {
      const int m = 2 * (s & 3) + rr;
      const int chn = GK == 128 ? 32 * tid + 16 * (s >> 2) + m : 64 * (s >> 2) + 16 * tid + m;
      const float f = pow2(qexp(h) + 24 - 2 * code_exp(m));
      float ha, la, hb, lb;
      split_half(sm.scr.pro.part[0][h][chn] * f, ha, la);
      split_half(sm.scr.pro.part[0][h][chn + 8] * f, hb, lb);
      word = (gid & 1) ? pack_half2(la, lb) : pack_half2(ha, hb);
    }
    dst[wi] = word;
  }
  float* consts = reinterpret_cast<float*>(dst + QFrag<G>::CONSTS);
  if (t < 8) consts[t] = t < G ? c.scale * LOG2E * pow2(-qexp(t)) : 0.0f;
  // slab sums: warp (slab, head) pairs, lane over the slab's 32 channels
  for (int pr = w; pr < SLABS * 8; pr += NTH / 32) {
    const int sl = pr / 8, h = pr % 8;
    float v = h < G ? sm.scr.pro.part[0][h][32 * sl + lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) consts[8 + 8 * sl + h] = v;
  }
  __syncthreads();
}

// The warps' states in shared memory (sm.state[w][h]: o[128], m, l) combined
// into one record per query head at part_out (o[128], M, L): warp 0 forms the
// per-(warp, head) factors 2^(m_w - M), then every thread sums (head, channel)
// pairs over the warps.
template <int G, int GK>
__device__ __forceinline__ void cta_combine(Smem<G, GK>& sm, float* part_out) {
  constexpr int NW = Tune<G, GK>::NW, NTH = Tune<G, GK>::THREADS;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  static_assert(G <= NW, "one warp per head forms the factors");
  __syncthreads();   // every warp's state is in shared memory
  if (warp < G) {
    // warp h: lane w holds warp w's (m, l) of head h
    const int h = warp;
    const float m = lane < NW ? sm.state[lane][h][PARTIAL_M] : -INFINITY;
    const float lw = lane < NW ? sm.state[lane][h][PARTIAL_L] : 0.0f;
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = m == -INFINITY ? 0.0f : exp2f(m - M);
    float l = lw * f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane < NW) sm.wf[lane][h] = f;
    if (lane == 0) {
      sm.mh[h] = M;
      sm.lh[h] = l;
    }
  }
  __syncthreads();
  for (int i = t; i < G * D; i += NTH) {
    const int h = i / D, ch = i % D;
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) acc = fmaf(sm.state[w][h][ch], sm.wf[w][h], acc);
    part_out[h * PART + ch] = acc;
  }
  if (t < G) {
    part_out[t * PART + PARTIAL_M] = sm.mh[t];
    part_out[t * PART + PARTIAL_L] = sm.lh[t];
  }
  __syncthreads();   // the states are read before the rings are reused
}

// Bounded wait (one thread) for the append of (request R, kv head) in this step
// launch: its BF16 CTA releases dec_flag = epoch once the demoted token is in the
// hot page (and a new page is in the page table).  False, with ERR_TIMEOUT
// reported, if it gave up.  The hot page is then read through the async proxy.
__device__ __noinline__ bool wait_append(const DevCache& c, const DecodeReq& R, int head, uint32_t epoch,
                                         uint32_t limit) {
  const uint32_t* f = c.dec_flag + (size_t)R.slot * c.Hkv + head;
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v == epoch) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    __nanosleep(256);
  }
  atomicOr(c.err, ERR_TIMEOUT);
  return false;
}

// The first STAGES page copies of warp w's share of a segment's pages [p0, p1)
// (pages p0 + w + NW j, j < STAGES), by lane 0, into stages nc + j; the hot page
// (written by this step's append, epoch != 0) only once that append is done.  Copy
// number `hold` of warp 0 is not issued (failure-detection hook; -1: none), and a
// warp whose earlier wait ran out issues nothing (it would never wait for it).
// phase 1 issues only the copies of pages below npages - 2 (those no decode step
// launched just before can be writing), phase 2 the others, phase 0 all.
template <int G, int GK>
__device__ __forceinline__ void int2_issue_first(const DevCache& c, int layer, const DecodeReq& R, int head, int p0,
                                                 int p1, Smem<G, GK>& sm, uint32_t epoch, uint32_t limit, uint32_t nc,
                                                 int hold, bool timed_out, int phase = 0) {
  constexpr int NW = Tune<G, GK>::NW;
  constexpr int REC = record_for(GK);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane != 0 || timed_out) return;
  // the rings may have been written through the generic proxy since their last copy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const int32_t* pt = c.hist_pt + (size_t)R.slot * c.max_pages;
  const uint8_t* base = c.int2 + layer * c.int2_layer_stride + (size_t)head * REC;
  int32_t ids[STAGES];
#pragma unroll
  for (int j = 0; j < STAGES; ++j) {
    const int pi = p0 + warp + NW * j;
    ids[j] = (pi < p1 && !(epoch != 0 && pi == R.hot_page)) ? __ldcg(pt + pi) : 0;
  }
#pragma unroll
  for (int j = 0; j < STAGES; ++j) {
    const int pi = p0 + warp + NW * j;
    if (pi >= p1) break;
    if (phase != 0 && (pi < R.npages - 2) != (phase == 1)) continue;
    int32_t id = ids[j];
    bool bad = false;
    if (epoch != 0 && pi == R.hot_page) {
      wait_append(c, R, head, epoch, limit);
      id = __ldcg(pt + pi);
    }
    if (id < 0 || id >= c.n_int2_pages) {
      atomicOr(c.err, ERR_INT2_PAGE);
      id = 0;
      bad = true;
    }
    // the page loop skips a bad page (page 0 is copied in its place)
    sm.skip0[warp] = bad ? (sm.skip0[warp] | (1u << j)) : (sm.skip0[warp] & ~(1u << j));
    if (warp == 0 && static_cast<int>(nc + j) == hold) continue;
    const int st = (nc + j) % STAGES;
    mbar_expect_tx(&sm.bar[warp][st], REC);
    tma_load_1d(sm.buf.ring[warp][st], base + (size_t)id * c.Hkv * REC, REC, &sm.bar[warp][st]);
  }
}

// The INT2 pages [p0, p1) of one (request, kv head) segment that this CTA holds:
// warp w takes pages p0 + w, p0 + w + NW, ... through its TMA ring (copy number
// nc counts the copies this warp has consumed so far, across segments); qf holds
// the segment's q operands.  Leaves the CTA's partial (rotated basis) for every
// query head of the group in part_out.  A wait that runs out (limit rounds) sets
// timed_out for the whole warp: it reports ERR_TIMEOUT, issues no further copy,
// lets the copies it has in flight land and skips the rest of its pages.  Copy
// number `hold` of warp 0 is never issued (failure-detection hook; -1: none).
template <int G, int GK>
__device__ __forceinline__ void int2_pages(const DevCache& c, int layer, const DecodeReq& R, int head, int p0,
                                           int p1, const uint32_t* __restrict__ qf, Smem<G, GK>& sm,
                                           float* part_out, uint32_t limit, uint32_t epoch, uint32_t& nc,
                                           bool& timed_out, int hold) {
  constexpr int NW = Tune<G, GK>::NW;
  constexpr int NT = QFrag<G>::NT;       // n-tiles of 8 columns = 4 heads x (hi, lo)
  constexpr int REC = record_for(GK);
  constexpr int NGR = D / GK;            // quantisation groups per token-head
  constexpr int KMETA = k_meta_off_for(GK), VMETA = v_meta_off_for(GK), MB = meta_bytes_for(GK);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid = lane & 3;
  const int nhist = R.hist_end - SINK;
  const int my_n = (p1 - p0 > warp) ? (p1 - p0 - warp + NW - 1) / NW : 0;
  const int32_t* pt = c.hist_pt + (size_t)R.slot * c.max_pages;
  const uint8_t* base = c.int2 + layer * c.int2_layer_stride + (size_t)head * REC;
  const size_t pstride = (size_t)c.Hkv * REC;
  const int hot = epoch != 0 ? R.hot_page : -1;

  // page ids of this warp's pages, read 32 at a time (lane l holds page 32 b + l of
  // batch b); page_src is called by the whole warp with increasing j.  An id is a
  // page (>= 0), HOT_ID (resolved at copy time) or BAD_ID: out of range, reported;
  // page 0 is copied in its place (keeping the ring's sequence) and skipped.
  constexpr int32_t HOT_ID = -1, BAD_ID = -2;
  int32_t batch_pages = 0;
  int batch_idx = -1;
  auto checked = [&](int32_t page) -> int32_t {
    if (page < 0 || page >= c.n_int2_pages) {
      atomicOr(c.err, ERR_INT2_PAGE);
      return BAD_ID;
    }
    return page;
  };
  // the hot page (written by this step's append) is read only after that append
  // is done: its id is fetched by lane 0 at copy time, after the wait
  auto page_src = [&](int j, bool& skip) -> const uint8_t* {
    const int b = j >> 5;
    if (b != batch_idx) {
      batch_idx = b;
      const int jj = 32 * b + lane;
      const int pj = p0 + warp + NW * jj;
      int32_t page = 0;
      if (jj < my_n) page = pj == hot ? HOT_ID : checked(__ldcg(pt + pj));
      batch_pages = page;
    }
    int32_t page = __shfl_sync(0xffffffffu, batch_pages, j & 31);
    if (page == HOT_ID) {   // warp-uniform
      if (lane == 0) {
        wait_append(c, R, head, epoch, limit);
        page = checked(__ldcg(pt + hot));
      }
      page = __shfl_sync(0xffffffffu, page, 0);
    }
    skip = page < 0;
    return base + (size_t)max(page, 0) * pstride;
  };
  // bit st: the page in stage st is skipped (bad id)
  uint32_t skip_bits = 0u;
  auto note = [&](int j, bool skip) {
    const uint32_t bit = 1u << ((nc + j) % STAGES);
    skip_bits = skip ? (skip_bits | bit) : (skip_bits & ~bit);
  };
  auto held = [&](int j) { return warp == 0 && static_cast<int>(nc + j) == hold; };
  // the first STAGES copies were issued by int2_issue_first, which left their skip
  // flags in skip0 (the page ids of the later copies are read at the first refill)
  {
    const uint32_t s0 = sm.skip0[warp];
#pragma unroll
    for (int j = 0; j < STAGES; ++j) note(j, (s0 >> j) & 1u);
  }
  // weights p * s_v are prescaled by 2^ew (formed with the q operands)
  const int ew = sm.ew;
  const float wscale = __int_as_float((ew + 127) << 23);

  // B operands of q_rot . c, and the per-head logit constants of this lane's head
  uint32_t bq[NT][8][2];
  {
    const uint4* src = reinterpret_cast<const uint4*>(qf + (size_t)lane * QFrag<G>::REGS);
    uint4 v[QFrag<G>::REGS / 4];
#pragma unroll
    for (int u = 0; u < QFrag<G>::REGS / 4; ++u) v[u] = src[u];
#pragma unroll
    for (int u = 0; u < QFrag<G>::REGS / 4; ++u) {
      const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 4 * u + e;
        bq[k >> 4][(k >> 1) & 7][k & 1] = w4[e];
      }
    }
  }
  // kz[nt][g]: scale log2(e) times the sum of q_rot over group g's channels (its slabs)
  float ks[NT], kz[NT][NGR];
  {
    const float* consts = reinterpret_cast<const float*>(qf + QFrag<G>::CONSTS);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      ks[nt] = consts[4 * nt + tid];
#pragma unroll
      for (int g = 0; g < NGR; ++g) {
        float sum = 0.0f;
#pragma unroll
        for (int sl = g * (SLABS / NGR); sl < (g + 1) * (SLABS / NGR); ++sl) sum += consts[8 + 8 * sl + 4 * nt + tid];
        kz[nt][g] = c.scale * LOG2E * sum;
      }
    }
  }

  float o[NT][8][4];
  // l and u are kept as two partial sums (tokens gid and gid + 8 of each m-tile)
  // so that the page's pairs update them with packed fp32 instructions
  float m_run[NT];
  float2 l_run[NT], u_run[NT][NGR];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int g = 0; g < NGR; ++g) u_run[nt][g] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][mt][e] = 0.0f;
  }

  int done = 0;   // copies of this segment consumed by this warp
  bool timed_here = false;
  for (int j = 0; j < my_n && !timed_out; ++j) {
    const int stg = (nc + j) % STAGES;
    const int pi = p0 + warp + NW * j;
    // one decision for the whole warp, so that its lanes never diverge
    const bool landed = mbar_wait(&sm.bar[warp][stg], ((nc + j) / STAGES) & 1, limit);
    if (!__all_sync(0xffffffffu, landed)) {
      timed_out = timed_here = true;
      if (lane == 0) atomicOr(c.err, ERR_TIMEOUT);
      break;
    }
    done = j + 1;
    if (!((skip_bits >> stg) & 1u)) {   // a page with a bad id contributes nothing
      const uint8_t* rec = sm.buf.ring[warp][stg];
      const int valid = min(PAGE, nhist - pi * PAGE);


      // ---- logits: 4 m-tiles of 16 tokens x NT n-tiles, K = 128 channels; with
      // G_K = 64 the k-steps of each group accumulate apart (acc[g])
      float acc[NGR][NT][4][4];
  #pragma unroll
      for (int g = 0; g < NGR; ++g)
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
          for (int mt = 0; mt < 4; ++mt)
  #pragma unroll
            for (int e = 0; e < 4; ++e) acc[g][nt][mt][e] = 0.0f;
  #pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint2 ka, kb;
        if constexpr (GK == 128) {
          // channels 32 tid .. 32 tid + 31 of tokens 16 mt + gid and + 8
          ka = *reinterpret_cast<const uint2*>(rec + K_CODES_OFF + (16 * mt + gid) * CODE_BYTES + 8 * tid);
          kb = *reinterpret_cast<const uint2*>(rec + K_CODES_OFF + (16 * mt + gid + 8) * CODE_BYTES + 8 * tid);
        } else {
          // channels 16 tid .. 16 tid + 15 of group 0 (.x) and of group 1 (.y)
          const uint8_t* ra = rec + K_CODES_OFF + (16 * mt + gid) * CODE_BYTES;
          const uint8_t* rb = ra + 8 * CODE_BYTES;
          ka = make_uint2(*reinterpret_cast<const uint32_t*>(ra + 4 * tid),
                          *reinterpret_cast<const uint32_t*>(ra + 16 + 4 * tid));
          kb = make_uint2(*reinterpret_cast<const uint32_t*>(rb + 4 * tid),
                          *reinterpret_cast<const uint32_t*>(rb + 16 + 4 * tid));
        }
        const uint2 kas = make_uint2(ka.x >> 10, ka.y >> 10);
        const uint2 kbs = make_uint2(kb.x >> 10, kb.y >> 10);
  #pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t wa = s < 4 ? ka.x : ka.y, was = s < 4 ? kas.x : kas.y;
          const uint32_t wb = s < 4 ? kb.x : kb.y, wbs = s < 4 ? kbs.x : kbs.y;
          const int m0 = 2 * (s & 3);
          const uint32_t a0 = code_pair2(wa, was, m0), a1 = code_pair2(wb, wbs, m0);
          const uint32_t a2 = code_pair2(wa, was, m0 + 1), a3 = code_pair2(wb, wbs, m0 + 1);
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma16816(acc[NGR == 2 ? (s >> 2) : 0][nt][mt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
        }
      }
      // token meta of this lane's 8 tokens: 16 mt + gid + 8 rr; a partial page (the
      // last of the history) masks the rows past its end
      // the page's metadata converted once per token (lanes l and l + 32), not once
      // per query head: {s_k, z_k, s_v 2^ew, z_v}, value terms zeroed past the end
  #pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int tok = lane + 32 * hh;
        const bool ok = tok < valid;
  #pragma unroll
        for (int g = 0; g < NGR; ++g) {
          const __half2 km = *reinterpret_cast<const __half2*>(rec + KMETA + tok * MB + 4 * g);
          const __half2 vm = *reinterpret_cast<const __half2*>(rec + VMETA + tok * MB + 4 * g);
          const float4 mv = make_float4(__low2float(km), __high2float(km), ok ? __low2float(vm) * wscale : 0.0f,
                                        ok ? __high2float(vm) : 0.0f);
          if (g == 0)
            sm.meta[warp][tok] = mv;
          else
            sm.meta2[warp][tok] = mv;
        }
      }
      __syncwarp();
      // logits in the log2 domain, as pairs (token 16 mt + gid, that token + 8)
      float2 lg[NT][4], sw[NGR][4], zv[NGR][4];
      auto epilogue = [&](auto full_page) {
        constexpr bool FULL = decltype(full_page)::value;
  #pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const int tok = 16 * mt + gid;
          const float4 m0 = sm.meta[warp][tok], m1 = sm.meta[warp][tok + 8];
          sw[0][mt] = make_float2(m0.z, m1.z);
          zv[0][mt] = make_float2(m0.w, m1.w);
          [[maybe_unused]] float4 n0 = m0, n1 = m1;   // group 1's meta (G_K = 64)
          if constexpr (NGR == 2) {
            n0 = sm.meta2[warp][tok];
            n1 = sm.meta2[warp][tok + 8];
            sw[NGR - 1][mt] = make_float2(n0.z, n1.z);
            zv[NGR - 1][mt] = make_float2(n0.w, n1.w);
          }
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            // hi + lo columns, then s_k kscale acc + z_k (scale log2 e sum q_rot), per group
            const float2 a = __fadd2_rn(make_float2(acc[0][nt][mt][0], acc[0][nt][mt][2]),
                                        make_float2(acc[0][nt][mt][1], acc[0][nt][mt][3]));
            const float2 sk = __fmul2_rn(make_float2(m0.x, m1.x), make_float2(ks[nt], ks[nt]));
            const float2 zk = __fmul2_rn(make_float2(m0.y, m1.y), make_float2(kz[nt][0], kz[nt][0]));
            float2 v = __ffma2_rn(sk, a, zk);
            if constexpr (NGR == 2) {
              const float2 a1 = __fadd2_rn(make_float2(acc[NGR - 1][nt][mt][0], acc[NGR - 1][nt][mt][2]),
                                           make_float2(acc[NGR - 1][nt][mt][1], acc[NGR - 1][nt][mt][3]));
              const float2 sk1 = __fmul2_rn(make_float2(n0.x, n1.x), make_float2(ks[nt], ks[nt]));
              const float2 zk1 = __fmul2_rn(make_float2(n0.y, n1.y),
                                            make_float2(kz[nt][NGR - 1], kz[nt][NGR - 1]));
              v = __ffma2_rn(sk1, a1, __fadd2_rn(v, zk1));
            }
            const bool head_ok = 4 * nt + 4 <= G || 4 * nt + tid < G;
            if (!FULL || !head_ok) {
              v.x = (head_ok && tok < valid) ? v.x : -INFINITY;
              v.y = (head_ok && tok + 8 < valid) ? v.y : -INFINITY;
            }
            lg[nt][mt] = v;
          }
        }
      };
      if (valid == PAGE)
        epilogue(std::true_type{});
      else
        epilogue(std::false_type{});
      // ---- online softmax per head (lanes with equal tid share a head); the
      // weights p s_v 2^ew go to shared memory as fp16 hi / lo halves.  Within each
      // 16-token group the weight rows hold token 16 g + r at position 16 g + 2 r
      // (r < 8) or 16 g + 2 (r - 8) + 1, so a lane's pair is one 32-bit store; the
      // value contraction below takes its k index in the same order.
      uint16_t(*wh)[2][WH_STRIDE];
      if constexpr (kWeightsInRing<G, GK>) {
        wh = reinterpret_cast<uint16_t(*)[2][WH_STRIDE]>(sm.buf.ring[warp][stg] + K_CODES_OFF);
        __syncwarp();   // every lane is done reading this page's K codes
      } else {
        wh = sm.w.wh[warp];
      }
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pm = fmaxf(lg[nt][0].x, lg[nt][0].y);
  #pragma unroll
        for (int mt = 1; mt < 4; ++mt) pm = fmaxf(pm, fmaxf(lg[nt][mt].x, lg[nt][mt].y));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
        // the reference max m_run moves only when a page exceeds it by more than
        // LAZY_MAX (log2 units): weights stay below 2^LAZY_MAX and the accumulators
        // are rescaled on few pages
        if (pm > m_run[nt] + LAZY_MAX) {
          const float corr = ex2(m_run[nt] - pm);
          m_run[nt] = pm;
          l_run[nt] = __fmul2_rn(l_run[nt], make_float2(corr, corr));
  #pragma unroll
          for (int g = 0; g < NGR; ++g) u_run[nt][g] = __fmul2_rn(u_run[nt][g], make_float2(corr, corr));
  #pragma unroll
          for (int mt = 0; mt < 8; ++mt)
  #pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][mt][e] *= corr;
        }
        const float2 neg_ref = make_float2(-m_run[nt], -m_run[nt]);
        const int h = 4 * nt + tid;
  #pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const float2 d = __fadd2_rn(lg[nt][mt], neg_ref);
          const float2 p = make_float2(ex2(d.x), ex2(d.y));
          l_run[nt] = __fadd2_rn(l_run[nt], p);
  #pragma unroll
          for (int g = 0; g < NGR; ++g) u_run[nt][g] = __ffma2_rn(p, zv[g][mt], u_run[nt][g]);
          if (h < G) {
            const int pos = 16 * mt + 2 * gid;
  #pragma unroll
            for (int g = 0; g < NGR; ++g) {
              const float2 w = __fmul2_rn(p, sw[g][mt]);
              const __half2 hi = __float22half2_rn(w);
              const float2 lo = __ffma2_rn(__half22float2(hi), make_float2(-1.0f, -1.0f), w);
              *reinterpret_cast<__half2*>(&wh[NGR * h + g][0][pos]) = hi;
              *reinterpret_cast<__half2*>(&wh[NGR * h + g][1][pos]) = __float22half2_rn(lo);
            }
          }
        }
      }
      __syncwarp();
      // ---- values: 8 m-tiles of 16 channels x NT n-tiles, K = 64 tokens; k index
      // 2 j + b of step s is token 16 s + j + 8 b
  #pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int ta = 16 * s + 2 * tid;
        uint32_t bw[NGR][NT][2];
  #pragma unroll
        for (int g = 0; g < NGR; ++g)
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int h = 4 * nt + (gid >> 1);
            if (h < G) {
              const uint16_t* row = wh[NGR * h + g][gid & 1];
              bw[g][nt][0] = *reinterpret_cast<const uint32_t*>(row + ta);
              bw[g][nt][1] = *reinterpret_cast<const uint32_t*>(row + ta + 8);
            } else {
              bw[g][nt][0] = bw[g][nt][1] = 0u;
            }
          }
        const int tb = 16 * s + tid;
        if constexpr (GK == 128) {
          // row gid of m-tile mt: channel 16 gid + mt; row gid + 8: 16 gid + 8 + mt
          const uint32_t* vrow = reinterpret_cast<const uint32_t*>(rec + V_CODES_OFF) + gid;
          const uint32_t wa = vrow[tb * (CODE_BYTES / 4)], wb = vrow[(tb + 8) * (CODE_BYTES / 4)];
          const uint32_t wc = vrow[(tb + 4) * (CODE_BYTES / 4)], wd = vrow[(tb + 12) * (CODE_BYTES / 4)];
          const uint32_t x1 = __byte_perm(wa, wb, 0x5410), y1 = __byte_perm(wa, wb, 0x7632);
          const uint32_t x2 = __byte_perm(wc, wd, 0x5410), y2 = __byte_perm(wc, wd, 0x7632);
          const uint32_t x1s = x1 >> 10, y1s = y1 >> 10;
          const uint32_t x2s = x2 >> 10, y2s = y2 >> 10;
  #pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t a0 = code_pair2(x1, x1s, mt), a1 = code_pair2(y1, y1s, mt);
            const uint32_t a2 = code_pair2(x2, x2s, mt), a3 = code_pair2(y2, y2s, mt);
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(o[nt][mt], a0, a1, a2, a3, bw[0][nt][0], bw[0][nt][1]);
          }
        } else {
          // group-pure m-tiles: m-tile 4 g + j, row gid holds channel 64 g + 8 gid + j and
          // row gid + 8 channel 64 g + 8 gid + 4 + j (16-bit half gid & 1 of word 4 g + gid / 2)
          const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
  #pragma unroll
          for (int g = 0; g < NGR; ++g) {
            const uint32_t* vrow = reinterpret_cast<const uint32_t*>(rec + V_CODES_OFF) + 4 * g + (gid >> 1);
            const uint32_t wa = vrow[tb * (CODE_BYTES / 4)], wb = vrow[(tb + 8) * (CODE_BYTES / 4)];
            const uint32_t wc = vrow[(tb + 4) * (CODE_BYTES / 4)], wd = vrow[(tb + 12) * (CODE_BYTES / 4)];
            const uint32_t x1 = __byte_perm(wa, wb, sel), x2 = __byte_perm(wc, wd, sel);
            const uint32_t x1s = x1 >> 10, x2s = x2 >> 10;
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t a0 = code_pair2(x1, x1s, j), a1 = code_pair2(x1, x1s, j + 4);
              const uint32_t a2 = code_pair2(x2, x2s, j), a3 = code_pair2(x2, x2s, j + 4);
  #pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma16816(o[nt][4 * g + j], a0, a1, a2, a3, bw[g][nt][0], bw[g][nt][1]);
            }
          }
        }
      }
      __syncwarp();
    }
    if (j + STAGES < my_n) {
      bool skip;
      const uint8_t* src = page_src(j + STAGES, skip);
      note(j + STAGES, skip);
      if (lane == 0 && !held(j + STAGES)) {
        // the weights were written to this buffer through the generic proxy
        if constexpr (kWeightsInRing<G, GK>) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(&sm.bar[warp][stg], REC);
        tma_load_1d(sm.buf.ring[warp][stg], src, REC, &sm.bar[warp][stg]);
      }
    }
  }
  if (timed_here && lane == 0) {
    // let every copy this warp issued land (bounded) before the buffers are reused:
    // the copies done .. min(done + STAGES, my_n) - 1 may still be in flight
    for (int j = done; j < min(done + STAGES, my_n); ++j)
      if (!held(j)) mbar_wait(&sm.bar[warp][(nc + j) % STAGES], ((nc + j) / STAGES) & 1, DECODE_WAIT_LIMIT);
  }
  nc += static_cast<uint32_t>(my_n);

  // ---- this warp's state -> shared memory (rotated basis, unscaled, z term added)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float l = l_run[nt].x + l_run[nt].y, u[NGR];
#pragma unroll
    for (int g = 0; g < NGR; ++g) u[g] = u_run[nt][g].x + u_run[nt][g].y;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
      for (int g = 0; g < NGR; ++g) u[g] += __shfl_xor_sync(0xffffffffu, u[g], off);
    }
    const int h = 4 * nt + tid;
    if (h < G) {
      float* st = sm.state[warp][h];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        if constexpr (GK == 128) {
          const float f = ldexpf(1.0f, 24 - 2 * code_exp(mt) - ew);
          st[16 * gid + mt] = fmaf(o[nt][mt][0] + o[nt][mt][1], f, u[0]);
          st[16 * gid + 8 + mt] = fmaf(o[nt][mt][2] + o[nt][mt][3], f, u[0]);
        } else {
          const int g = mt >> 2, j = mt & 3;
          const float f0 = ldexpf(1.0f, 24 - 2 * code_exp(j) - ew);
          const float f1 = ldexpf(1.0f, 24 - 2 * code_exp(j + 4) - ew);
          st[64 * g + 8 * gid + j] = fmaf(o[nt][mt][0] + o[nt][mt][1], f0, u[g]);
          st[64 * g + 8 * gid + 4 + j] = fmaf(o[nt][mt][2] + o[nt][mt][3], f1, u[g]);
        }
      }
      if (gid == 0) {
        st[PARTIAL_M] = m_run[nt];
        st[PARTIAL_L] = l;
      }
    }
  }
  cta_combine<G, GK>(sm, part_out);
}

// ---- BF16 sink and recent pages ------------------------------------------------------
constexpr int BF_SUB = 16;                            // rows per sub-page (one k-step of P V)
constexpr int BF_SUBS = BF16_ITEMS * PAGE / BF_SUB;   // 20 sub-pages per segment
constexpr int BF_WPITCH = BF_SUB + 8;                 // bf16 per weight column

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ uint32_t word_of(const uint4 (&v)[4], int w) {
  const uint4 x = v[w >> 2];
  return (w & 3) == 0 ? x.x : (w & 3) == 1 ? x.y : (w & 3) == 2 ? x.z : x.w;
}
__device__ __forceinline__ uint32_t word_of(const uint4 (&v)[2], int w) {
  const uint4 x = v[w >> 2];
  return (w & 3) == 0 ? x.x : (w & 3) == 1 ? x.y : (w & 3) == 2 ? x.z : x.w;
}

// Whether BF16 row r of item `which` (0 sink, 1..4 ring pages) holds a cached token:
// sink rows [0, min(T, 64)); ring slot s = 64 (which - 1) + r holds position
// he + ((s - (he - 64)) mod 256), cached while below T.
__device__ __forceinline__ bool bf16_row_valid(const DecodeReq& R, int which, int r) {
  const int T = R.tokens, he = R.hist_end;
  if (which == 0) return r < min(T, SINK);
  if (T <= SINK) return false;
  const int s = PAGE * (which - 1) + r;
  const int p = he + ((s - (he - SINK)) % RECENT + RECENT) % RECENT;
  return p < T;
}

// The sink page and the four recent-ring pages of one (request, kv head), with the
// unrotated q, as 16-row sub-pages spread over the CTA's warps (warp w takes
// sub-pages w, w + NW, ... of the twenty; a sub-page without a cached row is
// skipped).  q K^T and P V run on mma.sync m16n8k16 bf16 with fp32 accumulation: q
// is exact in bf16, P is carried as bf16 hi + lo, so every product is exact.  The
// K and V rows go from global memory straight into the fragments (no shared
// memory staging), so the block runs while the segment's INT2 copies land in the
// rings:
//   * q K^T: A = K (16 rows x 16 channels per k-step); k index 2 tid + e of step s
//     is channel 32 tid + 4 s + e and 2 tid + 8 + e is 32 tid + 4 s + 2 + e, so
//     lane (gid, tid) reads 64 contiguous bytes of rows gid and gid + 8; B = q with
//     column n = head 4 nt + (n >> 1) (each head twice, the hi / lo pair of P V);
//   * P V^T: A = V^T (16 channels x 16 tokens); row gid of m-tile mt is channel
//     16 gid + 2 mt and row gid + 8 is that channel + 1, so lane (gid, tid) reads 32
//     contiguous bytes of each of its tokens 2 tid, 2 tid + 1, 2 tid + 8, 2 tid + 9
//     and pairs tokens with byte permutes; B = P, columns (head, hi / lo), through
//     the warp's weight columns in its meta rows.
// Rows outside the window are masked (K) or zeroed (V).  After a fused append the
// row of the appended token is read from that step's input (knew / vnew, the row
// of this request and kv head) rather than from the ring page the append writes,
// so no row depends on the append kernel's completion.  The CTA's partial for
// every query head of the group goes to part_out.
template <int G, int GK>
__device__ void bf16_block(const DevCache& c, int layer, const DecodeReq& R, int head,
                           const uint16_t* __restrict__ q, const uint16_t* knew, const uint16_t* vnew,
                           Smem<G, GK>& sm, float* part_out) {
  constexpr int NW = Tune<G, GK>::NW;
  constexpr int NT = QFrag<G>::NT;
  static_assert(NT * 8 * BF_WPITCH * 2 <= PAGE * sizeof(float4), "BF16 weights in the meta rows");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const float scale2 = c.scale * LOG2E;
  uint16_t(*wc)[8][BF_WPITCH] = reinterpret_cast<uint16_t(*)[8][BF_WPITCH]>(&sm.meta[warp][0]);
  // q as the B operand of K q^T
  uint32_t bq[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + (gid >> 1);
    uint4 qw[4];
    const uint4* qs =
        reinterpret_cast<const uint4*>(q + ((size_t)R.batch_row * c.Hq + (size_t)head * G + (h < G ? h : 0)) * D +
                                       32 * tid);
#pragma unroll
    for (int i = 0; i < 4; ++i) qw[i] = h < G ? __ldg(qs + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      bq[nt][st][0] = word_of(qw, 2 * st);
      bq[nt][st][1] = word_of(qw, 2 * st + 1);
    }
  }
  float o[NT][8][4];
  float m_run[NT], l_run[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][mt][e] = 0.0f;
  }
  // item and row of the appended token (position T - 1), when it is read from the step's input
  int new_which = -1, new_row = -1;
  if (knew != nullptr) {
    const int p = R.tokens - 1;
    if (p < SINK) {
      new_which = 0;
      new_row = p;
    } else {
      const int slot = (p - SINK) % RECENT;
      new_which = 1 + slot / PAGE;
      new_row = slot % PAGE;
    }
  }
  for (int sp = warp; sp < BF_SUBS; sp += NW) {
    const int which = sp / (PAGE / BF_SUB), r0 = BF_SUB * (sp % (PAGE / BF_SUB));
    // rows of this sub-page holding a cached token (bit i: row r0 + i); lanes 0..15 test one row each
    const uint32_t rows = __ballot_sync(0xffffffffu, lane < BF_SUB && bf16_row_valid(R, which, r0 + lane)) & 0xffffu;
    if (rows == 0u) continue;
    int page = which == 0 ? R.sink_page : R.ring_page[which - 1];
    if (page < 0 || page >= c.n_bf16_pages) {
      if (lane == 0) atomicOr(c.err, ERR_BF16_PAGE);
      page = 0;
    }
    const uint16_t* kb = c.bf16 + layer * c.bf16_layer_stride + ((size_t)page * c.Hkv + head) * BF16_RECORD_ELEMS +
                         (size_t)r0 * D;
    const uint16_t* vb = kb + (size_t)PAGE * D;
    const int nrow = which == new_which ? new_row - r0 : -1;   // row of the appended token in this sub-page
    auto krow = [&](int r) { return r == nrow ? knew : kb + (size_t)r * D; };
    auto vrow = [&](int r) { return r == nrow ? vnew : vb + (size_t)r * D; };
    // K rows gid and gid + 8, channels 32 tid .. 32 tid + 31 (a row outside the
    // window is read all the same -- in bounds -- and its logits are masked)
    uint4 ka[4], kc[4];
    {
      const uint4* pa = reinterpret_cast<const uint4*>(krow(gid) + 32 * tid);
      const uint4* pc = reinterpret_cast<const uint4*>(krow(gid + 8) + 32 * tid);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ka[i] = __ldg(pa + i);
        kc[i] = __ldg(pc + i);
      }
    }
    // V rows of tokens 2 tid, 2 tid + 1, 2 tid + 8, 2 tid + 9, channels 16 gid .. 16 gid + 15;
    // zero outside the window (P is zero there, and 0 x NaN would not be)
    uint4 vv[4][2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = 2 * tid + (k & 1) + 8 * (k >> 1);
      const bool ok = (rows >> r) & 1u;
      const uint4* pv = reinterpret_cast<const uint4*>(vrow(r) + 16 * gid);
      vv[k][0] = ok ? __ldg(pv) : make_uint4(0u, 0u, 0u, 0u);
      vv[k][1] = ok ? __ldg(pv + 1) : make_uint4(0u, 0u, 0u, 0u);
    }
    // ---- logits: S [16 rows x 8 columns] per n-tile over the 128 channels
    float sa[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[nt][e] = 0.0f;
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      const uint32_t a0 = word_of(ka, 2 * st), a1 = word_of(kc, 2 * st);
      const uint32_t a2 = word_of(ka, 2 * st + 1), a3 = word_of(kc, 2 * st + 1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(sa[nt], a0, a1, a2, a3, bq[nt][st][0], bq[nt][st][1]);
    }
    // ---- softmax of the lane's head 4 nt + tid over rows gid, gid + 8 (column 2 tid;
    // column 2 tid + 1 repeats it); the weights go to the warp's weight columns as
    // bf16 hi (column 2 tid) and lo (2 tid + 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const bool hok = 4 * nt + tid < G;
      const float la = (hok && ((rows >> gid) & 1u)) ? sa[nt][0] * scale2 : -INFINITY;
      const float lb = (hok && ((rows >> (gid + 8)) & 1u)) ? sa[nt][2] * scale2 : -INFINITY;
      float pm = fmaxf(la, lb);
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      if (pm > m_run[nt] + LAZY_MAX) {
        const float corr = m_run[nt] == -INFINITY ? 0.0f : ex2(m_run[nt] - pm);
        m_run[nt] = pm;
        l_run[nt] *= corr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][mt][e] *= corr;
      }
      const float pa = la == -INFINITY ? 0.0f : ex2(la - m_run[nt]);
      const float pb = lb == -INFINITY ? 0.0f : ex2(lb - m_run[nt]);
      l_run[nt] += pa + pb;
      const uint16_t ha = bf16_bits(pa), hb = bf16_bits(pb);
      wc[nt][2 * tid][gid] = ha;
      wc[nt][2 * tid][gid + 8] = hb;
      wc[nt][2 * tid + 1][gid] = bf16_bits(pa - __uint_as_float(static_cast<uint32_t>(ha) << 16));
      wc[nt][2 * tid + 1][gid + 8] = bf16_bits(pb - __uint_as_float(static_cast<uint32_t>(hb) << 16));
    }
    __syncwarp();
    // ---- values: O [128 channels x 8 columns] += V^T P over the 16 rows
    uint32_t bw[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bw[nt][0] = *reinterpret_cast<const uint32_t*>(&wc[nt][gid][2 * tid]);
      bw[nt][1] = *reinterpret_cast<const uint32_t*>(&wc[nt][gid][2 * tid + 8]);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint32_t w0 = word_of(vv[0], mt), w1 = word_of(vv[1], mt);
      const uint32_t w2 = word_of(vv[2], mt), w3 = word_of(vv[3], mt);
      const uint32_t a0 = __byte_perm(w0, w1, 0x5410), a1 = __byte_perm(w0, w1, 0x7632);
      const uint32_t a2 = __byte_perm(w2, w3, 0x5410), a3 = __byte_perm(w2, w3, 0x7632);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(o[nt][mt], a0, a1, a2, a3, bw[nt][0], bw[nt][1]);
    }
    __syncwarp();   // the weight columns are free
  }
  // ---- this warp's state -> shared memory: lane (gid, tid) holds head 4 nt + tid,
  // channels 16 gid .. 16 gid + 15
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float l = l_run[nt];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const int h = 4 * nt + tid;
    if (h < G) {
      float4* st = reinterpret_cast<float4*>(&sm.state[warp][h][16 * gid]);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st[k] = make_float4(o[nt][2 * k][0] + o[nt][2 * k][1], o[nt][2 * k][2] + o[nt][2 * k][3],
                            o[nt][2 * k + 1][0] + o[nt][2 * k + 1][1], o[nt][2 * k + 1][2] + o[nt][2 * k + 1][3]);
      if (gid == 0) {
        sm.state[warp][h][PARTIAL_M] = m_run[nt];
        sm.state[warp][h][PARTIAL_L] = l;
      }
    }
  }
  cta_combine<G, GK>(sm, part_out);
}

// ---- the decode kernel --------------------------------------------------------------
// First cost unit of INT2 CTA c: c total / n2 (64-bit), computed on the host at
// launch so that no CTA runs 64-bit divisions before its first pages.
__device__ __forceinline__ int64_t cta_begin(const DecodeArgs& a, int c) { return a.cstart[c]; }

// Cost units of one segment on the INT2 line: a set-up (the q rotation and the
// latency of the first pages, paid again by a CTA that enters the segment from
// another) then its pages; none for a request without history pages.
__device__ __forceinline__ int64_t seg_units(const DecodeReq& R) {
  return R.npages > 0 ? (int64_t)R.npages + DECODE_SEGMENT_SETUP_COST : 0;
}

// Segment containing INT2 cost unit u: request index, kv head, its first unit
// (requests without history pages hold no unit and are passed over).
__device__ __forceinline__ void segment_of(const DecodeArgs& a, int Hkv, int64_t u, int& ri, int& h, int64_t& s0) {
  ri = 0;
  while (ri + 1 < a.n && a.r[ri + 1].cost_start <= u) ++ri;
  const int64_t per = seg_units(a.r[ri]);
  h = static_cast<int>(static_cast<int32_t>(u - a.r[ri].cost_start) / static_cast<int32_t>(per));   // < 2^31
  if (h >= Hkv) h = Hkv - 1;
  s0 = a.r[ri].cost_start + (int64_t)h * per;
}

// INT2 CTA (index among the INT2 CTAs) whose cost range holds unit u.
__device__ __forceinline__ int cta_of(const DecodeArgs& a, int64_t u) {
  int lo = 0, hi = a.ncta - a.nbc - 1;   // the last CTA c with cstart[c] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.cstart[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// The INT2 CTAs that hold pages of a segment starting at cost unit s0 with
// units seg units: those whose ranges meet [page 0's unit, end).  A CTA whose
// range meets only the segment's set-up units takes no part in it.
__device__ __forceinline__ void segment_ctas(const DecodeArgs& a, int64_t s0, int64_t units, int& c_lo, int& c_hi) {
  c_lo = cta_of(a, s0 + DECODE_SEGMENT_SETUP_COST);
  c_hi = cta_of(a, s0 + units - 1);
}

// The segment holding INT2 cost unit u of this INT2 CTA's range [u0, u1), or
// the one before it where the range meets only u's segment's set-up units
// (invalid once u drops below u0); prev receives the unit before the segment.
// A CTA walks its segments from the last one back: a segment's last page (which
// a decode step's append may be filling) is then one of the last pages the CTA
// reads, long after the append is done.
__device__ Seg plan_segment(const DecodeArgs& a, int Hkv, int icta, int64_t u, int64_t u0, int64_t u1,
                            int64_t& prev) {
  Seg e{};
  prev = u0 - 1;
  while (u >= u0) {
    int ri, h;
    int64_t s0;
    segment_of(a, Hkv, u, ri, h, s0);
    const int64_t np = a.r[ri].npages;
    const int64_t f0 = s0 + DECODE_SEGMENT_SETUP_COST;   // unit of page 0
    const int64_t p0 = u0 > f0 ? (u0 - f0 < np ? u0 - f0 : np) : 0;
    const int64_t p1 = u1 > f0 ? (u1 - f0 < np ? u1 - f0 : np) : 0;
    if (p1 <= p0) {   // set-up units only: the next CTA takes this segment
      u = s0 - 1;
      continue;
    }
    prev = s0 - 1;
    e.valid = 1;
    e.ri = ri;
    e.head = h;
    e.p0 = static_cast<int>(p0);
    e.p1 = static_cast<int>(p1);
    e.slot = ri * Hkv + h + icta;
    segment_ctas(a, s0, seg_units(a.r[ri]), e.c_lo, e.c_hi);
    return e;
  }
  return e;
}

// Atomic add with release (this CTA's records, made visible to thread 0 by the
// barrier before it, are visible before the count) and acquire (the records of
// the CTAs counted before are visible after it) semantics at GPU scope.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The ring tail where a merge stages R_V^T (64 KiB; the records go to the start).
template <int G, int GK>
__device__ __forceinline__ float* merge_rvt(Smem<G, GK>& sm) {
  return reinterpret_cast<float*>(&sm.buf.ring[0][0][0] + sizeof(sm.buf.ring) - D * D * sizeof(float));
}
// R_V^T of (layer, kv head) into the ring tail, completion on mbar_r (one thread;
// the rings hold no copy in flight and were last written through the generic proxy).
template <int G, int GK>
__device__ __forceinline__ void issue_rvt(const DevCache& c, int layer, int head, Smem<G, GK>& sm) {
  constexpr uint32_t RVB = D * D * sizeof(float);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(&sm.mbar_r, RVB);
  tma_load_1d(merge_rvt(sm), c.rot_vt + ((size_t)layer * c.Hkv + head) * D * D, RVB, &sm.mbar_r);
}

// Merge of segment s = (ri, head) by the last CTA to finish it: the INT2 records
// of its n2 INT2 CTAs c_lo .. c_lo + n2 - 1 and its BF16 record, online-softmax
// combined per (query head, channel); then out = (O_bf16 + O_hist R_V^T) / L for
// the G query heads.  The records (consecutive in the workspace) are staged into
// the rings, which hold no copy at this point, by bulk copies of up to CAP
// records; the first copy also brings the BF16 record and R_V^T (to the end of
// the rings), so that everything the merge reads lands after one wait.
template <int G, int GK>
__device__ void merge_segment(const DevCache& c, int layer, const DecodeArgs& a, int ri, int head, int c_lo, int n2,
                              const float* recs, const float* bf16_recs, float* __restrict__ out, Smem<G, GK>& sm,
                              uint32_t& mphase, bool rvt_issued = false) {
  constexpr int NTH = Tune<G, GK>::THREADS, NPART = Smem<G, GK>::NPART;
  constexpr int PAIRS = (G * D + NTH - 1) / NTH;          // (head, channel) pairs per thread
  constexpr int RF = G * PART;                            // floats per record
  constexpr int RVB = D * D * int(sizeof(float));                            // R_V^T bytes
  constexpr int CAP = int((sizeof(sm.buf.ring) - RVB) / (RF * sizeof(float))) - 1;   // records per chunk
  constexpr int RP = (D + NPART - 1) / NPART;                                // R_V^T rows per part
  constexpr int U = 4;
  static_assert(CAP >= 1, "staging");
  const int t = threadIdx.x;
  const DecodeReq& R = a.r[ri];
  const int s = ri * c.Hkv + head;
  const int items = n2;
  float* stage = reinterpret_cast<float*>(&sm.buf.ring[0][0][0]);   // [CAP][RF], then the BF16 record
  float* rvt_s = merge_rvt(sm);   // R_V^T [D][D]
  // the copies are issued from the last warp, which has no head of its own below
  // (the issue of a large bulk copy holds up its warp for a while)
  auto issue = [&](int j0, int nk) {
    if (t == NTH - 32) {
      // the rings were last written through the generic proxy (weights), and the
      // records by other CTAs' generic stores (acquired through the counter)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_expect_tx(&sm.mbar_m, (nk + (j0 == 0 ? 1 : 0)) * RF * 4);
      if (nk > 0) tma_load_1d(stage, recs + (size_t)(s + c_lo + j0) * RF, nk * RF * 4, &sm.mbar_m);
      if (j0 == 0) {
        tma_load_1d(stage + CAP * RF, bf16_recs + (size_t)s * RF, RF * 4, &sm.mbar_m);
        if (!rvt_issued) issue_rvt(c, layer, head, sm);
      }
    }
  };
  issue(0, min(CAP, items));
  const int rch = t % D, rpart = t / D, r0 = rpart * RP;
  // per head g: running max M and sum L (warp g keeps them in registers, lane 0's
  // copy in sm.mh / sm.lh), and per chunk the records' weights 2^(m_j - M)
  float* wj = reinterpret_cast<float*>(&sm.meta[0][0]);   // [CAP][G]
  static_assert(CAP * G * sizeof(float) <= sizeof(sm.meta), "chunk weights in the meta rows");
  float Mw = -INFINITY, Lw = 0.0f;                          // warp g < G: head g
  float oh[PAIRS];
#pragma unroll
  for (int k = 0; k < PAIRS; ++k) oh[k] = 0.0f;
  const int warp = t >> 5, lane = t & 31;
  for (int j0 = 0; j0 == 0 || j0 < items; j0 += CAP) {   // the first chunk also brings the BF16 record
    const int nk = min(CAP, items - j0);
    if (j0 > 0) issue(j0, nk);
    if (!mbar_wait(&sm.mbar_m, mphase & 1u, DECODE_WAIT_LIMIT) && t == NTH - 32) atomicOr(c.err, ERR_TIMEOUT);
    mphase ^= 1u;
    if (warp < G) {
      const float* r = stage + warp * PART;
      float mn = Mw;
      for (int j = lane; j < nk; j += 32) mn = fmaxf(mn, r[j * RF + PARTIAL_M]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mn = fmaxf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      const float resc = Mw == -INFINITY ? 0.0f : exp2f(Mw - mn);
      float ls = 0.0f;
      for (int j = lane; j < nk; j += 32) {
        const float mj = r[j * RF + PARTIAL_M];
        const float f = mj == -INFINITY ? 0.0f : exp2f(mj - mn);
        wj[j * G + warp] = f;
        ls = fmaf(r[j * RF + PARTIAL_L], f, ls);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      Mw = mn;
      Lw = fmaf(Lw, resc, ls);
      if (lane == 0) {
        sm.mh[warp] = mn;
        sm.lh[warp] = Lw;
        sm.wf[0][warp] = resc;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < PAIRS; ++k) {
      const int i = t + k * NTH;
      if (i < G * D) {
        const int g = i / D, ch = i % D;
        const float* r = stage + g * PART + ch;
        float acc = oh[k] * sm.wf[0][g];
        for (int j = 0; j < nk; j += U) {
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (j + u < nk) acc = fmaf(r[(j + u) * RF], wj[(j + u) * G + g], acc);
        }
        oh[k] = acc;
      }
    }
    if (j0 + CAP >= items) break;   // the BF16 record is still staged: read below
    __syncthreads();                // the stage and the weights are read before the next chunk lands
  }
  float ob[PAIRS], lt[PAIRS];
#pragma unroll
  for (int k = 0; k < PAIRS; ++k) {
    const int i = t + k * NTH;
    const int g = i < G * D ? i / D : 0, ch = i % D;
    const float* rb = stage + CAP * RF + g * PART;   // the BF16 record
    const float bm = rb[PARTIAL_M], M = sm.mh[g];
    const float Mt = fmaxf(M, bm);
    const float fh = M == -INFINITY ? 0.0f : exp2f(M - Mt);
    const float fb = bm == -INFINITY ? 0.0f : exp2f(bm - Mt);
    if (i < G * D) sm.scr.mrg.hist[ch][g] = oh[k] * fh;
    ob[k] = rb[ch] * fb;
    lt[k] = fmaf(sm.lh[g], fh, rb[PARTIAL_L] * fb);
  }
  if (!mbar_wait(&sm.mbar_r, (mphase >> 1) & 1u, DECODE_WAIT_LIMIT) && t == NTH - 32) atomicOr(c.err, ERR_TIMEOUT);
  mphase ^= 2u;
  __syncthreads();
  {
    // O_hist R_V^T: thread (part p, column c) sums rows [p RP, (p + 1) RP) of column c
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.0f;
    const int r1 = min(D, r0 + RP);
#pragma unroll 4
    for (int j = r0; j < r1; ++j) {
      const float rv = rvt_s[j * D + rch];
      const float* hr = sm.scr.mrg.hist[j];
      const float2 r2 = make_float2(rv, rv);
      // the G heads of row j in one load, two heads per packed fma (each an fmaf)
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 x = *reinterpret_cast<const float4*>(hr + g);
          const float2 a = __ffma2_rn(make_float2(x.x, x.y), r2, make_float2(acc[g], acc[g + 1]));
          const float2 b = __ffma2_rn(make_float2(x.z, x.w), r2, make_float2(acc[g + 2], acc[g + 3]));
          acc[g] = a.x;
          acc[g + 1] = a.y;
          acc[g + 2] = b.x;
          acc[g + 3] = b.y;
        }
      } else if constexpr (G == 2) {
        const float2 a = __ffma2_rn(*reinterpret_cast<const float2*>(hr), r2, make_float2(acc[0], acc[1]));
        acc[0] = a.x;
        acc[1] = a.y;
      } else {
        acc[0] = fmaf(hr[0], rv, acc[0]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) sm.scr.mrg.part[rpart][g][rch] = acc[g];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < PAIRS; ++k) {
    const int i = t + k * NTH;
    if (i < G * D) {
      const int g = i / D, ch = i % D;
      float v = ob[k];
#pragma unroll
      for (int p = 0; p < NPART; ++p) v += sm.scr.mrg.part[p][g][ch];
      out[((size_t)R.batch_row * c.Hq + (size_t)head * G + g) * D + ch] = v / lt[k];
    }
  }
  __syncthreads();   // the scratch is free for the next q rotation
}

// The BF16 pages of segment (ri, head) into its BF16 record.
template <int G, int GK>
__device__ __forceinline__ void bf16_segment(const DevCache& c, int layer, const DecodeArgs& a, int ri, int head,
                                             const uint16_t* q, Smem<G, GK>& sm, float* bf16_recs) {
  const DecodeReq& R = a.r[ri];
  const size_t row = ((size_t)R.batch_row * c.Hkv + head) * D;
  bf16_block<G, GK>(c, layer, R, head, q, a.k_new ? a.k_new + row : nullptr, a.v_new ? a.v_new + row : nullptr, sm,
                    bf16_recs + (size_t)(ri * c.Hkv + head) * G * PART);
}

// This CTA is done with segment (ri, head), whose records come from n2 INT2 CTAs
// (c_lo ..) and one BF16 CTA: count it in the segment's counter.  When the BF16
// CTAs merge (bm: one segment each), an INT2 CTA only counts; otherwise the CTA
// that completes the count (n2 + 1) merges the segment.  The block before ends
// with a barrier, so every record store of this CTA comes before the count.
template <int G, int GK>
__device__ __forceinline__ void count_and_merge(const DevCache& c, int layer, const DecodeArgs& a, int ri, int head,
                                                int c_lo, int n2, const float* recs, const float* bf16_recs,
                                                float* out, Smem<G, GK>& sm, uint32_t& mphase, bool bm) {
  if (threadIdx.x == 32 * (Tune<G, GK>::NW - 1) + 1) {   // a thread that issues no page copy
    int* cnt = c.dec_count + (size_t)a.r[ri].slot * c.Hkv + head;
    const int last = !bm && atomic_add_acq_rel(cnt, 1) + 1 == n2 + 1;
    if (bm) atomic_add_acq_rel(cnt, 1);
    if (last) atomicExch(cnt, 0);   // ready for the next launch
    sm.last = last;
  }
  if (bm) return;
  __syncthreads();
  if (sm.last) merge_segment<G, GK>(c, layer, a, ri, head, c_lo, n2, recs, bf16_recs, out, sm, mphase);
}

// The BF16 CTA of segment (ri, head) merges it (bm): R_V^T is staged while it waits
// (bounded) for the count of the n2 INT2 CTAs, then the records are merged.
template <int G, int GK>
__device__ __forceinline__ void wait_and_merge(const DevCache& c, int layer, const DecodeArgs& a, int ri, int head,
                                               int c_lo, int n2, const float* recs, const float* bf16_recs,
                                               float* out, Smem<G, GK>& sm, uint32_t& mphase) {
  constexpr int NTH = Tune<G, GK>::THREADS;
  const int t = threadIdx.x;
  __syncthreads();   // the BF16 record is stored and the rings are free
  if (t == NTH - 32) issue_rvt(c, layer, head, sm);
  if (t == 32 * (Tune<G, GK>::NW - 1) + 1) {
    int* cnt = c.dec_count + (size_t)a.r[ri].slot * c.Hkv + head;
    bool done = false;
    // about as long as a page wait of the same limit (rounds of up to 20 us)
    for (uint32_t it = 0; it < 16u * a.dbg.wait_limit && !done; ++it) {
      int v;
      asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      done = v >= n2;
      if (!done) __nanosleep(64);
    }
    if (!done) atomicOr(c.err, ERR_TIMEOUT);
    atomicExch(cnt, 0);   // ready for the next launch
  }
  __syncthreads();
  merge_segment<G, GK>(c, layer, a, ri, head, c_lo, n2, recs, bf16_recs, out, sm, mphase, true);
}

// The append of the step's new token for (request ri, kv head), K and V: the
// demotion of the oldest recent token into the hot page where reqs[ri].hot_page is
// set, then the new rows (the inputs the write path would be given, derived from
// the post-step lengths), by two units of APPEND_THREADS threads (one after the
// other when the CTA has fewer than 2 APPEND_THREADS); then dec_flag = epoch is
// released for the CTA that streams the hot page.
template <int G, int GK>
__device__ void step_append(const DevCache& c, int layer, const DecodeArgs& a, int ri, int head, Smem<G, GK>& sm) {
  constexpr int NTH = Tune<G, GK>::THREADS;
  static_assert(NTH >= APPEND_THREADS && 2 * sizeof(AppendSmem) <= sizeof(sm.buf.ring), "append units");
  const DecodeReq& R = a.r[ri];
  AppendReq q;
  q.slot = R.slot;
  q.in_row = R.batch_row;
  const int p = R.tokens - 1;   // the appended token
  if (p < SINK) {
    q.dst_page = R.sink_page;
    q.dst_row = p;
  } else {
    const int sl = (p - SINK) % RECENT;
    q.dst_page = R.ring_page[sl / PAGE];
    q.dst_row = sl % PAGE;
  }
  q.demote_slot = q.hist_page = q.src_page = q.src_row = q.pt_index = -1;
  if (R.hot_page >= 0) {
    const int h = R.hist_end - 1 - SINK;   // history position of the demoted token; its ring slot is h mod 256
    q.demote_slot = h % PAGE;
    q.src_page = R.ring_page[(h % RECENT) / PAGE];
    q.src_row = (h % RECENT) % PAGE;
    if (R.hot_new >= 0) {
      q.hist_page = R.hot_new;
      q.pt_index = R.hot_page;
    } else {
      q.hist_page = __ldcg(c.hist_pt + (size_t)R.slot * c.max_pages + R.hot_page);
    }
  }
  AppendSmem* as = reinterpret_cast<AppendSmem*>(&sm.buf.ring[0][0][0]);   // the rings hold no copy here
  const int t = threadIdx.x;
  if constexpr (NTH >= 2 * APPEND_THREADS) {
    const int u = t / APPEND_THREADS;
    if (u < 2)
      append_work<GK>(c, layer, a.k_new, a.v_new, q, head, u, as[u], t % APPEND_THREADS,
                      [u] { bar_sync(1 + u, APPEND_THREADS); });
  } else {
    if (t < APPEND_THREADS) {
      for (int which = 0; which < 2; ++which)
        append_work<GK>(c, layer, a.k_new, a.v_new, q, head, which, as[0], t, [] { bar_sync(1, APPEND_THREADS); });
    }
  }
  __syncthreads();   // every write of the append is done (and seen by thread 0)
  if (t == 0) {
    uint32_t* f = c.dec_flag + (size_t)R.slot * c.Hkv + head;
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(a.epoch) : "memory");
  }
}

// Records in the workspace: INT2 record of (segment s, INT2 CTA c) at slot s + c
// (the INT2 CTAs meeting one segment are consecutive, so the slots are unique),
// then the BF16 record of segment s.
template <int G, int GK>
__global__ void __launch_bounds__(Tune<G, GK>::THREADS, 1)
    decode_kernel(DevCache c, int layer, DecodeArgs a, const uint16_t* __restrict__ q, float* __restrict__ recs,
                  float* __restrict__ out) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<G, GK>& sm = *reinterpret_cast<Smem<G, GK>*>(smem_raw);
  const int t = threadIdx.x, warp = t >> 5;
  // Roles: the last nbc blocks are the BF16 CTAs.  Blocks are placed on SMs in index
  // order as the preceding launch's CTAs leave them, and the SMs left last are those
  // that merged; the BF16 CTAs' work is short enough to start there late.
  const int hi0 = a.ncta - a.nbc;
  const int cta = (int)blockIdx.x >= hi0 ? (int)blockIdx.x - hi0 : (int)blockIdx.x + a.nbc;
  float* int2_recs = recs;
  float* bf16_recs = recs + ((size_t)a.n * c.Hkv + a.ncta) * G * PART;
  const uint32_t epoch = a.epoch;
  const int n2cta = a.ncta - a.nbc;   // INT2 CTAs
  const bool bm = a.n * c.Hkv <= a.nbc;   // one segment per BF16 CTA: the BF16 CTAs merge

  if ((t & 31) == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(&sm.bar[warp][st], 1);
    if (t == 0) {
      mbar_init(&sm.mbar_m, 1);
      mbar_init(&sm.mbar_r, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  uint32_t mphase = 0;        // phase of the merge staging barrier

  if (cta < a.nbc) {
    // ---- a BF16 CTA: the BF16 blocks of segments cta, cta + nbc, ... (none of
    // their rows is written by a fused append: the appended token comes from k / v)
    __syncthreads();
    if (epoch != 0 && warp == 0) {
      // the rotations the appends read (written once, at set-up): into L2 while waiting
      const int lane = t & 31;
      for (int s = cta; s < a.n * c.Hkv; s += a.nbc) {
        if (a.r[s / c.Hkv].hot_page < 0 || lane >= 16) continue;
        const size_t off = ((size_t)layer * c.Hkv + s % c.Hkv) * D * D;
        const float* m = lane < 4 ? c.rot_k : lane < 8 ? c.rot_v : lane < 12 ? c.rot_kt : c.rot_vt;
        prefetch_l2(m + off + (size_t)(lane & 3) * (D * D / 4), D * D);
      }
    }
    if (warp == 1) {
      // q (and k / v of a step) of this CTA's segments into L2: the preceding grid may
      // still write them, which L2 (the coherence point) then holds when they are read
      // after the wait
      const int lane = t & 31;
      for (int s = cta + (lane >> 2) * a.nbc; s < a.n * c.Hkv; s += 8 * a.nbc) {
        const size_t row = (size_t)a.r[s / c.Hkv].batch_row;
        if ((lane & 3) == 0) prefetch_l2(q + (row * c.Hq + (size_t)(s % c.Hkv) * G) * D, G * D * 2);
        if (epoch != 0 && (lane & 3) == 1) prefetch_l2(a.k_new + (row * c.Hkv + s % c.Hkv) * D, D * 2);
        if (epoch != 0 && (lane & 3) == 2) prefetch_l2(a.v_new + (row * c.Hkv + s % c.Hkv) * D, D * 2);
      }
    }
    grid_dep_wait();    // q, k / v and the cache may have been written by the preceding grid
    grid_dep_launch();  // the next launch may be scheduled (every CTA of this one is running); it waits for it
    if (epoch != 0) {
      // a decode step: the append of this CTA's (request, kv head) pairs first, so
      // that the hot pages are ready early for the CTAs that stream them
      for (int s = cta; s < a.n * c.Hkv; s += a.nbc) step_append<G, GK>(c, layer, a, s / c.Hkv, s % c.Hkv, sm);
    }
    for (int s = cta; s < a.n * c.Hkv; s += a.nbc) {
      const int ri = s / c.Hkv, head = s % c.Hkv;
      const DecodeReq& R = a.r[ri];
      if (warp == 0 && (t & 31) < 4) {   // R_V^T of the merge, should this CTA do it
        const float* rvt = c.rot_vt + ((size_t)layer * c.Hkv + head) * D * D;
        prefetch_l2(rvt + (size_t)(t & 31) * (D * D / 4), D * D);
      }
      bf16_segment<G, GK>(c, layer, a, ri, head, q, sm, bf16_recs);
      int c_lo = 0, n2 = 0;
      if (R.npages > 0 && n2cta > 0) {
        int c_hi;
        segment_ctas(a, R.cost_start + (int64_t)head * seg_units(R), seg_units(R), c_lo, c_hi);
        n2 = c_hi - c_lo + 1;
      }
      if (bm)
        wait_and_merge<G, GK>(c, layer, a, ri, head, c_lo, n2, int2_recs, bf16_recs, out, sm, mphase);
      else
        count_and_merge<G, GK>(c, layer, a, ri, head, c_lo, n2, int2_recs, bf16_recs, out, sm, mphase, false);
    }
    return;
  }

  // ---- an INT2 CTA: its range [u0, u1) of the INT2 pages, segment by segment
  const int icta = cta - a.nbc;
  const int64_t u0 = cta_begin(a, icta), u1 = cta_begin(a, icta + 1);
  if (t == 0) {
    int64_t prev;
    sm.seg[0] = plan_segment(a, c.Hkv, icta, u1 - 1, u0, u1, prev);
    sm.u_next = prev;
  }
  __syncthreads();
  uint32_t nc = 0;            // copies this warp has consumed
  bool timed_out = false;     // a wait of this warp ran out: no further copies
  const int hold = a.dbg.hold_copy;   // failure-detection hook: warp 0 of every INT2 CTA
  {
    const Seg S = sm.seg[0];
    RkRows<G, GK> rk;
    if (S.valid) load_rk<G, GK>(c, layer, S.head, rk);
    // q of the first segment into L2 (the preceding grid may still write it; L2 then
    // holds what it wrote when q is read after the wait)
    if (S.valid && t == 32)
      prefetch_l2(q + ((size_t)a.r[S.ri].batch_row * c.Hq + (size_t)S.head * G) * D, G * D * 2);
    // After a decode launch of this cache, the history pages below npages - 2 (and
    // their page-table entries) are not written by any grid that may still run:
    // their first copies go out before the wait, while that grid finishes
    if (S.valid && a.prefetch)
      int2_issue_first<G, GK>(c, layer, a.r[S.ri], S.head, S.p0, S.p1, sm, epoch, a.dbg.wait_limit, nc, hold,
                              timed_out, 1);
    grid_dep_wait();    // the cache and q may have been written by the preceding grid
    grid_dep_launch();  // the next launch may be scheduled (every CTA of this one is running); it waits for it
    if (S.valid) {
      QRows<G, GK> qv;
      load_q<G, GK>(c, layer, a.r[S.ri], S.head, q, qv);   // in flight with the page-id loads of the copies
      int2_issue_first<G, GK>(c, layer, a.r[S.ri], S.head, S.p0, S.p1, sm, epoch, a.dbg.wait_limit, nc, hold,
                              timed_out, a.prefetch ? 2 : 0);
      build_qfrag<G, GK>(c, qv, rk, sm);
    }
  }
  // segment e is in slot e & 1; its fields are read from shared memory where they
  // are needed, so that none stays in registers across the page loop
  for (int e = 0; sm.seg[e & 1].valid; ++e) {
    const int cur = e & 1, nxt = cur ^ 1;
    // planned by the last warp: warp w takes pages w, w + NW, ... of the segment, so
    // the last warp has the fewest (one page of slack, where warp 0 has the most)
    if (t == 32 * (Tune<G, GK>::NW - 1)) {
      int64_t prev;
      sm.seg[nxt] = plan_segment(a, c.Hkv, icta, sm.u_next, u0, u1, prev);
      sm.u_next = prev;
    }
    {
      const Seg& S = sm.seg[cur];
      int2_pages<G, GK>(c, layer, a.r[S.ri], S.head, S.p0, S.p1, sm.qf, sm, int2_recs + (size_t)S.slot * G * PART,
                        a.dbg.wait_limit, epoch, nc, timed_out, hold);
    }
    {
      const Seg& S = sm.seg[cur];
      count_and_merge<G, GK>(c, layer, a, S.ri, S.head, S.c_lo, S.c_hi - S.c_lo + 1, int2_recs, bf16_recs, out, sm,
                             mphase, bm);
    }
    // the next segment: first copies, q rotation
    if (sm.seg[nxt].valid) {
      const Seg& N = sm.seg[nxt];
      RkRows<G, GK> rk;
      QRows<G, GK> qv;
      load_rk<G, GK>(c, layer, N.head, rk);
      load_q<G, GK>(c, layer, a.r[N.ri], N.head, q, qv);
      int2_issue_first<G, GK>(c, layer, a.r[N.ri], N.head, N.p0, N.p1, sm, epoch, a.dbg.wait_limit, nc, hold,
                              timed_out);
      build_qfrag<G, GK>(c, qv, rk, sm);
    }
  }
}

template <int G, int GK>
cudaError_t launch_decode_t(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& p,
                            const uint16_t* q, float* out, void* workspace, const uint16_t* k_new,
                            const uint16_t* v_new, uint32_t epoch, bool prefetch, DecodeDebug dbg, cudaStream_t s) {
  static_assert(sizeof(Smem<G, GK>) <= 227 * 1024, "shared memory");
  using SM = Smem<G, GK>;
  static_assert(offsetof(SM, qf) % 16 == 0 && (QFrag<G>::WORDS * 4) % 16 == 0, "q operands: uint4 loads");
  static_assert(offsetof(SM, meta) % 16 == 0 && offsetof(SM, bar) % 8 == 0, "shared memory alignment");
  static unsigned attr_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(attr_done & (1u << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<G, GK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(Smem<G, GK>)));
    if (e != cudaSuccess) return e;
    if (dev < 32) attr_done |= 1u << dev;
  }
  DecodeArgs a;
  a.n = p.n;
  a.ncta = p.ncta;
  a.nbc = p.nbc;
  a.prefetch = prefetch ? 1 : 0;
  a.epoch = k_new != nullptr ? epoch : 0u;
  a.total_cost = p.total_cost;
  a.dbg = dbg;
  {
    const int n2 = p.ncta - p.nbc;
    if (n2 > DECODE_MAX_INT2 || p.total_cost > INT32_MAX) return cudaErrorInvalidValue;
    for (int i = 0; i <= n2; ++i) a.cstart[i] = static_cast<int32_t>((int64_t)i * p.total_cost / (n2 > 0 ? n2 : 1));
  }
  a.k_new = a.epoch != 0 ? k_new : nullptr;
  a.v_new = a.epoch != 0 ? v_new : nullptr;
  for (int i = 0; i < p.n; ++i) a.r[i] = reqs[i];
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.ncta));
  cfg.blockDim = dim3(Tune<G, GK>::THREADS);
  cfg.dynamicSmemBytes = sizeof(Smem<G, GK>);
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<G, GK>, c, layer, a, q, static_cast<float*>(workspace), out);
}

template <int GK>
cudaError_t launch_decode_g(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& p,
                            const uint16_t* q, float* out, void* ws, const uint16_t* kn, const uint16_t* vn,
                            uint32_t ep, bool pf, DecodeDebug dbg, cudaStream_t s) {
  switch (c.G) {
    case 1: return launch_decode_t<1, GK>(c, layer, reqs, p, q, out, ws, kn, vn, ep, pf, dbg, s);
    case 2: return launch_decode_t<2, GK>(c, layer, reqs, p, q, out, ws, kn, vn, ep, pf, dbg, s);
    case 4: return launch_decode_t<4, GK>(c, layer, reqs, p, q, out, ws, kn, vn, ep, pf, dbg, s);
    case 8: return launch_decode_t<8, GK>(c, layer, reqs, p, q, out, ws, kn, vn, ep, pf, dbg, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& p,
                          const uint16_t* q, float* out, void* workspace, const uint16_t* k_new,
                          const uint16_t* v_new, uint32_t epoch, bool prefetch, DecodeDebug dbg, cudaStream_t s) {
  if (p.n < 1 || p.n > DECODE_PER_LAUNCH || p.nbc < 1 || p.ncta < p.nbc || p.total_cost < p.ncta - p.nbc)
    return cudaErrorInvalidValue;
  if ((k_new != nullptr) != (v_new != nullptr) || (k_new != nullptr && epoch == 0)) return cudaErrorInvalidValue;
  return c.gk == 64
             ? launch_decode_g<64>(c, layer, reqs, p, q, out, workspace, k_new, v_new, epoch, prefetch, dbg, s)
             : launch_decode_g<128>(c, layer, reqs, p, q, out, workspace, k_new, v_new, epoch, prefetch, dbg, s);
}

}  // namespace oscar
