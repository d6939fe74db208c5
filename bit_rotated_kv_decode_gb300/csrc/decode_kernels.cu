// Three-segment decode attention on the fifth-generation tensor cores.
//
// "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计": at decode time the
// INT2 history is unpacked, dequantised with its scale / zero point and
// accumulated in floating point; the BF16 sink and recent window are handled
// separately; the partials are merged with an online softmax (max / sum).
// "Together AI Open-Sources OSCAR" (MarkTechPost), section "The Serving
// System": the value path is inverse-rotated.
//
// Two launches per layer (and per 64 requests), chained with programmatic
// dependent launch:
//   1. decode   one persistent CTA per SM.  The work -- every INT2 history page
//               and every BF16 half-page of every (request, kv head) segment --
//               is cut into equal-cost contiguous ranges, one per CTA.  A CTA
//               rotates q itself (q_rot = q R_K, in its prologue, while the first
//               page copies are in flight), then its warpgroups stream page pairs
//               (128 tokens) through per-warpgroup TMA rings and write one partial
//               (o, m, l) per segment it touched, INT2 part in the rotated basis;
//   2. merge    one CTA per segment: online-softmax merge of the partials,
//               R_V^T applied to the INT2 part (staged in shared memory while the
//               decode grid still runs), out = (O_bf16 + O_hist R_V^T) / L.
//
// The INT2 contractions of a page pair run as tcgen05.mma (kind::f16, M = 128,
// fp32 accumulators in tensor memory, issued by one thread per warpgroup):
//   logits   D_K[token][col] = sum_k A_K[token][k] Bq[k][col]
//            A_K: the pair's 128 tokens x 128 K codes, in tensor memory;
//            Bq:  q_rot split into fp16 hi + lo columns, in shared memory;
//   values   D_V[chan][col] += sum_k A_V[chan][k] Bw[k][col]
//            A_V: 128 channels x the pair's 128 V codes, in tensor memory;
//            Bw:  the softmax weights p s_v (fp16 hi + lo), in shared memory.
// A 2-bit code masked out of a packed word, with every other bit zero, is the
// fp16 subnormal code 2^(2e - 24) (e = 0..4 by its bit position): one LOP3 gives
// two codes, and the factor 2^(8 - 2e) of the row goes into the B operand, so
// every product is code * b 2^-16 exactly in fp32.  Each thread unpacks one row
// of A_K (its token: K codes are stored token-major) and one row of A_V (its
// channel: V codes are stored channel-major) and stores it with tcgen05.st.
// For a token j with K codes c_j and fp16 (s_j, z_j) per quantisation group:
//   logit_j = scale (s_j (q_rot . c_j) + z_j sum(q_rot))   (per group),
//   value_j = s_j c_j + z_j                                 (p s_j c_j, plus sum p z_j).
// Every wait is bounded and reports ERR_TIMEOUT instead of hanging.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int PART = PARTIAL_FLOATS;
constexpr int WGT = 128;           // threads per warpgroup
constexpr int STAGES = 4;          // page-pair stages of a warpgroup's ring
constexpr int SEG_PRE = 2;         // segments whose q operands the prologue builds
constexpr int SEGMAX = 16;         // segments one CTA may touch
constexpr float LAZY_MAX = 8.0f;   // softmax reference max kept within 2^8 of the true one
constexpr uint32_t SUSPEND_NS = 10000;
constexpr int MERGE_THREADS = 256;

template <int G, int GK>
struct Cfg {
  static constexpr int NG = D / GK;                     // quantisation groups per token-head
  static constexpr int NC = 2 * G * NG;                 // used columns: (group, head, hi | lo)
  static constexpr int N = NC <= 16 ? 16 : 32;          // MMA N
  static constexpr int NWG = N == 16 ? 3 : 2;           // warpgroups per CTA (tensor-memory budget)
  static constexpr int THREADS = NWG * WGT;
  static constexpr int REC = record_for(GK);
  static constexpr int STAGE = 2 * REC;
  static constexpr int BT = D * N * 2;                  // bytes of a 128-row B tile
  static constexpr int TW = 128 + 2 * N;                // tensor-memory columns per warpgroup
  static constexpr int KMETA = k_meta_off_for(GK), VMETA = v_meta_off_for(GK), MB = meta_bytes_for(GK);
  static_assert(NWG * TW <= 512, "tensor memory");
};

__host__ __device__ constexpr int code_exp(int m) { return m <= 4 ? m : m - 5; }
__device__ __forceinline__ int col_of(int g, int h, int part, int G) { return 2 * G * g + 2 * h + part; }

struct Seg {
  int ri, head;    // request index in the launch, kv head
  int p0, p1;      // INT2 pages [p0, p1) of this CTA
  int bf16;        // the segment's BF16 block belongs to this CTA
  int slot;        // INT2 partial record: segment + CTA
};

struct DecodeArgs {
  int n, ncta, front_writes;
  int64_t total_cost;
  DecodeDebug dbg;
  DecodeReq r[DECODE_PER_LAUNCH];
};

template <int G, int GK>
struct Smem {
  using C = Cfg<G, GK>;
  __align__(128) uint8_t ring[C::NWG][STAGES][C::STAGE];
  __align__(128) uint8_t bw[C::NWG][C::BT];       // value-side B tiles (BF16 phase: q and logits)
  __align__(128) uint8_t bq[SEG_PRE][C::BT];      // logit-side B tiles of the first segments
  union {
    struct {                                      // prologue: q and the row-part sums of q R_K
      float q[G][D];
      float part[C::NWG][G][D];
      float amax[G];
    } pro;
    struct {                                      // end of a segment: one partial per warpgroup
      float o[C::NWG][G][D];
      float ml[C::NWG][G][2];
    } fl;
  } u;
  float qc[SEG_PRE][G][1 + C::NG];                // per segment and head: ks, kz[group]
  int ew[SEG_PRE];                                // value prescale exponent of the segment's head
  float wmax[C::NWG][4][G];
  float red[C::NWG][4][G * (1 + C::NG)];
  int flag[C::NWG][2];
  __align__(8) uint64_t full[C::NWG][STAGES];
  __align__(8) uint64_t mk[C::NWG], mv[C::NWG];
  uint32_t tmem;
  int abort;
  int nseg;
  Seg seg[SEGMAX];
};

// ---- PTX helpers ---------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
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
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
template <int NR>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&f)[NR]);
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&f)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&f)[16]) {
  float a[8], b[8];
  tmem_ld<8>(taddr, a);
  tmem_ld<8>(taddr + 8, b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[i] = a[i];
    f[8 + i] = b[i];
  }
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&f)[32]) {
  float a[16], b[16];
  tmem_ld<16>(taddr, a);
  tmem_ld<16>(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    f[i] = a[i];
    f[16 + i] = b[i];
  }
}
template <int NR>
__device__ __forceinline__ void tmem_st_f(uint32_t taddr, const float (&f)[NR]) {
#pragma unroll
  for (int c0 = 0; c0 < NR; c0 += 8) {
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(f[c0 + i]);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr + c0),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
  }
}

// Shared-memory matrix descriptor of a B tile: 16-bit elements, N-major without
// swizzle, core matrices of 8 k-rows x 16 bytes; LBO = 128 (next 8 k-rows),
// SBO = 2048 (next 8 columns).
__device__ __forceinline__ uint64_t b_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(2048 >> 4) << 32) |
         ((uint64_t)1 << 46);
}
// Instruction descriptor: kind::f16, fp16 A and B, fp32 D, A K-major, B N-major, M = 128.
template <int N>
__device__ __forceinline__ constexpr uint32_t idesc_f16() {
  return (1u << 4) | (1u << 16) | ((uint32_t)(N >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float warp_max(float x) {
  float y;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ uint32_t h2_bits(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

// The 16 codes of a packed word as eight fp16x2 subnormal pairs: register m holds
// the codes at bit position m of the low and the high half, code 2^(2 e(m) - 24).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t* r) {
  const uint32_t ws = w >> 10;
  r[0] = w & 0x00030003u;
  r[1] = w & 0x000C000Cu;
  r[2] = w & 0x00300030u;
  r[3] = w & 0x00C000C0u;
  r[4] = w & 0x03000300u;
  r[5] = ws & 0x00030003u;
  r[6] = ws & 0x000C000Cu;
  r[7] = ws & 0x00300030u;
}
// Eight packed words -> 64 tensor-memory columns of one row (column 8 w + m).
__device__ __forceinline__ void store_row(uint32_t taddr, const uint32_t (&w)[8]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t r[16];
    unpack_word(w[2 * q], r);
    unpack_word(w[2 * q + 1], r + 8);
    tmem_st16(taddr + 16 * q, r);
  }
}

// ---- the plan ------------------------------------------------------------------------
__device__ __forceinline__ int64_t cta_begin(int c, int ncta, int64_t total) { return (int64_t)c * total / ncta; }

// Segment containing cost unit u: request index, kv head, its first unit.
__device__ __forceinline__ void segment_of(const DecodeArgs& a, int Hkv, int64_t u, int& ri, int& h, int64_t& s0) {
  ri = 0;
  while (ri + 1 < a.n && a.r[ri + 1].cost_start <= u) ++ri;
  const int64_t per = a.r[ri].npages + a.r[ri].bf16_cost;
  h = static_cast<int>((u - a.r[ri].cost_start) / per);
  if (h >= Hkv) h = Hkv - 1;
  s0 = a.r[ri].cost_start + (int64_t)h * per;
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

// ---- q operands of a segment --------------------------------------------------------
// q_rot = q R_K for the G query heads of (request, kv head), then the logit-side
// B tile: row k (channel chi(k) = 16 (k >> 4) + 8 (k & 1) + ((k >> 1) & 7), the
// channel whose codes A_K column k >> 1 holds in half k & 1) carries, in column
// (group, head, part), part of fp16 hi / lo of q_rot[head][chi] 2^eq(head) 2^(8 - 2e)
// when chi lies in that group, else 0.  2^eq(h) puts max |q_rot[h]| in (2^6, 2^7],
// so every entry is below 2^15.  Every thread of the CTA takes part.
template <int G, int GK>
__device__ void build_q_operands(const DevCache& c, int layer, const DecodeReq& R, int head,
                                 const uint16_t* __restrict__ q, Smem<G, GK>& sm, int slot_b) {
  using C = Cfg<G, GK>;
  constexpr int NTH = C::THREADS, NP = C::NWG;
  constexpr int RP = (D + NP - 1) / NP;   // rows per part
  const int t = threadIdx.x;
  const uint16_t* qrow = q + ((size_t)R.batch_row * c.Hq + (size_t)head * G) * D;
  for (int i = t; i < G * D; i += NTH) sm.u.pro.q[i / D][i % D] = __uint_as_float(static_cast<uint32_t>(qrow[i]) << 16);
  const float* __restrict__ RK = c.rot_k + ((size_t)layer * c.Hkv + head) * D * D;
  const int ch = t % D, part = t / D;
  const int r0 = part * RP, r1 = min(D, r0 + RP);
  float rk[RP];
#pragma unroll
  for (int i = 0; i < RP; ++i) rk[i] = (r0 + i < r1) ? __ldg(RK + (size_t)(r0 + i) * D + ch) : 0.0f;
  __syncthreads();
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.0f;
#pragma unroll
  for (int i = 0; i < RP; ++i) {
    if (r0 + i < r1) {
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = fmaf(sm.u.pro.q[h][r0 + i], rk[i], acc[h]);
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) sm.u.pro.part[part][h][ch] = acc[h];
  __syncthreads();
  // q_rot into part[0]; per-head max |q_rot| (warp-wide, then per head by lane 0)
  if (t < D) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = sm.u.pro.part[0][h][t];
#pragma unroll
      for (int p = 1; p < NP; ++p) v += sm.u.pro.part[p][h][t];
      sm.u.pro.part[0][h][t] = v;
    }
  }
  if (t < G) sm.u.pro.amax[t] = 0.0f;
  __syncthreads();
  if (t < D) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float m = warp_max(fabsf(sm.u.pro.part[0][h][t]));
      if ((t & 31) == 0) atomicMax(reinterpret_cast<int*>(&sm.u.pro.amax[h]), __float_as_int(m));
    }
  }
  __syncthreads();
  // B tile rows (threads 0..127), logit constants (warp per head among the rest)
  if (t < D) {
    const int k = t;
    const int m = (k >> 1) & 7, chi = 16 * (k >> 4) + 8 * (k & 1) + m;
    const int grp = chi / GK;
    uint32_t row[C::N / 2];
#pragma unroll
    for (int i = 0; i < C::N / 2; ++i) row[i] = 0u;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float am = sm.u.pro.amax[h];
      int eq = 0;
      if (am > 0.0f) {
        const uint32_t b = __float_as_uint(am);
        const int ceil_log2 = static_cast<int>((b >> 23) & 0xffu) - 127 + ((b & 0x7fffffu) != 0u ? 1 : 0);
        eq = max(-100, min(100, 7 - ceil_log2));
      }
      const float v = sm.u.pro.part[0][h][chi] * ldexpf(1.0f, eq + 8 - 2 * code_exp(m));
      const __half hi = __float2half_rn(v);
      const __half lo = __float2half_rn(v - __half2float(hi));
      const int cc = col_of(grp, h, 0, G);   // even: hi and lo share one word
      row[cc >> 1] = h2_bits(hi, lo);
    }
    uint8_t* base = sm.bq[slot_b] + (k >> 3) * 128 + (k & 7) * 16;
#pragma unroll
    for (int ng = 0; ng < C::N / 8; ++ng)
      *reinterpret_cast<uint4*>(base + 2048 * ng) =
          make_uint4(row[4 * ng], row[4 * ng + 1], row[4 * ng + 2], row[4 * ng + 3]);
  }
  // logit constants: ks = scale log2(e) 2^16 / 2^eq, kz[group] = scale log2(e) sum q_rot
  const int w = t >> 5, lane = t & 31;
  for (int h = w - 4; h >= 0 && h < G; h += C::THREADS / 32 - 4) {
    const float am = sm.u.pro.amax[h];
    int eq = 0;
    if (am > 0.0f) {
      const uint32_t b = __float_as_uint(am);
      const int ceil_log2 = static_cast<int>((b >> 23) & 0xffu) - 127 + ((b & 0x7fffffu) != 0u ? 1 : 0);
      eq = max(-100, min(100, 7 - ceil_log2));
    }
    const float s2 = c.scale * LOG2E;
#pragma unroll
    for (int g = 0; g < C::NG; ++g) {
      float sum = 0.0f;
      for (int i = lane; i < GK; i += 32) sum += sm.u.pro.part[0][h][GK * g + i];
      sum = warp_sum(sum);
      if (lane == 0) sm.qc[slot_b][h][1 + g] = s2 * sum;
    }
    if (lane == 0) sm.qc[slot_b][h][0] = s2 * ldexpf(1.0f, 16 - eq);
  }
  if (t == 0) {
    // weights p s_v 2^ew with p <= 2^8 and s_v <= fp16(2 tau_V / 3): p s_v 2^ew 2^8 <= 2^15.9
    const float smax = c.tau_v[(size_t)layer * c.Hkv + head] * (2.0f / 3.0f) * 1.002f;
    int ew = smax > 0.0f ? static_cast<int>(floorf(log2f(0.93f / smax))) : 0;
    sm.ew[slot_b] = max(-60, min(60, ew));
  }
  fence_async_smem();
  __syncthreads();
}

// ---- the decode kernel --------------------------------------------------------------
template <int G, int GK>
__global__ void __launch_bounds__(Cfg<G, GK>::THREADS, 1)
    decode_kernel(DevCache c, int layer, DecodeArgs a, const uint16_t* __restrict__ q, float* __restrict__ recs) {
  using C = Cfg<G, GK>;
  constexpr int NG = C::NG, NC = C::NC, N = C::N, NWG = C::NWG, REC = C::REC;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem<G, GK>& sm = *reinterpret_cast<Smem<G, GK>*>(smem_raw);
  const int t = threadIdx.x, wg = t / WGT, wt = t % WGT, wiw = wt >> 5, lane = t & 31;
  const int cta = blockIdx.x;
  const uint32_t limit = a.dbg.wait_limit;
  float* int2_recs = recs;
  float* bf16_recs = recs + ((size_t)a.n * c.Hkv + a.ncta) * G * PART;

  // ---- prologue: plan, tensor memory, barriers
  if (!a.front_writes) grid_dep_wait();   // the cache may have been written by the preceding grid
  grid_dep_launch();
  if (t == 0) {
    const int64_t u0 = cta_begin(cta, a.ncta, a.total_cost), u1 = cta_begin(cta + 1, a.ncta, a.total_cost);
    int n = 0;
    for (int64_t u = u0; u < u1;) {
      int ri, h;
      int64_t s0;
      segment_of(a, c.Hkv, u, ri, h, s0);
      const DecodeReq& R = a.r[ri];
      const int64_t np = R.npages, end = s0 + np + R.bf16_cost;
      if (n == SEGMAX) {
        atomicOr(c.err, ERR_PLAN);
        break;
      }
      Seg& e = sm.seg[n++];
      e.ri = ri;
      e.head = h;
      const int64_t lo = u0 - s0 > 0 ? u0 - s0 : 0, hi = u1 - s0 < np ? u1 - s0 : np;
      e.p0 = static_cast<int>(lo < np ? lo : np);
      e.p1 = static_cast<int>(hi > e.p0 ? hi : e.p0);
      e.bf16 = (R.bf16_cost > 0 && s0 + np >= u0 && s0 + np < u1) ? 1 : 0;
      e.slot = ri * c.Hkv + h + cta;
      u = end;
    }
    sm.nseg = n;
    sm.abort = 0;
    for (int w = 0; w < NWG; ++w) {
      for (int st = 0; st < STAGES; ++st) mbar_init(&sm.full[w][st], 1);
      mbar_init(&sm.mk[w], 1);
      mbar_init(&sm.mv[w], 1);
      sm.flag[w][0] = sm.flag[w][1] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (t < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm.tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nseg = sm.nseg;
  const uint32_t tw = sm.tmem + (uint32_t)(wg * C::TW);
  const uint32_t lane_off = (uint32_t)(32 * wiw) << 16;
  const uint32_t tAK = tw, tAV = tw + 64, tDK = tw + 128, tDV = tw + 128 + N;

  // ---- page-pair iteration of this warpgroup: pairs j = wg, wg + NWG, ... of each segment
  auto npairs_of = [&](int e) { return (sm.seg[e].p1 - sm.seg[e].p0 + 1) >> 1; };
  auto advance = [&](int& e, int& j) {
    while (e < nseg && j >= npairs_of(e)) {
      ++e;
      j = wg;
    }
  };
  // the copies of one pair into stage st; page ids are loaded by the caller
  auto pair_pages = [&](int e, int j, int& pa, int& pb) {
    const Seg& s = sm.seg[e];
    pa = s.p0 + 2 * j;
    pb = pa + 1 < s.p1 ? pa + 1 : -1;
  };
  // a page id as stored (checked at copy time, so the load's latency is hidden)
  auto page_id_raw = [&](int e, int pi) -> int {
    return __ldcg(c.hist_pt + (size_t)a.r[sm.seg[e].ri].slot * c.max_pages + pi);
  };
  auto checked = [&](int id) -> int {
    if (id < 0 || id >= c.n_int2_pages) {
      atomicOr(c.err, ERR_INT2_PAGE);
      id = 0;
    }
    return id;
  };
  auto page_id = [&](int e, int pi) -> int { return checked(page_id_raw(e, pi)); };
  auto is_hot = [&](int e, int pi) { return a.front_writes && pi >= 0 && pi == a.r[sm.seg[e].ri].hot_page; };
  auto issue = [&](int st, int e, int pa, int pb, int ida, int idb) {
    const Seg& s = sm.seg[e];
    const uint8_t* base = c.int2 + layer * c.int2_layer_stride + (size_t)s.head * REC;
    const size_t pstride = (size_t)c.Hkv * REC;
    mbar_expect_tx(&sm.full[wg][st], pb >= 0 ? 2 * REC : REC);
    tma_load_1d(sm.ring[wg][st], base + (size_t)ida * pstride, REC, &sm.full[wg][st]);
    if (pb >= 0) tma_load_1d(sm.ring[wg][st] + REC, base + (size_t)idb * pstride, REC, &sm.full[wg][st]);
  };
  // prefetch cursor (thread wt == 0): the pair to copy next, its page ids loaded one refill ahead
  int pf_e = 0, pf_j = wg, pf_seq = 0;
  int nx_pa = -1, nx_pb = -1, nx_ida = 0, nx_idb = 0;
  bool nx_valid = false, nx_hot = false;
  uint32_t issued_mask = 0;   // stages with a copy in flight (for the bounded drain on abort)
  auto load_next_ids = [&]() {
    advance(pf_e, pf_j);
    nx_valid = pf_e < nseg;
    if (!nx_valid) return;
    pair_pages(pf_e, pf_j, nx_pa, nx_pb);
    // the hot page's id is read at copy time, after the preceding grid has completed
    nx_hot = is_hot(pf_e, nx_pa) || is_hot(pf_e, nx_pb);
    nx_ida = is_hot(pf_e, nx_pa) ? 0 : page_id_raw(pf_e, nx_pa);
    nx_idb = (nx_pb < 0 || is_hot(pf_e, nx_pb)) ? 0 : page_id_raw(pf_e, nx_pb);
  };
  auto issue_next = [&]() {
    if (!nx_valid) return;
    const int st = pf_seq % STAGES;
    if (nx_hot) {
      grid_dep_wait();
      if (is_hot(pf_e, nx_pa)) nx_ida = page_id_raw(pf_e, nx_pa);
      if (is_hot(pf_e, nx_pb)) nx_idb = page_id_raw(pf_e, nx_pb);
    }
    nx_ida = checked(nx_ida);
    if (nx_pb >= 0) nx_idb = checked(nx_idb);
    const bool held = a.dbg.hold_pair >= 0 && cta == 0 && wg == 0 && pf_seq == a.dbg.hold_pair;
    if (!held) {
      issue(st, pf_e, nx_pa, nx_pb, nx_ida, nx_idb);
      issued_mask |= 1u << st;
    }
    ++pf_seq;
    pf_j += NWG;
    load_next_ids();
  };
  if (wt == 0) {
    // the first STAGES pairs: all page ids in flight at once, then the copies
    int pe[STAGES], pj[STAGES], pa[STAGES], pb[STAGES], ia[STAGES], ib[STAGES];
    int cnt = 0;
    for (; cnt < STAGES; ++cnt) {
      advance(pf_e, pf_j);
      if (pf_e >= nseg) break;
      pe[cnt] = pf_e;
      pj[cnt] = pf_j;
      pair_pages(pf_e, pf_j, pa[cnt], pb[cnt]);
      pf_j += NWG;
    }
    for (int i = 0; i < cnt; ++i) {
      ia[i] = is_hot(pe[i], pa[i]) ? -1 : page_id(pe[i], pa[i]);
      ib[i] = pb[i] < 0 ? 0 : (is_hot(pe[i], pb[i]) ? -1 : page_id(pe[i], pb[i]));
    }
    for (int i = 0; i < cnt; ++i) {
      nx_pa = pa[i];
      nx_pb = pb[i];
      nx_ida = ia[i];
      nx_idb = ib[i];
      nx_valid = true;
      const int save_e = pf_e, save_j = pf_j;
      pf_e = pe[i];
      pf_j = pj[i];
      const int st = pf_seq % STAGES;
      if (nx_ida < 0 || (nx_pb >= 0 && nx_idb < 0)) {
        grid_dep_wait();
        if (nx_ida < 0) nx_ida = page_id(pf_e, nx_pa);
        if (nx_pb >= 0 && nx_idb < 0) nx_idb = page_id(pf_e, nx_pb);
      }
      const bool held = a.dbg.hold_pair >= 0 && cta == 0 && wg == 0 && pf_seq == a.dbg.hold_pair;
      if (!held) {
        issue(st, pf_e, nx_pa, nx_pb, nx_ida, nx_idb);
        issued_mask |= 1u << st;
      }
      ++pf_seq;
      pf_e = save_e;
      pf_j = save_j;
    }
    load_next_ids();
  }

  // ---- q operands of the first segments (every thread)
  for (int e = 0; e < min(nseg, SEG_PRE); ++e)
    build_q_operands<G, GK>(c, layer, a.r[sm.seg[e].ri], sm.seg[e].head, q, sm, e);

  // ---- the INT2 pairs, segment by segment
  int seq = 0;           // pairs this warpgroup consumed
  int mv_count = 0;      // value-side commits of this warpgroup
  for (int e = 0; e < nseg; ++e) {
    const Seg S = sm.seg[e];
    const DecodeReq& R = a.r[S.ri];
    int bslot = e;
    if (e >= SEG_PRE) {
      // later segments rebuild the operands in slot (e & 1): every warpgroup is done
      // with the segment that used that slot (the end-of-segment barriers)
      bslot = e & 1;
      build_q_operands<G, GK>(c, layer, R, S.head, q, sm, bslot);
    }
    float ks[G], kz[G][NG];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      ks[h] = sm.qc[bslot][h][0];
#pragma unroll
      for (int g = 0; g < NG; ++g) kz[h][g] = sm.qc[bslot][h][1 + g];
    }
    const float wscale = ldexpf(1.0f, sm.ew[bslot]);
    const uint32_t bq_addr = smem_u32(sm.bq[bslot]);
    const uint32_t bw_addr = smem_u32(sm.bw[wg]);
    const int nhist = R.hist_end - SINK;
    float m_ref[G], l_acc[G], u_acc[G][NG];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_ref[h] = -INFINITY;
      l_acc[h] = 0.0f;
#pragma unroll
      for (int g = 0; g < NG; ++g) u_acc[h][g] = 0.0f;
    }
    bool has_acc = false;
    const int npairs = (S.p1 - S.p0 + 1) >> 1;
    for (int j = wg; j < npairs; j += NWG, ++seq) {
      const int st = seq % STAGES;
      const uint8_t* stage = sm.ring[wg][st];
      const int pa = S.p0 + 2 * j;
      const int va = min(PAGE, nhist - PAGE * pa);
      const int vb = pa + 1 < S.p1 ? min(PAGE, nhist - PAGE * (pa + 1)) : 0;
      if (!sm.abort && !mbar_wait(&sm.full[wg][st], (seq / STAGES) & 1, limit)) {
        if (wt == 0) {
          sm.abort = 1;
          atomicOr(c.err, ERR_TIMEOUT);
        }
      }
      bar_sync(1 + wg, WGT);
      const bool ab = sm.abort != 0;
      if (wt == 0) {
        if (seq >= 1) sm.flag[wg][(seq + 1) & 1] = 0;   // the flag of the next pair
        issued_mask &= ~(1u << st);
      }
      // -- K side: thread = token wt of the pair
      const int tp = wt >> 6, tr = wt & 63;
      const bool valid = tr < (tp ? vb : va);
      if (!ab) {
        const uint4* kc = reinterpret_cast<const uint4*>(stage + tp * REC + K_CODES_OFF + CODE_BYTES * tr);
        const uint4 c0 = kc[0], c1 = kc[1];
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        store_row(tAK + lane_off, w);
        tc_wait_st();
      }
      tc_fence_before();
      bar_sync(1 + wg, WGT);
      if (wt == 0 && !ab) {
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s) umma(tDK, tAK + 8 * s, b_desc(bq_addr + 256 * s), idesc_f16<N>(), s > 0 ? 1u : 0u);
        umma_commit(&sm.mk[wg]);
      }
      // -- V side: thread = channel wt; the previous value MMA must have read A_V
      if (!ab) {
        if (mv_count > 0 && !mbar_wait(&sm.mv[wg], (mv_count - 1) & 1, limit) && wt == 0) {
          sm.abort = 1;
          atomicOr(c.err, ERR_TIMEOUT);
        }
        tc_fence_after();
        const uint4 v0 = *reinterpret_cast<const uint4*>(stage + V_CODES_OFF + 16 * wt);
        const uint4 v1 = *reinterpret_cast<const uint4*>(stage + REC + V_CODES_OFF + 16 * wt);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        store_row(tAV + lane_off, w);
        tc_wait_st();
      }
      // -- token meta: {s, z} of K and V per group, value terms zeroed past the end
      float sk[NG], zk[NG], sv[NG], zv[NG];
      {
        const uint8_t* rb = stage + tp * REC;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const __half2 km = *reinterpret_cast<const __half2*>(rb + C::KMETA + C::MB * tr + 4 * g);
          const __half2 vm = *reinterpret_cast<const __half2*>(rb + C::VMETA + C::MB * tr + 4 * g);
          sk[g] = __low2float(km);
          zk[g] = __high2float(km);
          sv[g] = valid ? __low2float(vm) * wscale : 0.0f;
          zv[g] = valid ? __high2float(vm) : 0.0f;
        }
      }
      // -- logits (log2 domain)
      float lg[G];
      if (!ab) {
        if (!mbar_wait(&sm.mk[wg], seq & 1, limit) && wt == 0) {
          sm.abort = 1;
          atomicOr(c.err, ERR_TIMEOUT);
        }
        tc_fence_after();
        float d[NC <= 8 ? 8 : (NC <= 16 ? 16 : 32)];
        tmem_ld(tDK + lane_off, d);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float v = 0.0f;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const float acc = d[col_of(g, h, 0, G)] + d[col_of(g, h, 1, G)];
            v = fmaf(ks[h] * sk[g], acc, fmaf(kz[h][g], zk[g], v));
          }
          lg[h] = valid ? v : -INFINITY;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) lg[h] = -INFINITY;
      }
      // -- softmax: the reference max m_ref moves only when a pair exceeds it by more
      // than LAZY_MAX; the warps of the warpgroup agree on it through shared memory
      bool exceed = false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float wm = warp_max(lg[h]);
        exceed |= wm > m_ref[h] + LAZY_MAX;
        if (lane == 0) sm.wmax[wg][wiw][h] = wm;
      }
      if (exceed && lane == 0) sm.flag[wg][seq & 1] = 1;
      // row of the value-side B tile fed by this token, and its position factor
      const int kr = 2 * (8 * (4 * tp + (tr >> 4)) + (tr & 7)) + ((tr >> 3) & 1);
      const float fpos = ldexpf(1.0f, 8 - 2 * code_exp(tr & 7));
      uint8_t* brow = sm.bw[wg] + (kr >> 3) * 128 + (kr & 7) * 16;
      float p[G];
      auto write_weights = [&]() {
        uint32_t row[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) row[i] = 0u;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const float v = p[h] * sv[g] * fpos;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            row[col_of(g, h, 0, G) >> 1] = h2_bits(hi, lo);
          }
#pragma unroll
        for (int ng = 0; ng < N / 8; ++ng)
          *reinterpret_cast<uint4*>(brow + 2048 * ng) =
              make_uint4(row[4 * ng], row[4 * ng + 1], row[4 * ng + 2], row[4 * ng + 3]);
      };
#pragma unroll
      for (int h = 0; h < G; ++h) p[h] = lg[h] == -INFINITY ? 0.0f : ex2(lg[h] - m_ref[h]);
      write_weights();
      fence_async_smem();
      tc_fence_before();
      bar_sync(1 + wg, WGT);
      if (sm.flag[wg][seq & 1]) {
        // a new reference max: recompute this pair's weights, rescale the sums and
        // the value accumulator (once the previous value MMA has completed)
        float corr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float mn = m_ref[h];
#pragma unroll
          for (int w = 0; w < 4; ++w) mn = fmaxf(mn, sm.wmax[wg][w][h]);
          corr[h] = (m_ref[h] == -INFINITY || mn == -INFINITY) ? (mn == -INFINITY ? 1.0f : 0.0f) : ex2(m_ref[h] - mn);
          m_ref[h] = mn;
          l_acc[h] *= corr[h];
#pragma unroll
          for (int g = 0; g < NG; ++g) u_acc[h][g] *= corr[h];
          p[h] = lg[h] == -INFINITY ? 0.0f : ex2(lg[h] - m_ref[h]);
        }
        write_weights();
        if (has_acc && !ab) {
          tc_fence_after();
          float d[NC <= 8 ? 8 : (NC <= 16 ? 16 : 32)];
          tmem_ld(tDV + lane_off, d);
          tc_wait_ld();
#pragma unroll
          for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int h = 0; h < G; ++h) {
              d[col_of(g, h, 0, G)] *= corr[h];
              d[col_of(g, h, 1, G)] *= corr[h];
            }
          tmem_st_f(tDV + lane_off, d);
          tc_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        bar_sync(1 + wg, WGT);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        l_acc[h] += p[h];
#pragma unroll
        for (int g = 0; g < NG; ++g) u_acc[h][g] = fmaf(p[h], zv[g], u_acc[h][g]);
      }
      if (wt == 0) {
        if (!ab) {
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < 8; ++s)
            umma(tDV, tAV + 8 * s, b_desc(bw_addr + 256 * s), idesc_f16<N>(), (has_acc || s > 0) ? 1u : 0u);
          umma_commit(&sm.mv[wg]);
        }
        // every thread has read this stage: refill it with the pair STAGES ahead
        if (!sm.abort) issue_next();
      }
      if (!ab) ++mv_count;
      has_acc = true;
    }
    // ---- end of the segment: this warpgroup's partial, then the CTA's record
    {
      float l_tot[G], u_tot[G][NG];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float lw = warp_sum(l_acc[h]);
        if (lane == 0) sm.red[wg][wiw][h * (1 + NG)] = lw;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float uw = warp_sum(u_acc[h][g]);
          if (lane == 0) sm.red[wg][wiw][h * (1 + NG) + 1 + g] = uw;
        }
      }
      bar_sync(1 + wg, WGT);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        l_tot[h] = 0.0f;
#pragma unroll
        for (int g = 0; g < NG; ++g) u_tot[h][g] = 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          l_tot[h] += sm.red[wg][w][h * (1 + NG)];
#pragma unroll
          for (int g = 0; g < NG; ++g) u_tot[h][g] += sm.red[wg][w][h * (1 + NG) + 1 + g];
        }
      }
      const bool acc_ok = has_acc && mv_count > 0 && !sm.abort;
      float d[NC <= 8 ? 8 : (NC <= 16 ? 16 : 32)];
      if (acc_ok) {
        if (!mbar_wait(&sm.mv[wg], (mv_count - 1) & 1, limit) && wt == 0) {
          sm.abort = 1;
          atomicOr(c.err, ERR_TIMEOUT);
        }
        tc_fence_after();
        tmem_ld(tDV + lane_off, d);
        tc_wait_ld();
      }
      const int g = wt / GK;
      const float f = ldexpf(1.0f, 16) / wscale;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float o = 0.0f;
        if (acc_ok) {
          if constexpr (NG == 1) {
            o = fmaf(d[col_of(0, h, 0, G)] + d[col_of(0, h, 1, G)], f, u_tot[h][0]);
          } else {
            const float a0 = d[col_of(0, h, 0, G)] + d[col_of(0, h, 1, G)];
            const float a1 = d[col_of(1, h, 0, G)] + d[col_of(1, h, 1, G)];
            o = fmaf(g ? a1 : a0, f, g ? u_tot[h][1] : u_tot[h][0]);
          }
        }
        sm.u.fl.o[wg][h][wt] = o;
      }
      if (wt < G) {
        sm.u.fl.ml[wg][wt][0] = acc_ok ? m_ref[wt] : -INFINITY;
        sm.u.fl.ml[wg][wt][1] = acc_ok ? l_tot[wt] : 0.0f;
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (wg == 0) {
        float* rec = int2_recs + (size_t)S.slot * G * PART;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < NWG; ++w) M = fmaxf(M, sm.u.fl.ml[w][h][0]);
          float o = 0.0f, L = 0.0f;
#pragma unroll
          for (int w = 0; w < NWG; ++w) {
            const float mw = sm.u.fl.ml[w][h][0];
            if (mw == -INFINITY) continue;
            const float fw = ex2(mw - M);
            o = fmaf(sm.u.fl.o[w][h][wt], fw, o);
            L = fmaf(sm.u.fl.ml[w][h][1], fw, L);
          }
          rec[h * PART + wt] = o;
          if (wt == 0) {
            rec[h * PART + PARTIAL_M] = M;
            rec[h * PART + PARTIAL_L] = L;
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- BF16 blocks: 32-row half-pages in the warpgroups' own ring memory (every
  // INT2 copy of this CTA has been consumed), unrotated q
  bool any_bf16 = false;
  for (int e = 0; e < nseg; ++e) any_bf16 |= sm.seg[e].bf16 != 0;
  if (any_bf16) {
    if (a.front_writes) grid_dep_wait();   // the ring pages may hold the token just appended
    uint32_t phase_bits = 0;               // per stage: parity of its next completion
    for (int st = 0; st < STAGES; ++st)
      if (((seq - st + STAGES - 1) / STAGES) & 1) phase_bits |= 1u << st;   // completions so far, per stage
    for (int e = 0; e < nseg; ++e) {
      if (!sm.seg[e].bf16) continue;
      const Seg S = sm.seg[e];
      const DecodeReq& R = a.r[S.ri];
      float* qf = reinterpret_cast<float*>(sm.bw[wg]);   // [G][D]
      const uint16_t* qrow = q + ((size_t)R.batch_row * c.Hq + (size_t)S.head * G) * D;
      for (int i = wt; i < G * D; i += WGT) qf[i] = __uint_as_float(static_cast<uint32_t>(qrow[i]) << 16);
      // this warpgroup's half-pages: hp = wg, wg + NWG, ... of the ten, skipping empty ones
      int hps[10], nh = 0;
      for (int hp = wg; hp < 10; hp += NWG) {
        bool any = false;
        for (int r = 0; r < 32 && !any; ++r) any = bf16_row_valid(R, hp >> 1, 32 * (hp & 1) + r);
        if (any) hps[nh++] = hp;
      }
      auto bf16_src = [&](int hp, int which_kv) -> const uint16_t* {
        const int which = hp >> 1;
        int page = which == 0 ? R.sink_page : R.ring_page[which - 1];
        if (page < 0 || page >= c.n_bf16_pages) {
          if (wt == 0) atomicOr(c.err, ERR_BF16_PAGE);
          page = 0;
        }
        return c.bf16 + layer * c.bf16_layer_stride + ((size_t)page * c.Hkv + S.head) * BF16_RECORD_ELEMS +
               (size_t)which_kv * PAGE * D + (size_t)32 * (hp & 1) * D;
      };
      // K rows into stage 2 b, V rows into stage 2 b + 1 (8 KB each) for buffer b
      auto copy_half = [&](int i) {
        if (wt != 0 || sm.abort) return;
        const int b = i & 1;
        mbar_expect_tx(&sm.full[wg][2 * b], 8192);
        tma_load_1d(sm.ring[wg][2 * b], bf16_src(hps[i], 0), 8192, &sm.full[wg][2 * b]);
        mbar_expect_tx(&sm.full[wg][2 * b + 1], 8192);
        tma_load_1d(sm.ring[wg][2 * b + 1], bf16_src(hps[i], 1), 8192, &sm.full[wg][2 * b + 1]);
        issued_mask |= 3u << (2 * b);
      };
      bar_sync(1 + wg, WGT);
      if (nh > 0) copy_half(0);
      if (nh > 1) copy_half(1);
      // online state of heads wiw, wiw + 4 (lane: channels 4 lane .. + 3)
      float bm[2] = {-INFINITY, -INFINITY}, bl[2] = {0.0f, 0.0f}, bo[2][4] = {};
      for (int i = 0; i < nh; ++i) {
        const int b = i & 1, hp = hps[i];
        bool ok = !sm.abort;
        if (ok) {
          ok = mbar_wait(&sm.full[wg][2 * b], (phase_bits >> (2 * b)) & 1, limit) &&
               mbar_wait(&sm.full[wg][2 * b + 1], (phase_bits >> (2 * b + 1)) & 1, limit);
          if (!ok && wt == 0) {
            sm.abort = 1;
            atomicOr(c.err, ERR_TIMEOUT);
          }
        }
        phase_bits ^= 3u << (2 * b);
        if (wt == 0) issued_mask &= ~(3u << (2 * b));
        const uint16_t* kr = reinterpret_cast<const uint16_t*>(sm.ring[wg][2 * b]);
        const uint16_t* vr = reinterpret_cast<const uint16_t*>(sm.ring[wg][2 * b + 1]);
        float* lgs = reinterpret_cast<float*>(sm.ring[wg][2 * b] + 8192);   // [G][32]
        // logits: thread -> row wt / 4, channel quarter wt % 4 (chunks in rotated order)
        {
          const int r = wt >> 2, qq = wt & 3;
          float acc[G];
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] = 0.0f;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const int chunk = 4 * qq + ((bb + r) & 3);
            const uint4 kw = *reinterpret_cast<const uint4*>(kr + (size_t)r * D + 8 * chunk);
            const uint32_t ww[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float k0 = __uint_as_float(ww[e2] << 16), k1 = __uint_as_float(ww[e2] & 0xffff0000u);
              const int chn = 8 * chunk + 2 * e2;
#pragma unroll
              for (int h = 0; h < G; ++h) acc[h] = fmaf(qf[h * D + chn + 1], k1, fmaf(qf[h * D + chn], k0, acc[h]));
            }
          }
          const bool okr = ok && bf16_row_valid(R, hp >> 1, 32 * (hp & 1) + r);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
            acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
            if (qq == 0) lgs[h * 32 + r] = okr ? acc[h] * (c.scale * LOG2E) : -INFINITY;
          }
        }
        bar_sync(1 + wg, WGT);
        // softmax and values: warp wiw handles heads wiw, wiw + 4
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = wiw + 4 * hh;
          if (h >= G) continue;
          const float x = lgs[h * 32 + lane];
          const float mn = fmaxf(bm[hh], warp_max(x));
          if (mn == -INFINITY) continue;
          const float corr = bm[hh] == -INFINITY ? 0.0f : ex2(bm[hh] - mn);
          const float pv = x == -INFINITY ? 0.0f : ex2(x - mn);
          bl[hh] = bl[hh] * corr + warp_sum(pv);
#pragma unroll
          for (int k = 0; k < 4; ++k) bo[hh][k] *= corr;
          bm[hh] = mn;
          for (int r = 0; r < 32; ++r) {
            const float pr = __shfl_sync(0xffffffffu, pv, r);
            if (pr == 0.0f) continue;   // rows outside the window may hold anything
            const uint2 vv = *reinterpret_cast<const uint2*>(vr + (size_t)r * D + 4 * lane);
            bo[hh][0] = fmaf(pr, __uint_as_float(vv.x << 16), bo[hh][0]);
            bo[hh][1] = fmaf(pr, __uint_as_float(vv.x & 0xffff0000u), bo[hh][1]);
            bo[hh][2] = fmaf(pr, __uint_as_float(vv.y << 16), bo[hh][2]);
            bo[hh][3] = fmaf(pr, __uint_as_float(vv.y & 0xffff0000u), bo[hh][3]);
          }
        }
        bar_sync(1 + wg, WGT);   // every thread is done with buffer b
        if (i + 2 < nh) copy_half(i + 2);
      }
      // this warpgroup's BF16 state -> shared memory; warpgroup 0 combines
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = wiw + 4 * hh;
        if (h >= G) continue;
        *reinterpret_cast<float4*>(&sm.u.fl.o[wg][h][4 * lane]) = make_float4(bo[hh][0], bo[hh][1], bo[hh][2], bo[hh][3]);
        if (lane == 0) {
          sm.u.fl.ml[wg][h][0] = bm[hh];
          sm.u.fl.ml[wg][h][1] = bl[hh];
        }
      }
      __syncthreads();
      if (wg == 0) {
        float* rec = bf16_recs + (size_t)(S.ri * c.Hkv + S.head) * G * PART;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < NWG; ++w) M = fmaxf(M, sm.u.fl.ml[w][h][0]);
          float o = 0.0f, L = 0.0f;
#pragma unroll
          for (int w = 0; w < NWG; ++w) {
            const float mw = sm.u.fl.ml[w][h][0];
            if (mw == -INFINITY) continue;
            const float fw = ex2(mw - M);
            o = fmaf(sm.u.fl.o[w][h][wt], fw, o);
            L = fmaf(sm.u.fl.ml[w][h][1], fw, L);
          }
          rec[h * PART + wt] = o;
          if (wt == 0) {
            rec[h * PART + PARTIAL_M] = M;
            rec[h * PART + PARTIAL_L] = L;
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- drain: copies still in flight after an abort land (bounded) before exit
  if (wt == 0 && sm.abort) {
    for (int st = 0; st < STAGES; ++st)
      if (issued_mask & (1u << st)) mbar_wait(&sm.full[wg][st], 0, limit), mbar_wait(&sm.full[wg][st], 1, limit);
  }
  if (wt == 0 && mv_count > 0) mbar_wait(&sm.mv[wg], (mv_count - 1) & 1, limit);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t < 32) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(sm.tmem) : "memory");
}

// ---- merge: one CTA per segment (request, kv head) --------------------------------------
struct MergeSmem {
  float rvt[D][D];          // R_V^T of the kv head: rvt[j][c] = R_V[c][j]
  float oh[MAX_G][D];       // merged INT2 part (rotated basis)
  float ob[MAX_G][D];       // merged BF16 part
  float L[MAX_G];
};

template <int G>
__global__ void __launch_bounds__(MERGE_THREADS) merge_kernel(DevCache c, int layer, DecodeArgs a,
                                                              const float* __restrict__ recs, float* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t merge_raw[];
  MergeSmem& sm = *reinterpret_cast<MergeSmem*>(merge_raw);
  const int s = blockIdx.x, ri = s / c.Hkv, head = s % c.Hkv;
  const int t = threadIdx.x, ch = t % D, hg = t / D;   // hg: heads hg, hg + 2, ...
  {
    // R_V^T is written once at set-up: stage it while the decode grid runs
    const float4* src = reinterpret_cast<const float4*>(c.rot_vt + ((size_t)layer * c.Hkv + head) * D * D);
    float4* dst = reinterpret_cast<float4*>(&sm.rvt[0][0]);
    constexpr int N4 = D * D / 4 / MERGE_THREADS;
    float4 v[N4];
#pragma unroll
    for (int u = 0; u < N4; ++u) v[u] = __ldg(src + u * MERGE_THREADS + t);
#pragma unroll
    for (int u = 0; u < N4; ++u) dst[u * MERGE_THREADS + t] = v[u];
  }
  grid_dep_wait();
  grid_dep_launch();
  const DecodeReq& R = a.r[ri];
  // the CTAs whose cost ranges meet the segment: c_lo .. c_hi, record slot s + cta
  const int64_t per = (int64_t)R.npages + R.bf16_cost;
  const int64_t s0 = R.cost_start + (int64_t)head * per, s1 = s0 + per;
  int c_lo = static_cast<int>(s0 * a.ncta / a.total_cost);
  while (c_lo > 0 && cta_begin(c_lo, a.ncta, a.total_cost) > s0) --c_lo;
  while (cta_begin(c_lo + 1, a.ncta, a.total_cost) <= s0) ++c_lo;
  int c_hi = static_cast<int>((s1 - 1) * a.ncta / a.total_cost);
  while (c_hi > 0 && cta_begin(c_hi, a.ncta, a.total_cost) > s1 - 1) --c_hi;
  while (cta_begin(c_hi + 1, a.ncta, a.total_cost) <= s1 - 1) ++c_hi;
  const float* int2_recs = recs;
  const float* bf16_rec = recs + ((size_t)a.n * c.Hkv + a.ncta) * G * PART + (size_t)s * G * PART;
  for (int h = hg; h < G; h += MERGE_THREADS / D) {
    float M = -INFINITY;
    const float mb = __ldcg(bf16_rec + h * PART + PARTIAL_M);
    M = fmaxf(M, mb);
    for (int cc = c_lo; cc <= c_hi; ++cc) M = fmaxf(M, __ldcg(int2_recs + ((size_t)(s + cc) * G + h) * PART + PARTIAL_M));
    float L = 0.0f, oh = 0.0f, ob = 0.0f;
    if (mb != -INFINITY) {
      const float f = ex2(mb - M);
      L = __ldcg(bf16_rec + h * PART + PARTIAL_L) * f;
      ob = __ldcg(bf16_rec + h * PART + ch) * f;
    }
    for (int cc = c_lo; cc <= c_hi; ++cc) {
      const float* rp = int2_recs + ((size_t)(s + cc) * G + h) * PART;
      const float m = __ldcg(rp + PARTIAL_M);
      if (m == -INFINITY) continue;
      const float f = ex2(m - M);
      L = fmaf(__ldcg(rp + PARTIAL_L), f, L);
      oh = fmaf(__ldcg(rp + ch), f, oh);
    }
    sm.oh[h][ch] = oh;
    sm.ob[h][ch] = ob;
    if (ch == 0) sm.L[h] = L;
  }
  __syncthreads();
  for (int h = hg; h < G; h += MERGE_THREADS / D) {
    float acc = sm.ob[h][ch];
#pragma unroll 8
    for (int j = 0; j < D; ++j) acc = fmaf(sm.oh[h][j], sm.rvt[j][ch], acc);
    out[((size_t)R.batch_row * c.Hq + (size_t)head * G + h) * D + ch] = acc / sm.L[h];
  }
}

template <int G, int GK>
cudaError_t launch_decode_t(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& p,
                            const uint16_t* q, float* out, void* workspace, bool front_writes, DecodeDebug dbg,
                            cudaStream_t s) {
  using Cf = Cfg<G, GK>;
  static unsigned attr_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(attr_done & (1u << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<G, GK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(Smem<G, GK>)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(merge_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(MergeSmem)));
    if (e != cudaSuccess) return e;
    if (dev < 32) attr_done |= 1u << dev;
  }
  DecodeArgs a;
  a.n = p.n;
  a.ncta = p.ncta;
  a.front_writes = front_writes ? 1 : 0;
  a.total_cost = p.total_cost;
  a.dbg = dbg;
  for (int i = 0; i < p.n; ++i) a.r[i] = reqs[i];
  float* recs = static_cast<float*>(workspace);
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.ncta));
  cfg.blockDim = dim3(Cf::THREADS);
  cfg.dynamicSmemBytes = sizeof(Smem<G, GK>);
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel<G, GK>, c, layer, a, q, recs);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(p.segments));
  cfg.blockDim = dim3(MERGE_THREADS);
  cfg.dynamicSmemBytes = sizeof(MergeSmem);
  return cudaLaunchKernelEx(&cfg, merge_kernel<G>, c, layer, a, static_cast<const float*>(recs), out);
}

template <int GK>
cudaError_t launch_decode_g(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& p,
                            const uint16_t* q, float* out, void* ws, bool fw, DecodeDebug dbg, cudaStream_t s) {
  switch (c.G) {
    case 1: return launch_decode_t<1, GK>(c, layer, reqs, p, q, out, ws, fw, dbg, s);
    case 2: return launch_decode_t<2, GK>(c, layer, reqs, p, q, out, ws, fw, dbg, s);
    case 4: return launch_decode_t<4, GK>(c, layer, reqs, p, q, out, ws, fw, dbg, s);
    case 8: return launch_decode_t<8, GK>(c, layer, reqs, p, q, out, ws, fw, dbg, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DevCache& c, int layer, const DecodeReq* reqs, const DecodePlan& p,
                          const uint16_t* q, float* out, void* workspace, bool front_writes, DecodeDebug dbg,
                          cudaStream_t s) {
  if (p.n < 1 || p.n > DECODE_PER_LAUNCH || p.ncta < 1) return cudaErrorInvalidValue;
  return c.gk == 64 ? launch_decode_g<64>(c, layer, reqs, p, q, out, workspace, front_writes, dbg, s)
                    : launch_decode_g<128>(c, layer, reqs, p, q, out, workspace, front_writes, dbg, s);
}

cudaError_t launch_step(const DevCache& c, int layer, const AppendReq* app, int n_app, const uint16_t* k,
                        const uint16_t* v, const DecodeReq* reqs, const DecodePlan& p, const uint16_t* q,
                        float* out, void* workspace, DecodeDebug dbg, cudaStream_t s) {
  const cudaError_t e = launch_append(c, layer, app, n_app, k, v, s);
  if (e != cudaSuccess) return e;
  return launch_decode(c, layer, reqs, p, q, out, workspace, true, dbg, s);
}

}  // namespace oscar
