// Uncompressed BF16 paged decode attention: the baseline the INT2 path is
// measured against.
//
// "Together AI Open-Sources OSCAR" (MarkTechPost), section "Results": decode
// speed of the 2-bit cache is reported against a BF16 KV cache of the same
// context.  This is that baseline written for the same GPU and the same
// measurement: plain softmax attention of every query head over all T cached
// tokens, out = softmax(q K^T / sqrt(d)) V, with the KV in 64-token pages
// [page][kv head][K rows, V rows][64][128] bf16.
//
// Two launches.  The stream kernel splits the pages of each (request, kv head)
// into chunks, one block each; its four warps take 16-token sub-pages through a
// two-stage cp.async ring into padded shared rows.  q K^T and P V run on
// mma.sync m16n8k16 bf16 with fp32 accumulation: q is exact in bf16, and P is
// carried as bf16 hi + lo parts, so every product is exact in fp32.  Columns of
// both contractions are (query head, part) pairs, so a lane's logits, weights
// and output accumulators all belong to one head.  The softmax keeps a
// reference max that moves only when exceeded by 2^8.  Rows past a request's
// length are zero-filled by the copies and masked out.  The merge kernel folds
// the chunk partials of each query head.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "oscar.h"

namespace oscar {
namespace {

constexpr float BF_LOG2E = 1.4426950408889634f;
constexpr int BF_WARPS = 4;
constexpr int BF_THREADS = 32 * BF_WARPS;
constexpr int BF_SUB = 16;                 // tokens per sub-page (one k-step of P V)
constexpr int BF_SUBS = PAGE / BF_SUB;     // sub-pages per page
constexpr int BF_PITCH = D + 8;            // bf16 per staged row: ldmatrix without bank conflicts
constexpr int BF_WPITCH = BF_SUB + 8;      // bf16 per weight column
constexpr float BF_LAZY = 8.0f;            // the reference max moves only when exceeded by 2^8
constexpr int BF_MERGE_THREADS = 128;
constexpr int BF_MERGE_WARPS = BF_MERGE_THREADS / 32;
constexpr int BF_MERGE_UNROLL = 4;         // chunk partials in flight per merge warp
constexpr int BF_MAX_REQ = 64;             // requests per launch

struct BfArgs {
  int n, Hq, Hkv, max_pages, ppc;
  int64_t num_pages;
  float scale;
  int block_start[BF_MAX_REQ];   // first stream block of request i
  int chunks[BF_MAX_REQ];        // chunks (blocks) per kv head of request i
  int len[BF_MAX_REQ];           // tokens of request i
};

struct BfStage {
  __align__(16) uint16_t k[BF_SUB][BF_PITCH];
  __align__(16) uint16_t v[BF_SUB][BF_PITCH];
};
template <int G>
struct BfSmem {
  static constexpr int NT = (2 * G + 7) / 8;
  union {
    BfStage ring[BF_WARPS][2];
    float state[BF_WARPS][G][PARTIAL_FLOATS];   // after the page loop
  } u;
  __align__(16) uint16_t w[BF_WARPS][NT][8][BF_WPITCH];   // P: [n-tile][column][token]
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm4_t(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ float bf16_value(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Chunk c of the pages of (request ri, kv head h): pages [c ppc, (c + 1) ppc).
// Warp w takes sub-pages w, w + 4, ... of the chunk.  Partial of query head g of
// the group: partials[blockIdx.x][g][PARTIAL_FLOATS] (log2-domain max).
template <int G>
__global__ void __launch_bounds__(BF_THREADS, 3) bf16_stream_kernel(BfArgs a, const uint16_t* __restrict__ kv,
                                                                    const int32_t* __restrict__ pt,
                                                                    const uint16_t* __restrict__ q,
                                                                    float* __restrict__ partials, int32_t* err) {
  constexpr int NT = BfSmem<G>::NT;   // n-tiles of 8 (head, hi / lo) columns
  extern __shared__ __align__(16) uint8_t bf_raw[];
  BfSmem<G>& sm = *reinterpret_cast<BfSmem<G>*>(bf_raw);
  // the merge grid may be scheduled now; it waits for this grid's completion
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  int ri = 0;
  while (ri + 1 < a.n && a.block_start[ri + 1] <= (int)blockIdx.x) ++ri;
  const int local = blockIdx.x - a.block_start[ri];
  const int head = local / a.chunks[ri], chunk = local % a.chunks[ri];
  const int T = a.len[ri];
  const int npages = (T + PAGE - 1) / PAGE;
  const int p0 = chunk * a.ppc, p1 = min(npages, p0 + a.ppc);
  const int nsub = max(0, p1 - p0) * BF_SUBS;
  const int32_t* prow = pt + (size_t)ri * a.max_pages;
  const float scale2 = a.scale * BF_LOG2E;

  // q as the B operand of K q^T: column n of n-tile nt is query head 4 nt + (n >> 1)
  // (each head twice), k-step s, registers (b0, b1)
  uint32_t bq[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 4 * nt + (gid >> 1);
    const uint16_t* qh = q + ((size_t)ri * a.Hq + (size_t)head * G + (g < G ? g : 0)) * D;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t x0 = *reinterpret_cast<const uint32_t*>(qh + 16 * s + 2 * tid);
      const uint32_t x1 = *reinterpret_cast<const uint32_t*>(qh + 16 * s + 2 * tid + 8);
      bq[nt][s][0] = g < G ? x0 : 0u;
      bq[nt][s][1] = g < G ? x1 : 0u;
    }
  }
  // copy of this warp's j-th sub-page into stage st (a group is committed even
  // when there is nothing to copy, so the waits below stay in step)
  const int my_n = nsub > warp ? (nsub - warp + BF_WARPS - 1) / BF_WARPS : 0;
  auto copy_sub = [&](int j, int st) {
    if (j < my_n) {
      const int sp = warp + BF_WARPS * j;
      const int pi = p0 + sp / BF_SUBS, r0 = (sp % BF_SUBS) * BF_SUB;
      int32_t page = prow[pi];
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0) atomicOr(err, 1);
        page = 0;
      }
      const uint16_t* kb = kv + ((size_t)page * a.Hkv + head) * (2 * PAGE * D) + (size_t)r0 * D;
      const uint16_t* vb = kb + (size_t)PAGE * D;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = u * 32 + lane, row = idx >> 4, part = idx & 15;
        const bool ok = pi * PAGE + r0 + row < T;
        cp_async16(&sm.u.ring[warp][st].k[row][8 * part], kb + (ok ? row * D + 8 * part : 0), ok);
        cp_async16(&sm.u.ring[warp][st].v[row][8 * part], vb + (ok ? row * D + 8 * part : 0), ok);
      }
    }
    cp_async_commit();
  };
  copy_sub(0, 0);
  copy_sub(1, 1);

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
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = 8 * (lane >> 4);   // K as A (ldmatrix)
  const int vrow = (lane & 7) + 8 * (lane >> 4), vcol = 8 * ((lane >> 3) & 1);   // V^T as A (ldmatrix.trans)

  for (int j = 0; j < my_n; ++j) {
    const int st = j & 1;
    cp_async_wait1();
    __syncwarp();
    const BfStage& sg = sm.u.ring[warp][st];
    const int sp = warp + BF_WARPS * j;
    const int tok0 = (p0 + sp / BF_SUBS) * PAGE + (sp % BF_SUBS) * BF_SUB;
    // ---- logits: S [16 tokens x 8 columns] per n-tile over the 128 channels
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t af[4];
      ldsm4(af, &sg.k[arow][16 * ks + acol]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(s[nt], af, bq[nt][ks][0], bq[nt][ks][1]);
    }
    // ---- softmax of the lane's head 4 nt + tid over tokens gid, gid + 8; the
    // weights go to shared memory as bf16 hi (column 2 tid) and lo (2 tid + 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const bool hok = 4 * nt + tid < G;
      const float la = (hok && tok0 + gid < T) ? s[nt][0] * scale2 : -INFINITY;
      const float lb = (hok && tok0 + gid + 8 < T) ? s[nt][2] * scale2 : -INFINITY;
      float pm = fmaxf(la, lb);
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      if (pm > m_run[nt] + BF_LAZY) {
        const float corr = m_run[nt] == -INFINITY ? 0.0f : ex2f(m_run[nt] - pm);
        m_run[nt] = pm;
        l_run[nt] *= corr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][mt][e] *= corr;
      }
      const float pa = la == -INFINITY ? 0.0f : ex2f(la - m_run[nt]);
      const float pb = lb == -INFINITY ? 0.0f : ex2f(lb - m_run[nt]);
      l_run[nt] += pa + pb;
      const uint16_t ha = bf16_bits(pa), hb = bf16_bits(pb);
      uint16_t(*wc)[BF_WPITCH] = sm.w[warp][nt];
      wc[2 * tid][gid] = ha;
      wc[2 * tid][gid + 8] = hb;
      wc[2 * tid + 1][gid] = bf16_bits(pa - bf16_value(ha));
      wc[2 * tid + 1][gid + 8] = bf16_bits(pb - bf16_value(hb));
    }
    __syncwarp();
    // ---- values: O [128 channels x 8 columns] += V^T P over the 16 tokens
    uint32_t bw[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bw[nt][0] = *reinterpret_cast<const uint32_t*>(&sm.w[warp][nt][gid][2 * tid]);
      bw[nt][1] = *reinterpret_cast<const uint32_t*>(&sm.w[warp][nt][gid][2 * tid + 8]);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t af[4];
      ldsm4_t(af, &sg.v[vrow][16 * mt + vcol]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(o[nt][mt], af, bw[nt][0], bw[nt][1]);
    }
    __syncwarp();   // the stage and the weights are free
    copy_sub(j + 2, st);
  }

  // ---- this warp's state -> shared memory (over the rings: every warp is done
  // with its ring first), then the warps merged per channel
  __syncthreads();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float l = l_run[nt];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const int g = 4 * nt + tid;
    if (g < G) {
      float* stt = sm.u.state[warp][g];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        // o rows: channels 16 mt + gid and + 8; columns hi and lo of head g
        stt[16 * mt + gid] = o[nt][mt][0] + o[nt][mt][1];
        stt[16 * mt + gid + 8] = o[nt][mt][2] + o[nt][mt][3];
      }
      if (gid == 0) {
        stt[PARTIAL_M] = m_run[nt];
        stt[PARTIAL_L] = l;
      }
    }
  }
  __syncthreads();
  const int t = threadIdx.x;   // channel t (BF_THREADS == D)
  float* part = partials + (size_t)blockIdx.x * G * PARTIAL_FLOATS;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < BF_WARPS; ++w) M = fmaxf(M, sm.u.state[w][g][PARTIAL_M]);
    float acc_o = 0.0f, acc_l = 0.0f;
#pragma unroll
    for (int w = 0; w < BF_WARPS; ++w) {
      const float mw = sm.u.state[w][g][PARTIAL_M];
      if (mw == -INFINITY) continue;
      const float f = exp2f(mw - M);
      acc_o = fmaf(sm.u.state[w][g][t], f, acc_o);
      acc_l = fmaf(sm.u.state[w][g][PARTIAL_L], f, acc_l);
    }
    part[g * PARTIAL_FLOATS + t] = acc_o;
    if (t == 0) {
      part[g * PARTIAL_FLOATS + PARTIAL_M] = M;
      part[g * PARTIAL_FLOATS + PARTIAL_L] = acc_l;
    }
  }
}

// One block per (request, query head): fold the chunk partials.  Warp w takes
// chunks w, w + 4, ..., BF_MERGE_UNROLL at a time with lane l holding channels
// 4 l .. 4 l + 3; the warps' states are then folded per channel.
template <int G>
__global__ void __launch_bounds__(BF_MERGE_THREADS) bf16_merge_kernel(BfArgs a, const float* __restrict__ partials,
                                                                      float* __restrict__ out) {
  __shared__ float s_m[BF_MERGE_WARPS], s_l[BF_MERGE_WARPS];
  __shared__ __align__(16) float s_o[BF_MERGE_WARPS][D];
  const int ri = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq;
  const int head = hq / G, g = hq % G;
  const int nch = a.chunks[ri];
  constexpr size_t STRIDE = (size_t)G * PARTIAL_FLOATS;
  const float* base = partials + ((size_t)a.block_start[ri] + (size_t)head * nch) * STRIDE + (size_t)g * PARTIAL_FLOATS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_wait();   // the stream grid's partials are complete and visible
  float m = -INFINITY, l = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int c0 = warp; c0 < nch; c0 += BF_MERGE_WARPS * BF_MERGE_UNROLL) {
    float mv[BF_MERGE_UNROLL], lv[BF_MERGE_UNROLL];
    float4 ov[BF_MERGE_UNROLL];
#pragma unroll
    for (int u = 0; u < BF_MERGE_UNROLL; ++u) {
      const int c = c0 + BF_MERGE_WARPS * u;
      mv[u] = -INFINITY;
      lv[u] = 0.0f;
      ov[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (c < nch) {
        const float* p = base + (size_t)c * STRIDE;
        mv[u] = __ldg(p + PARTIAL_M);
        lv[u] = __ldg(p + PARTIAL_L);
        ov[u] = __ldg(reinterpret_cast<const float4*>(p) + lane);
      }
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < BF_MERGE_UNROLL; ++u) mn = fmaxf(mn, mv[u]);
    if (mn == -INFINITY) continue;   // nothing seen yet (exp2f(-inf) is 0 from here on)
    const float f = exp2f(m - mn);
    l *= f;
    acc.x *= f;
    acc.y *= f;
    acc.z *= f;
    acc.w *= f;
#pragma unroll
    for (int u = 0; u < BF_MERGE_UNROLL; ++u) {
      const float fu = exp2f(mv[u] - mn);
      l = fmaf(lv[u], fu, l);
      acc.x = fmaf(ov[u].x, fu, acc.x);
      acc.y = fmaf(ov[u].y, fu, acc.y);
      acc.z = fmaf(ov[u].z, fu, acc.z);
      acc.w = fmaf(ov[u].w, fu, acc.w);
    }
    m = mn;
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
  reinterpret_cast<float4*>(s_o[warp])[lane] = acc;
  __syncthreads();
  const int t = threadIdx.x;   // channel t (BF_MERGE_THREADS == D)
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < BF_MERGE_WARPS; ++w) M = fmaxf(M, s_m[w]);
  float o = 0.0f, L = 0.0f;
#pragma unroll
  for (int w = 0; w < BF_MERGE_WARPS; ++w) {
    if (s_m[w] == -INFINITY) continue;
    const float f = exp2f(s_m[w] - M);
    o = fmaf(s_o[w][t], f, o);
    L = fmaf(s_l[w], f, L);
  }
  out[((size_t)ri * a.Hq + hq) * D + t] = o / L;
}

template <int G>
cudaError_t launch_bf16(const BfArgs& a, int blocks, const uint16_t* kv, const int32_t* pt, const uint16_t* q,
                        float* partials, int32_t* err, float* out, cudaStream_t s) {
  static unsigned done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(done & (1u << dev))) {
    e = cudaFuncSetAttribute(bf16_stream_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(BfSmem<G>)));
    if (e != cudaSuccess) return e;
    if (dev < 32) done |= 1u << dev;
  }
  bf16_stream_kernel<G><<<blocks, BF_THREADS, sizeof(BfSmem<G>), s>>>(a, kv, pt, q, partials, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the merge's launch overlaps the stream grid's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n * a.Hq);
  cfg.blockDim = dim3(BF_MERGE_THREADS);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bf16_merge_kernel<G>, a, static_cast<const float*>(partials), out);
}

constexpr int BF_CTAS_PER_SM = 3;
constexpr int64_t BF_MAX_CHUNKS = 256;  // chunks per (request, kv head) the plan considers
constexpr size_t BF_ERR_BYTES = 256;   // the error word, padded

// Chunks per kv head of each request and pages per chunk.  Blocks are equal in
// size, so the grid runs in ceil(blocks / slots) rounds of ppc pages each; a
// block also costs about one page of start-up and partial write.  The plan
// takes the ppc (one of ceil(max pages / c)) with the least estimated time.
int bf16_plan(int32_t n, const int32_t* lens, int32_t hkv, int sms, BfArgs& a) {
  int64_t max_np = 1;
  for (int32_t i = 0; i < n; ++i) max_np = std::max<int64_t>(max_np, (lens[i] + PAGE - 1) / PAGE);
  const int64_t slots = (int64_t)sms * BF_CTAS_PER_SM;
  auto blocks_for = [&](int64_t ppc) {
    int64_t b = 0;
    for (int32_t i = 0; i < n; ++i) b += hkv * std::max<int64_t>(1, ((lens[i] + PAGE - 1) / PAGE + ppc - 1) / ppc);
    return b;
  };
  int64_t best_ppc = max_np, best_cost = -1;
  for (int64_t c = 1; c <= std::min<int64_t>(max_np, BF_MAX_CHUNKS); ++c) {
    const int64_t ppc = (max_np + c - 1) / c;
    const int64_t rounds = (blocks_for(ppc) + slots - 1) / slots;
    const int64_t cost = rounds * (ppc + 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_ppc = ppc;
    }
  }
  int blocks = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t np = (lens[i] + PAGE - 1) / PAGE;
    const int ch = static_cast<int>(std::max<int64_t>(1, (np + best_ppc - 1) / best_ppc));
    a.block_start[i] = blocks;
    a.chunks[i] = ch;
    a.len[i] = lens[i];
    blocks += ch * hkv;
  }
  a.ppc = static_cast<int>(best_ppc);
  return blocks;
}

}  // namespace
}  // namespace oscar

using namespace oscar;

extern "C" {

size_t oscar_bf16_decode_workspace_bytes(int32_t n, const int32_t* lens, int32_t num_q_heads, int32_t num_kv_heads) {
  if (n <= 0 || n > BF_MAX_REQ || !lens || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  for (int32_t i = 0; i < n; ++i)
    if (lens[i] <= 0) return 0;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  BfArgs a{};
  const int blocks = bf16_plan(n, lens, num_kv_heads, sms, a);
  return BF_ERR_BYTES + (size_t)blocks * (num_q_heads / num_kv_heads) * PARTIAL_FLOATS * sizeof(float);
}

oscar_status oscar_bf16_decode(const void* kv, int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                               const int32_t* lens, int32_t n, int32_t num_q_heads, int32_t num_kv_heads,
                               float softmax_scale, const void* q, float* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!kv || !page_table || !lens || !q || !out || !workspace || num_pages <= 0 || max_pages <= 0 || n <= 0 ||
      n > BF_MAX_REQ || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads)
    return OSCAR_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return OSCAR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(workspace)) & 15)
    return OSCAR_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (lens[i] <= 0 || (int64_t)(lens[i] + PAGE - 1) / PAGE > max_pages) return OSCAR_ERR_INVALID_ARG;
  const size_t need = oscar_bf16_decode_workspace_bytes(n, lens, num_q_heads, num_kv_heads);
  if (need == 0 || workspace_bytes < need) return OSCAR_ERR_INVALID_ARG;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  BfArgs a{};
  a.n = n;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(D));
  const int blocks = bf16_plan(n, lens, num_kv_heads, sms, a);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* err = static_cast<int32_t*>(workspace);
  float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + BF_ERR_BYTES);
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
  const uint16_t* kvp = static_cast<const uint16_t*>(kv);
  const uint16_t* qp = static_cast<const uint16_t*>(q);
  if (e == cudaSuccess) {
    switch (G) {
      case 1: e = launch_bf16<1>(a, blocks, kvp, page_table, qp, partials, err, out, s); break;
      case 2: e = launch_bf16<2>(a, blocks, kvp, page_table, qp, partials, err, out, s); break;
      case 4: e = launch_bf16<4>(a, blocks, kvp, page_table, qp, partials, err, out, s); break;
      default: e = launch_bf16<8>(a, blocks, kvp, page_table, qp, partials, err, out, s); break;
    }
  }
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // extern "C"
