// Write path: page-table updates, rotation set-up, prefill-quantize and the
// fused append + demote kernel.
//
// "Together AI Open-Sources OSCAR" (MarkTechPost), section "The Serving
// System: Mixed-Precision Cache Layout": each history token is rotated by
// R_K / R_V, clipped to the calibration threshold and quantised to per-token
// asymmetric INT2; "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计":
// new tokens enter the BF16 recent window and the oldest recent token is
// rotated, clipped, quantised and packed (4 codes per byte) into INT2 history.
//
// Every quantisation decision is taken on fp32_rn(k . R) exactly (see
// quant_device.cuh), whatever order a kernel's fp32 FMA chain takes, so prefill
// and sequential appends write identical bytes.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "append_device.cuh"
#include "quant_device.cuh"

namespace oscar {
namespace {

struct PtArgs {
  int n;
  PtEntry e[PT_ENTRIES_PER_LAUNCH];
};

__global__ void pt_update_kernel(int32_t* hist_pt, int32_t* bf16_pt, PtArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < a.n) {
    int32_t* t = a.e[i].table == 0 ? hist_pt : bf16_pt;
    t[a.e[i].index] = a.e[i].value;
  }
}

__global__ void rotation_setup_kernel(const float* __restrict__ src_k, const float* __restrict__ src_v,
                                      float* rk, float* rv, float* rkt, float* rvt, size_t mats) {
  const size_t total = mats * D * D;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t m = idx / (D * D);
    const int i = static_cast<int>((idx / D) % D);
    const int j = static_cast<int>(idx % D);
    const float a = src_k[idx];
    const float b = src_v[idx];
    rk[idx] = a;
    rv[idx] = b;
    rkt[m * D * D + (size_t)j * D + i] = a;
    rvt[m * D * D + (size_t)j * D + i] = b;
  }
}

// Largest column norm of each matrix (K matrices, then V), rounded up so it
// bounds the exact norm: one block per matrix, one thread per column.
__global__ void __launch_bounds__(D) colnorm_kernel(const float* __restrict__ src_k, const float* __restrict__ src_v,
                                                    float* out, int mats) {
  __shared__ float red[D];
  const int m = blockIdx.x;
  const float* R = (m < mats ? src_k : src_v) + (size_t)(m % mats) * D * D;
  float acc = 0.0f;
  for (int i = 0; i < D; ++i) acc = __fmaf_ru(R[i * D + threadIdx.x], R[i * D + threadIdx.x], acc);
  red[threadIdx.x] = __fsqrt_ru(__fmul_ru(acc, 1.0001f));
  __syncthreads();
  for (int w = D / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) out[m] = red[0];
}

// One position of the sink or the recent ring per block (x), K or V (y).
__global__ void __launch_bounds__(128) prefill_bf16_kernel(DevCache c, int layer, const uint16_t* __restrict__ k,
                                                           const uint16_t* __restrict__ v, int64_t in_base,
                                                           int64_t p0, BF16Dest dst) {
  const int64_t p = p0 + blockIdx.x;
  const int which = blockIdx.y;
  const uint16_t* src = (which ? v : k) + (size_t)(p - in_base) * c.Hkv * D;
  int page, row;
  if (p < SINK) {
    page = dst.sink_page;
    row = static_cast<int>(p);
  } else {
    const int slot = static_cast<int>((p - SINK) % RECENT);
    page = dst.ring_page[slot / PAGE];
    row = slot % PAGE;
  }
  if (page < 0 || page >= c.n_bf16_pages) {
    if (threadIdx.x == 0) atomicOr(c.err, ERR_BF16_PAGE);
    return;
  }
  for (int idx = threadIdx.x; idx < c.Hkv * (D / 8); idx += blockDim.x) {
    const int head = idx / (D / 8);
    const int part = idx % (D / 8);
    const uint4 val = reinterpret_cast<const uint4*>(src + (size_t)head * D)[part];
    reinterpret_cast<uint4*>(bf16_row(c, layer, page, head, which, row))[part] = val;
  }
}

// ---- prefill_hist: rotation on the tensor cores -----------------------------------
// x = k . R for a tile of tokens is a dense [tokens x 128] . [128 x 128]
// contraction.  k is bf16, so with R split into bf16 parts R = R1 + R2 + d
// (R1 = bf16_rn(R), R2 = bf16_rn(R - R1), |d| <= 2^-18 |R|) every product
// k_i R_ij is exact in the MMA's fp32.  Each 16-channel k-step s is one
// mma.sync m16n8k16 into a zero accumulator, giving P1_s (R1) and P2_s (R2), and
//   x~ = fl(sum_s P1_s + sum_s P2_s)    (IEEE fp32 adds, s = 0 .. 7).
// Error bound, with S = sum_i |k_i R_ij| <= |k|_2 colnorm and u = 2^-24: one MMA
// adds 16 exact products; with them aligned to the largest, each truncated by
// under one fp32 ulp of it and the sum by under one ulp of itself, it errs by at
// most 34 u sum |p|.  The R1 part (eight MMAs, seven adds) so errs by at most
// (34 u + 7 u) S (1 + 2^-9), the R2 part by 2^-8 of that, d contributes 2^-18 S
// and the final add u |x|: in all below 6.4e-6 S, within the 2^-17 S used
// (= gamma_128, the bound of a 128-term fp32 FMA chain).
// (Measured on a GB300: the worst error of eight chained MMAs over 4000 random
// problems with outlier channels and a 2^24 exponent spread was 2^-20.4 of
// sum |p|, well inside the per-MMA model.)  The quantiser's decisions
// (quant_device.cuh) then stay exact for any value of that interval.
constexpr int PF_TILE = 32;          // history positions per tile
constexpr int PF_THREADS = 256;
constexpr int PF_PITCH = D + 8;      // bf16 elements per staged row (ldmatrix without bank conflicts)
constexpr float PF_MMA_ERR = 0x1p-17f;
struct PrefillSmem {
  __align__(16) uint16_t r1[D][PF_PITCH];      // R1^T: row n = output channel n, k contiguous
  __align__(16) uint16_t r2[D][PF_PITCH];      // R2^T
  __align__(16) uint16_t kb[2][PF_TILE][PF_PITCH];  // the tile as bf16, double-buffered (zero rows past its end)
  __align__(16) float xs[PF_TILE][D + 4];       // rotated values (row pad: no bank conflicts)
  float kn[PF_TILE];                            // |k|^2 of each token, rounded up
  int32_t page;                                 // id of the history page holding the tile
};
constexpr size_t PREFILL_SMEM = sizeof(PrefillSmem);

// 16-byte asynchronous global -> shared copy; a zero-size source fills zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

// One k-step into a zero accumulator, added to acc with IEEE fp32 adds.
__device__ __forceinline__ void mma_bf16_add(float (&acc)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  float d0, d1, d2, d3;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
  acc[0] = __fadd_rn(acc[0], d0);
  acc[1] = __fadd_rn(acc[1], d1);
  acc[2] = __fadd_rn(acc[2], d2);
  acc[3] = __fadd_rn(acc[3], d3);
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Block x of the history of one kv head (y), K or V (z): tiles
// [x tiles_per_cta, (x + 1) tiles_per_cta) of the launch.  Tile i covers history
// slots [PF_TILE (k0 + i), PF_TILE (k0 + i + 1)) -- aligned to PF_TILE, so a tile
// lies in one page -- restricted to the positions [h0, h1) being written.  The launch sizes the grid
// to two resident blocks per SM, so R is split and staged once per block.
template <int GK>
__global__ void __launch_bounds__(PF_THREADS, 2) prefill_hist_kernel(DevCache c, int layer, int slot,
                                                                  const uint16_t* __restrict__ k,
                                                                  const uint16_t* __restrict__ v,
                                                                  int64_t in_base, int64_t h0, int64_t h1,
                                                                  int64_t k0, int64_t tiles, int tiles_per_cta) {
  extern __shared__ __align__(16) uint8_t pf_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(pf_raw);
  const int head = blockIdx.y;
  const int which = blockIdx.z;
  const uint16_t* src = which ? v : k;
  const size_t lh = (size_t)layer * c.Hkv + head;
  const float* __restrict__ Rt = (which ? c.rot_vt : c.rot_kt) + lh * D * D;
  const float tau = (which ? c.tau_v : c.tau_k)[lh];
  const float colnorm = c.rot_cn[(size_t)which * c.L * c.Hkv + lh];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int gid = lane >> 2, tid = lane & 3;
  const int32_t* pt = c.hist_pt + (size_t)slot * c.max_pages;

  // R^T = (R1 + R2)^T in bf16, row n = output channel; the loads of a batch are
  // all in flight before any is used
  constexpr int RB = 8;
  for (int base = t; base < D * D / 4; base += RB * PF_THREADS) {
    float4 rb[RB];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int idx = base + u * PF_THREADS;
      rb[u] = idx < D * D / 4 ? *reinterpret_cast<const float4*>(Rt + (size_t)4 * idx) : make_float4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < RB; ++u) {
    const int idx = base + u * PF_THREADS;
    if (idx >= D * D / 4) break;
    const int n = idx / (D / 4), k4 = 4 * (idx % (D / 4));
    const float4 r = rb[u];
    const float rv[4] = {r.x, r.y, r.z, r.w};
    uint16_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hi[e] = bf16_rn_bits(rv[e]);
      lo[e] = bf16_rn_bits(rv[e] - bf16_bits_to_float(hi[e]));
    }
    *reinterpret_cast<uint2*>(&sm.r1[n][k4]) =
        make_uint2(hi[0] | (uint32_t(hi[1]) << 16), hi[2] | (uint32_t(hi[3]) << 16));
    *reinterpret_cast<uint2*>(&sm.r2[n][k4]) =
        make_uint2(lo[0] | (uint32_t(lo[1]) << 16), lo[2] | (uint32_t(lo[3]) << 16));
    }
  }

  // this warp's part of a tile's outputs: m-tile (warp & 1), n-tiles 4 (warp >> 1) .. + 3
  const int mrow = 16 * (warp & 1);
  const int ncol = 32 * (warp >> 1);
  const int64_t tile_begin = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t tile_end = min(tiles, tile_begin + tiles_per_cta);
  // a tile is PF_TILE tokens x 128 channels of bf16, 16 bytes per copy; the next
  // tile is copied while the current one is rotated and quantised.  Row j of tile
  // i is position t0 + j, t0 = SINK + PF_TILE (k0 + i); rows outside [h0, h1) are
  // zero-filled and skipped
  constexpr int CHUNKS = PF_TILE * D / 8 / PF_THREADS;
  auto copy_tile = [&](int64_t tile, int buf) {
    const int64_t t0 = SINK + PF_TILE * (k0 + tile);
#pragma unroll
    for (int u = 0; u < CHUNKS; ++u) {
      const int idx = u * PF_THREADS + t, j = idx / (D / 8), part = idx % (D / 8);
      const bool ok = t0 + j >= h0 && t0 + j < h1;
      const uint16_t* g = src + ((size_t)(ok ? t0 + j - in_base : 0) * c.Hkv + head) * D + 8 * part;
      cp_async16(&sm.kb[buf][j][8 * part], g, ok);
    }
    cp_async_commit();
  };
  if (tile_begin < tile_end) copy_tile(tile_begin, 0);
  for (int64_t tile = tile_begin; tile < tile_end; ++tile) {
    const int buf = static_cast<int>((tile - tile_begin) & 1);
    const int64_t t0 = SINK + PF_TILE * (k0 + tile);
    const int jlo = static_cast<int>(h0 - t0 > 0 ? h0 - t0 : 0);
    const int jhi = static_cast<int>(h1 - t0 < PF_TILE ? h1 - t0 : PF_TILE);
    cp_async_wait_all();
    __syncthreads();   // this tile has landed; the other buffer, xs and vb are free
    if (tile + 1 < tile_end) copy_tile(tile + 1, buf ^ 1);
    if (t == 0) sm.page = __ldg(pt + (t0 - SINK) / PAGE);   // read after the rotation
    {
      // |k|^2 of each token, rounded up: 16 consecutive threads share a token
#pragma unroll
      for (int u = 0; u < CHUNKS; ++u) {
        const int idx = u * PF_THREADS + t, j = idx / (D / 8), part = idx % (D / 8);
        const uint4 val = *reinterpret_cast<const uint4*>(&sm.kb[buf][j][8 * part]);
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
        float sq = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float f0 = __uint_as_float(w[e] << 16), f1 = __uint_as_float(w[e] & 0xffff0000u);
          sq = __fmaf_ru(f0, f0, sq);
          sq = __fmaf_ru(f1, f1, sq);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) sq = __fadd_ru(sq, __shfl_xor_sync(0xffffffffu, sq, off));
        if (part == 0) sm.kn[j] = sq;
      }
    }

    // x~ for rows mrow .. mrow + 15, channels ncol .. ncol + 31
    {
      float acc1[4][4], acc2[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc1[nt][e] = acc2[nt][e] = 0.0f;
      // ldmatrix lane addresses: A (rows of the tile), B (rows of R^T)
      const int arow = mrow + (lane & 7) + 8 * ((lane >> 3) & 1), akoff = 8 * (lane >> 4);
      const int brow = (lane & 7) + 8 * (lane >> 4), bkoff = 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, &sm.kb[buf][arow][16 * ks + akoff]);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          // n-tiles 2 np, 2 np + 1 of this warp: b0 / b1 of each
          uint32_t h0r, h1r, h2r, h3r, l0r, l1r, l2r, l3r;
          ldsm_x4(h0r, h1r, h2r, h3r, &sm.r1[ncol + 16 * np + brow][16 * ks + bkoff]);
          ldsm_x4(l0r, l1r, l2r, l3r, &sm.r2[ncol + 16 * np + brow][16 * ks + bkoff]);
          mma_bf16_add(acc1[2 * np], a0, a1, a2, a3, h0r, h1r);
          mma_bf16_add(acc1[2 * np + 1], a0, a1, a2, a3, h2r, h3r);
          mma_bf16_add(acc2[2 * np], a0, a1, a2, a3, l0r, l1r);
          mma_bf16_add(acc2[2 * np + 1], a0, a1, a2, a3, l2r, l3r);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = ncol + 8 * nt + 2 * tid;
        *reinterpret_cast<float2*>(&sm.xs[mrow + gid][col]) =
            make_float2(__fadd_rn(acc1[nt][0], acc2[nt][0]), __fadd_rn(acc1[nt][1], acc2[nt][1]));
        *reinterpret_cast<float2*>(&sm.xs[mrow + gid + 8][col]) =
            make_float2(__fadd_rn(acc1[nt][2], acc2[nt][2]), __fadd_rn(acc1[nt][3], acc2[nt][3]));
      }
    }
    __syncthreads();

    for (int j = jlo + warp; j < jhi; j += PF_THREADS / 32) {
      const float4 x = *reinterpret_cast<const float4*>(&sm.xs[j][4 * lane]);
      const uint2 kw = *reinterpret_cast<const uint2*>(&sm.kb[buf][j][4 * lane]);
      const float4 k4 = make_float4(__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xffff0000u),
                                    __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xffff0000u));
      const float sbound = __fmul_ru(__fsqrt_ru(__fmul_ru(sm.kn[j], 1.0001f)), colnorm);   // >= sum_i |k_i R_ic|
      const float err = __fmul_ru(sbound, PF_MMA_ERR);
      const GroupCode g = quantize_group_warp<GK>(x, make_float4(err, err, err, err),
                                                  make_float4(sbound, sbound, sbound, sbound), tau, k4, Rt);
      const int row = static_cast<int>((t0 + j - SINK) % PAGE);
      const int32_t page = sm.page;
      if (page < 0 || page >= c.n_int2_pages) {
        if (lane == 0) atomicOr(c.err, ERR_INT2_PAGE);
        continue;
      }
      store_group_code_t<GK>(c.int2 + layer * c.int2_layer_stride + ((size_t)page * c.Hkv + head) * record_for(GK),
                             which, row, g);
    }
  }
}

struct AppendArgs {
  int n;
  AppendReq r[APPEND_PER_LAUNCH];
};

template <int GK>
__global__ void __launch_bounds__(APPEND_THREADS) append_kernel(DevCache c, int layer,
                                                                const uint16_t* __restrict__ k,
                                                                const uint16_t* __restrict__ v, AppendArgs a) {
  __shared__ AppendSmem sm;
  append_block<GK>(c, layer, k, v, a.r[blockIdx.x], blockIdx.y, blockIdx.z, sm);
}

struct DemoteArgs {
  int n;
  DemoteEntry e[DEMOTE_PER_LAUNCH];
};

// Multi-layer demote: block (entry, kv head, K or V), each entry one layer of
// one request.  Layers write disjoint pool regions, and only the first layer
// to open a history page writes its page-table entry.
template <int GK>
__global__ void __launch_bounds__(APPEND_THREADS) demote_layers_kernel(DevCache c, DemoteArgs a) {
  __shared__ AppendSmem sm;
  const DemoteEntry& e = a.e[blockIdx.x];
  append_block<GK>(c, e.layer, nullptr, nullptr, e.r, blockIdx.y, blockIdx.z, sm);
}

}  // namespace

cudaError_t launch_pt_update(const DevCache& c, const PtEntry* entries, int n, cudaStream_t s) {
  for (int base = 0; base < n; base += PT_ENTRIES_PER_LAUNCH) {
    PtArgs a;
    a.n = n - base < PT_ENTRIES_PER_LAUNCH ? n - base : PT_ENTRIES_PER_LAUNCH;
    for (int i = 0; i < a.n; ++i) a.e[i] = entries[base + i];
    pt_update_kernel<<<(a.n + 127) / 128, 128, 0, s>>>(c.hist_pt, c.bf16_pt, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_rotation_setup(const DevCache& c, const float* rot_k_src, const float* rot_v_src, float* rot_k,
                                  float* rot_v, float* rot_kt, float* rot_vt, float* rot_cn, cudaStream_t s) {
  const size_t mats = (size_t)c.L * c.Hkv;
  rotation_setup_kernel<<<1024, 256, 0, s>>>(rot_k_src, rot_v_src, rot_k, rot_v, rot_kt, rot_vt, mats);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  colnorm_kernel<<<static_cast<unsigned>(2 * mats), D, 0, s>>>(rot_k_src, rot_v_src, rot_cn, static_cast<int>(mats));
  return cudaGetLastError();
}

cudaError_t launch_prefill_bf16(const DevCache& c, int layer, const uint16_t* k, const uint16_t* v, int64_t in_base,
                                int64_t p0, int64_t p1, BF16Dest dst, cudaStream_t s) {
  if (p1 <= p0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(p1 - p0), 2);
  prefill_bf16_kernel<<<grid, 128, 0, s>>>(c, layer, k, v, in_base, p0, dst);
  return cudaGetLastError();
}

cudaError_t launch_prefill_hist(const DevCache& c, int layer, int slot, const uint16_t* k, const uint16_t* v,
                                int64_t in_base, int64_t h0, int64_t h1, cudaStream_t s) {
  if (h1 <= h0) return cudaSuccess;
  static unsigned attr_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(attr_done & (1u << dev))) {
    e = cudaFuncSetAttribute(prefill_hist_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PREFILL_SMEM));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_hist_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(PREFILL_SMEM));
    if (e != cudaSuccess) return e;
    if (dev < 32) attr_done |= 1u << dev;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // tiles aligned to PF_TILE history slots; two resident blocks per SM over the
  // 2 Hkv (kv head, K or V) matrices
  const int64_t k0 = (h0 - SINK) / PF_TILE;
  const int64_t tiles = (h1 - SINK + PF_TILE - 1) / PF_TILE - k0;
  const int64_t per_matrix = std::max<int64_t>(1, std::min<int64_t>(tiles, (2 * (int64_t)sms) / (2 * c.Hkv)));
  const int64_t tiles_per_cta = (tiles + per_matrix - 1) / per_matrix;
  dim3 grid(static_cast<unsigned>((tiles + tiles_per_cta - 1) / tiles_per_cta), c.Hkv, 2);
  if (c.gk == 64)
    prefill_hist_kernel<64><<<grid, PF_THREADS, PREFILL_SMEM, s>>>(c, layer, slot, k, v, in_base, h0, h1, k0,
                                                                   tiles, static_cast<int>(tiles_per_cta));
  else
    prefill_hist_kernel<128><<<grid, PF_THREADS, PREFILL_SMEM, s>>>(c, layer, slot, k, v, in_base, h0, h1, k0,
                                                                    tiles, static_cast<int>(tiles_per_cta));
  return cudaGetLastError();
}

cudaError_t launch_append(const DevCache& c, int layer, const AppendReq* reqs, int n, const uint16_t* k,
                          const uint16_t* v, cudaStream_t s) {
  for (int base = 0; base < n; base += APPEND_PER_LAUNCH) {
    AppendArgs a;
    a.n = n - base < APPEND_PER_LAUNCH ? n - base : APPEND_PER_LAUNCH;
    for (int i = 0; i < a.n; ++i) a.r[i] = reqs[base + i];
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.n), static_cast<unsigned>(c.Hkv), 2);
    cfg.blockDim = dim3(APPEND_THREADS);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    const cudaError_t e = c.gk == 64 ? cudaLaunchKernelEx(&cfg, append_kernel<64>, c, layer, k, v, a)
                                     : cudaLaunchKernelEx(&cfg, append_kernel<128>, c, layer, k, v, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_demote_layers(const DevCache& c, const DemoteEntry* entries, int n, cudaStream_t s) {
  for (int base = 0; base < n; base += DEMOTE_PER_LAUNCH) {
    DemoteArgs a;
    a.n = n - base < DEMOTE_PER_LAUNCH ? n - base : DEMOTE_PER_LAUNCH;
    for (int i = 0; i < a.n; ++i) a.e[i] = entries[base + i];
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.n), static_cast<unsigned>(c.Hkv), 2);
    cfg.blockDim = dim3(APPEND_THREADS);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    const cudaError_t e = c.gk == 64 ? cudaLaunchKernelEx(&cfg, demote_layers_kernel<64>, c, a)
                                     : cudaLaunchKernelEx(&cfg, demote_layers_kernel<128>, c, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace oscar
