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

constexpr int PF_TILE = 32;   // history positions per block
constexpr size_t PREFILL_SMEM = (size_t)(2 * PF_TILE * D + PF_TILE) * sizeof(float);

// Tile of up to PF_TILE history positions (x) of one kv head (y), K or V (z).
// Shared memory: the input tile row-major ks[PF_TILE][128] (fp32), the rotated
// values xs[PF_TILE][128] and |k|^2 of each token (rounded up).
__global__ void __launch_bounds__(128) prefill_hist_kernel(DevCache c, int layer, int slot,
                                                           const uint16_t* __restrict__ k,
                                                           const uint16_t* __restrict__ v, int64_t in_base,
                                                           int64_t h0, int64_t h1) {
  extern __shared__ float4 smem4[];
  float* ks = reinterpret_cast<float*>(smem4);     // [PF_TILE][D] input tile
  float* xs = ks + PF_TILE * D;                    // [PF_TILE][D] rotated values
  float* kn = xs + PF_TILE * D;                    // [PF_TILE] |k|^2, rounded up
  const int head = blockIdx.y;
  const int which = blockIdx.z;
  const int64_t t0 = h0 + (int64_t)blockIdx.x * PF_TILE;
  const int ntok = static_cast<int>(h1 - t0 < PF_TILE ? h1 - t0 : PF_TILE);
  const uint16_t* src = which ? v : k;
  const size_t lh = (size_t)layer * c.Hkv + head;
  const float* __restrict__ R = (which ? c.rot_v : c.rot_k) + lh * D * D;
  const float* __restrict__ Rt = (which ? c.rot_vt : c.rot_kt) + lh * D * D;
  const float tau = (which ? c.tau_v : c.tau_k)[lh];
  const float colnorm = c.rot_cn[(size_t)which * c.L * c.Hkv + lh];
  const int t = threadIdx.x;

  {
    // PF_TILE tokens x 128 channels of bf16 in 16-byte chunks, all in flight;
    // 16 consecutive threads share a token and add up its |k|^2
    constexpr int CHUNKS = PF_TILE * D / 8 / 128;
    uint4 v[CHUNKS];
#pragma unroll
    for (int u = 0; u < CHUNKS; ++u) {
      const int idx = u * 128 + t, j = idx / (D / 8), part = idx % (D / 8);
      v[u] = j < ntok ? reinterpret_cast<const uint4*>(src + ((size_t)(t0 + j - in_base) * c.Hkv + head) * D)[part]
                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < CHUNKS; ++u) {
      const int idx = u * 128 + t, j = idx / (D / 8), part = idx % (D / 8);
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float f[8];
      float sq = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        sq = __fmaf_ru(f[2 * e], f[2 * e], sq);
        sq = __fmaf_ru(f[2 * e + 1], f[2 * e + 1], sq);
      }
      float4* row = reinterpret_cast<float4*>(ks + j * D + 8 * part);
      row[0] = make_float4(f[0], f[1], f[2], f[3]);
      row[1] = make_float4(f[4], f[5], f[6], f[7]);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sq = __fadd_ru(sq, __shfl_xor_sync(0xffffffffu, sq, off));
      if (part == 0) kn[j] = sq;
    }
  }
  __syncthreads();

  // rotation: thread co keeps the tile's FMA chains over i = 0 .. 127 in order;
  // a float4 of ks (4 channels of one token) is the same address across the warp
  const int co = t;
  float acc[PF_TILE];
#pragma unroll
  for (int j = 0; j < PF_TILE; ++j) acc[j] = 0.0f;
  for (int i4 = 0; i4 < D / 4; ++i4) {
    const float r0 = __ldg(R + (4 * i4 + 0) * D + co);
    const float r1 = __ldg(R + (4 * i4 + 1) * D + co);
    const float r2 = __ldg(R + (4 * i4 + 2) * D + co);
    const float r3 = __ldg(R + (4 * i4 + 3) * D + co);
#pragma unroll
    for (int j = 0; j < PF_TILE; ++j) {
      const float4 kk = *reinterpret_cast<const float4*>(ks + j * D + 4 * i4);
      acc[j] = fmaf(kk.x, r0, acc[j]);
      acc[j] = fmaf(kk.y, r1, acc[j]);
      acc[j] = fmaf(kk.z, r2, acc[j]);
      acc[j] = fmaf(kk.w, r3, acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < PF_TILE; ++j) xs[j * D + co] = acc[j];
  __syncthreads();

  const int warp = t >> 5;
  const int lane = t & 31;
  const int32_t* pt = c.hist_pt + (size_t)slot * c.max_pages;
  for (int j = warp; j < ntok; j += 4) {
    const float4 x = *reinterpret_cast<const float4*>(xs + j * D + 4 * lane);
    const float4 k4 = *reinterpret_cast<const float4*>(ks + j * D + 4 * lane);
    const float knj = kn[j];
    const float err = chain_error_bound(knj, colnorm);
    const float sbound = __fmul_ru(__fsqrt_ru(__fmul_ru(knj, 1.0001f)), colnorm);   // >= sum_i |k_i R_ic|
    const GroupCode g = quantize_group_warp(x, make_float4(err, err, err, err),
                                            make_float4(sbound, sbound, sbound, sbound), tau, k4, Rt);
    const int64_t h = t0 + j - SINK;
    const int32_t page = pt[h / PAGE];
    const int row = static_cast<int>(h % PAGE);
    if (page < 0 || page >= c.n_int2_pages) {
      if (lane == 0) atomicOr(c.err, ERR_INT2_PAGE);
      continue;
    }
    uint8_t* rec = int2_record(c, layer, page, head);
    rec[(which ? V_CODES_OFF : K_CODES_OFF) + row * CODE_BYTES + lane] = static_cast<uint8_t>(g.byte);
    if (lane == 0) {
      *reinterpret_cast<uint32_t*>(rec + (which ? V_META_OFF : K_META_OFF) + row * META_BYTES) =
          static_cast<uint32_t>(g.s_bits) | (static_cast<uint32_t>(g.z_bits) << 16);
    }
  }
}

struct AppendArgs {
  int n;
  AppendReq r[APPEND_PER_LAUNCH];
};

__global__ void __launch_bounds__(APPEND_THREADS) append_kernel(DevCache c, int layer,
                                                                const uint16_t* __restrict__ k,
                                                                const uint16_t* __restrict__ v, AppendArgs a) {
  __shared__ AppendSmem sm;
  append_block(c, layer, k, v, a.r[blockIdx.x], blockIdx.y, blockIdx.z, sm);
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
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(prefill_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(PREFILL_SMEM));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const size_t smem = PREFILL_SMEM;
  dim3 grid(static_cast<unsigned>((h1 - h0 + PF_TILE - 1) / PF_TILE), c.Hkv, 2);
  prefill_hist_kernel<<<grid, 128, smem, s>>>(c, layer, slot, k, v, in_base, h0, h1);
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
    const cudaError_t e = cudaLaunchKernelEx(&cfg, append_kernel, c, layer, k, v, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace oscar
