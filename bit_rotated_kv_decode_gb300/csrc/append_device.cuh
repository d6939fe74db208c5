// Device-side append + demote of one (request, kv head, K or V), shared by the
// append kernel and the fused decode-step kernel.
//
// "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计": a new token enters the
// BF16 recent window; when the window is full the oldest recent token is first
// rotated, clipped, quantised and packed into INT2 history ("Together AI
// Open-Sources OSCAR" (MarkTechPost), section "The Serving System").
#pragma once

#include "internal.h"
#include "quant_device.cuh"

namespace oscar {

__device__ __forceinline__ uint16_t* bf16_row(const DevCache& c, int layer, int page, int head, int which,
                                              int row) {
  return c.bf16 + layer * c.bf16_layer_stride + ((size_t)page * c.Hkv + head) * BF16_RECORD_ELEMS +
         (size_t)which * PAGE * D + (size_t)row * D;
}

__device__ __forceinline__ uint8_t* int2_record(const DevCache& c, int layer, int page, int head) {
  return c.int2 + layer * c.int2_layer_stride + ((size_t)page * c.Hkv + head) * c.record;
}

// {s, z} of the lane's group at token slot `slot`, from the first lane of each
// group (lane 0; lanes 0 and 16 at G_K = 64).
template <int GK>
__device__ __forceinline__ void store_group_meta(uint8_t* rec, int which, int slot, const GroupCode& g) {
  const int lane = threadIdx.x & 31;
  constexpr int LPG = GK / 4, MB = meta_bytes_for(GK);
  if ((lane & (LPG - 1)) == 0) {
    const int off = which ? v_meta_off_for(GK) : k_meta_off_for(GK);
    *reinterpret_cast<uint32_t*>(rec + off + slot * MB + 4 * (lane / LPG)) =
        static_cast<uint32_t>(g.s_bits) | (static_cast<uint32_t>(g.z_bits) << 16);
  }
}

// The lane's group code of one token into a record: 32 code bytes at slot * 32 of
// the K or V code region (lane l's byte at l), then {s, z}.
template <int GK>
__device__ __forceinline__ void store_group_code_t(uint8_t* rec, int which, int slot, const GroupCode& g) {
  const int lane = threadIdx.x & 31;
  rec[(which ? V_CODES_OFF : K_CODES_OFF) + slot * CODE_BYTES + lane] = static_cast<uint8_t>(g.byte);
  store_group_meta<GK>(rec, which, slot, g);
}

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_GROUPS = APPEND_THREADS / 32;    // row groups of the rotation
constexpr int APPEND_ROWS = D / APPEND_GROUPS;        // rows per group

// One request, kv head, K or V per block of APPEND_THREADS threads: demote the
// token in the ring slot (if any), then write the new token into its slot.
//
// Rotation: thread (row group g, lane l) accumulates channels 4l .. 4l+3 over
// rows 16g .. 16g+15 with 16 independent float4 loads of R; the 8 partial sums
// are added in order.  Each value has at most 16 + 8 roundings, so its error
// is below gamma_24 * sum_i |k_i R_ic|, which is accumulated alongside.
struct AppendSmem {
  float xin[D];
  __align__(16) float part[APPEND_GROUPS][D];
  __align__(16) float apart[APPEND_GROUPS][D];
};

// The work of one (request, kv head, K or V) by a unit of APPEND_THREADS
// consecutive threads (whole warps): t is the thread's index in the unit and
// sync() a barrier over the unit.
template <int GK, typename Sync>
__device__ __forceinline__ void append_work(const DevCache& c, int layer, const uint16_t* __restrict__ k,
                                            const uint16_t* __restrict__ v, const AppendReq& q, int head, int which,
                                            AppendSmem& sm, int t, Sync sync) {
  float* xin = sm.xin;
  float (*part)[D] = sm.part;
  float (*apart)[D] = sm.apart;
  const int lane = t & 31, grp = t >> 5;
  const size_t lh = (size_t)layer * c.Hkv + head;

  if (q.demote_slot >= 0) {
    const bool ok_src = q.src_page >= 0 && q.src_page < c.n_bf16_pages;
    const bool ok_dst = q.hist_page >= 0 && q.hist_page < c.n_int2_pages;
    if (!ok_src || !ok_dst) {
      if (t == 0) atomicOr(c.err, ok_src ? ERR_INT2_PAGE : ERR_BF16_PAGE);
    } else {
      const float* __restrict__ R = (which ? c.rot_v : c.rot_k) + lh * D * D;
      float4 r[APPEND_ROWS];
#pragma unroll
      for (int i = 0; i < APPEND_ROWS; ++i)
        r[i] = __ldg(reinterpret_cast<const float4*>(R + (size_t)(APPEND_ROWS * grp + i) * D) + lane);
      if (t < D) xin[t] = bf16_bits_to_float(bf16_row(c, layer, q.src_page, head, which, q.src_row)[t]);
      sync();
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, aac[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int i = 0; i < APPEND_ROWS; ++i) {
        const float kv = xin[APPEND_ROWS * grp + i];
        const float ka = fabsf(kv);
        acc[0] = fmaf(kv, r[i].x, acc[0]);
        acc[1] = fmaf(kv, r[i].y, acc[1]);
        acc[2] = fmaf(kv, r[i].z, acc[2]);
        acc[3] = fmaf(kv, r[i].w, acc[3]);
        aac[0] = __fmaf_ru(ka, fabsf(r[i].x), aac[0]);
        aac[1] = __fmaf_ru(ka, fabsf(r[i].y), aac[1]);
        aac[2] = __fmaf_ru(ka, fabsf(r[i].z), aac[2]);
        aac[3] = __fmaf_ru(ka, fabsf(r[i].w), aac[3]);
      }
      reinterpret_cast<float4*>(part[grp])[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      reinterpret_cast<float4*>(apart[grp])[lane] = make_float4(aac[0], aac[1], aac[2], aac[3]);
      sync();
      if (grp == 0) {
        float x[4], e[4], sabs[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float sum = part[0][4 * lane + j], asum = apart[0][4 * lane + j];
#pragma unroll
          for (int g2 = 1; g2 < APPEND_GROUPS; ++g2) {
            sum += part[g2][4 * lane + j];
            asum = __fadd_ru(asum, apart[g2][4 * lane + j]);
          }
          x[j] = sum;
          e[j] = __fmul_ru(gamma_n(APPEND_ROWS + APPEND_GROUPS), asum);
          sabs[j] = __fmul_ru(asum, 1.0001f);   // >= sum_i |k_i R_ic| (asum is accumulated rounding up)
        }
        const float tau = (which ? c.tau_v : c.tau_k)[lh];
        const float* __restrict__ Rt = (which ? c.rot_vt : c.rot_kt) + lh * D * D;
        const float4 k4 = make_float4(xin[4 * lane], xin[4 * lane + 1], xin[4 * lane + 2], xin[4 * lane + 3]);
        const GroupCode g = quantize_group_warp<GK>(make_float4(x[0], x[1], x[2], x[3]),
                                                    make_float4(e[0], e[1], e[2], e[3]),
                                                    make_float4(sabs[0], sabs[1], sabs[2], sabs[3]), tau, k4, Rt);
        store_group_code_t<GK>(int2_record(c, layer, q.hist_page, head), which, q.demote_slot, g);
      }
      if (q.pt_index >= 0 && head == 0 && which == 0 && t == 0) {
        c.hist_pt[(size_t)q.slot * c.max_pages + q.pt_index] = q.hist_page;
      }
    }
  }
  sync();   // the demoted row has been read before its slot is overwritten
  if (q.in_row >= 0 && t < D) {
    if (q.dst_page < 0 || q.dst_page >= c.n_bf16_pages) {
      if (t == 0) atomicOr(c.err, ERR_BF16_PAGE);
      return;
    }
    const uint16_t* src = (which ? v : k) + ((size_t)q.in_row * c.Hkv + head) * D;
    bf16_row(c, layer, q.dst_page, head, which, q.dst_row)[t] = src[t];
  }
}

// One block of APPEND_THREADS threads per (request, kv head, K or V), launched
// with programmatic dependent launch: R is written once at set-up, so L2 is warmed
// with this thread's rows while the preceding grid (which may still be writing
// k / v or reading the cache) finishes; nothing else is read before the wait.
template <int GK>
__device__ __forceinline__ void append_block(const DevCache& c, int layer, const uint16_t* __restrict__ k,
                                             const uint16_t* __restrict__ v, const AppendReq& q, int head,
                                             int which, AppendSmem& sm) {
  const int t = threadIdx.x, lane = t & 31, grp = t >> 5;
  if (q.demote_slot >= 0) {
    const float* R = (which ? c.rot_v : c.rot_k) + ((size_t)layer * c.Hkv + head) * D * D;
#pragma unroll
    for (int i = 0; i < APPEND_ROWS; ++i)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(R + (size_t)(APPEND_ROWS * grp + i) * D + 4 * lane));
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  append_work<GK>(c, layer, k, v, q, head, which, sm, t, [] { __syncthreads(); });
}

}  // namespace oscar
