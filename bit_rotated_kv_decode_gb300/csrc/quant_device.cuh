// Device-side INT2 quantiser of one 128-channel token-head group.
//
// Write path of "Together AI Open-Sources OSCAR" (MarkTechPost), section "The
// Serving System: Mixed-Precision Cache Layout": rotate, clip to the stored
// threshold, per-token asymmetric INT2 with a scale and a zero point ("scale /
// zero point" in "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计"),
// four codes per byte.  The decisions are defined on x = fp32_rn(k . R), the
// exactly rounded rotated value, in IEEE fp32 / fp16 round-to-nearest-even:
//   xc = clip(x, -tau, tau) + 0          (signed zero canonicalised to +0)
//   z  = fp16_rn(min xc)
//   s  = fp16_rn(fl32(fl32(max xc - min xc) / 3))
//   code = clamp(rint(fl32(fl32(xc - z) / s)), 0, 3), 0 when s == 0
//
// The kernels compute x with an fp32 FMA chain of 128 steps, whose error is at
// most gamma_128 * sum_i |k_i R_ij| <= gamma_128 * |k|_2 * |R_:j|_2 (recursive
// summation bound, one rounding per step), plus half an ulp for the final
// rounding.  Every decision is taken on the interval [x - e, x + e]; the steps
// above are monotone in x, so equal decisions at both ends are the exact
// decision.  Where the ends differ (rare), the value is recomputed exactly: a
// compensated (TwoSum) double-precision dot product -- each bf16 x fp32 product
// is exact in double -- rounded once to fp32.  That result equals
// fp32_rn(k . R) unless the exact value lies within ~2^-90 sum|k_i R_ij| of an
// fp32 rounding midpoint.
#pragma once

#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {

struct GroupCode {
  uint32_t byte;      // packed codes of this lane's 4 channels
  uint16_t s_bits;    // fp16 scale
  uint16_t z_bits;    // fp16 zero point
  int exact_calls;    // values recomputed exactly by this lane
};

// gamma_128 = 128 u / (1 - 128 u), u = 2^-24, rounded up with margin.
constexpr float GAMMA_128 = 7.6295e-6f;

__device__ __forceinline__ float clip_canon(float x, float tau) {
  return __fadd_rn(fminf(fmaxf(x, -tau), tau), 0.0f);
}

__device__ __forceinline__ uint32_t code_of(float xc, float z, float s) {
  if (s == 0.0f) return 0u;
  const float t = __fdiv_rn(__fsub_rn(xc, z), s);
  return static_cast<uint32_t>(fminf(fmaxf(rintf(t), 0.0f), 3.0f));
}

__device__ __forceinline__ float scale_of(float mx, float mn) {
  return __half2float(__float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f)));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32_rn of sum_i k_i * rt_i, k given as fp32 values that are exactly bf16.
__device__ __forceinline__ float exact_dot_fp32(const float* k, int k_stride, const float* __restrict__ rt) {
  double s = 0.0, c = 0.0;
  for (int i = 0; i < D; ++i) {
    const double p = static_cast<double>(k[i * k_stride]) * static_cast<double>(__ldg(rt + i));
    const double t = s + p;
    const double bp = t - s;
    c += (s - (t - bp)) + (p - bp);
    s = t;
  }
  const double hi = s + c;
  const double bh = hi - s;
  const double lo = (s - (hi - bh)) + (c - bh);   // hi + lo == s + c exactly
  float f = __double2float_rn(hi);
  const double fd = static_cast<double>(f);
  if (hi != fd && lo != 0.0) {
    // hi may sit exactly on an fp32 rounding midpoint; then the remainder decides
    const float nb = nextafterf(f, hi > fd ? INFINITY : -INFINITY);
    const double mid = 0.5 * (fd + static_cast<double>(nb));
    if (hi == mid) f = (lo > 0.0) ? fmaxf(f, nb) : fminf(f, nb);
  }
  return f;
}

// A full warp holds the group: lane l owns channels 4l .. 4l+3 (rotated by the
// FMA chain, not yet clipped); err bounds the chain's error for this token.
// exact(ch) returns fp32_rn(k . R_:ch) for channel ch.
template <class Exact>
__device__ __forceinline__ GroupCode quantize_group_warp(float4 xv, float err, float tau, Exact exact) {
  const int lane = threadIdx.x & 31;
  float x[4] = {xv.x, xv.y, xv.z, xv.w};
  float lo[4], hi[4];
  GroupCode g;
  g.exact_calls = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float e = __fmaf_ru(fabsf(x[i]), 0x1.0001p-24f, err);
    lo[i] = clip_canon(__fsub_rd(x[i], e), tau);
    hi[i] = clip_canon(__fadd_ru(x[i], e), tau);
  }
  auto reduce_min = [](float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
  };
  auto reduce_max = [](float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
  };
  float mn_lo = reduce_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
  float mn_hi = reduce_min(fminf(fminf(hi[0], hi[1]), fminf(hi[2], hi[3])));
  float mx_lo = reduce_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
  float mx_hi = reduce_max(fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3])));
  const bool meta_sure = __half_as_ushort(__float2half_rn(mn_lo)) == __half_as_ushort(__float2half_rn(mn_hi)) &&
                         scale_of(mx_lo, mn_hi) == scale_of(mx_hi, mn_lo);
  if (!meta_sure) {
    // (warp-uniform) the group's min or max is too close to an fp16 boundary: exact values
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float xe = clip_canon(exact(4 * lane + i), tau);
      lo[i] = hi[i] = xe;
    }
    g.exact_calls += 4;
    mn_lo = mn_hi = reduce_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
    mx_lo = mx_hi = reduce_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
  }
  const __half zh = __float2half_rn(mn_lo);
  const float z = __half2float(zh);
  const float sr = __fdiv_rn(__fsub_rn(mx_lo, mn_lo), 3.0f);
  const __half sh = __float2half_rn(sr);
  const float s = __half2float(sh);
  g.byte = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t c = code_of(lo[i], z, s);
    if (c != code_of(hi[i], z, s)) {
      c = code_of(clip_canon(exact(4 * lane + i), tau), z, s);
      g.exact_calls += 1;
    }
    g.byte |= c << (2 * i);
  }
  g.s_bits = __half_as_ushort(sh);
  g.z_bits = __half_as_ushort(zh);
  return g;
}

// Error bound of the FMA chain for a token with |k|_2^2 = knorm2 and a matrix
// whose columns have norm at most colnorm.
__device__ __forceinline__ float chain_error_bound(float knorm2, float colnorm) {
  return GAMMA_128 * 1.0001f * sqrtf(knorm2 * 1.0001f) * colnorm;
}

}  // namespace oscar
